"""bsa_gather_rows (token rows permuted into gathered order in HBM) and the
forward pass on pre-gathered keys/values.

The copy is checked bit for bit against plain host indexing; the forward on
gathered K/V (kv_map = NULL) must equal the forward that gathers the same
rows inside the kernel bit for bit, and match the oracle."""
import numpy as np
import pytest
import torch

import long_context_mask_gb300 as bsa
import synth
from gpu_util import DEV, compare, cuda, gpu_index, run_forward, sample_rows, status_ok

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.contiguous().view(torch.int16).cpu()


@pytest.mark.parametrize("D,heads,N", [(128, 3, 1000), (64, 2, 4096), (128, 1, 1), (64, 5, 33)])
def test_gather_rows_equals_indexing(D, heads, N):
    g = np.random.default_rng(D * 7 + N)
    src = torch.from_numpy(g.standard_normal((heads, N, D)).astype(np.float32)).to(torch.bfloat16)
    m = np.stack([g.permutation(N) for _ in range(heads)]).astype(np.int32)
    m[0, : min(N, 7)] = m[0, 0]  # repeated rows are allowed
    dst = bsa.gather_rows(src.to(DEV), cuda(m))
    status_ok()
    expect = torch.stack([src[h][torch.from_numpy(m[h]).long()] for h in range(heads)])
    assert torch.equal(_bits(dst), _bits(expect))


def test_gather_rows_bad_entry_is_flagged_and_zeroed():
    heads, N, D = 2, 256, 128
    g = np.random.default_rng(11)
    src = torch.from_numpy(g.standard_normal((heads, N, D)).astype(np.float32)).to(torch.bfloat16)
    m = np.stack([g.permutation(N) for _ in range(heads)]).astype(np.int32)
    m[1, 5], m[0, 200] = -1, N
    dst = bsa.gather_rows(src.to(DEV), cuda(m)).cpu()
    assert bsa.device_status() == 6  # BSA_ERR_BOUNDS
    assert not dst[1, 5].any() and not dst[0, 200].any()
    ok = m.copy()
    ok[1, 5], ok[0, 200] = 0, 0
    expect = torch.stack([src[h][torch.from_numpy(ok[h]).long()] for h in range(heads)])
    expect[1, 5] = 0
    expect[0, 200] = 0
    assert torch.equal(_bits(dst), _bits(expect))


def _forward_pregathered(prob, idx, cnt, lw):
    q, k, v = cuda(prob.q), cuda(prob.k), cuda(prob.v)
    kv_map = cuda(prob.kv_map)
    kg, vg = bsa.gather_rows(k, kv_map), bsa.gather_rows(v, kv_map)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=DEV)
    bsa.forward(q, kg, vg, idx, cnt, o, lse, log_w=lw, q_map=cuda(prob.q_map), kv_map=None)
    return o, lse


def test_pregathered_equals_in_kernel_gather():
    prob = synth.sampled(seed=21, H=3, N=8192)  # 64 blocks: top-16 exact + 8 sampled, random perms
    idx, cnt, lw = gpu_index(prob)
    o1, lse1 = run_forward(prob, idx, cnt, lw=lw)
    o2, lse2 = _forward_pregathered(prob, idx, cnt, lw)
    status_ok()
    assert torch.equal(_bits(o1), _bits(o2))
    assert torch.equal(lse1.cpu(), lse2.cpu())
    compare(prob, o2, lse2, idx, cnt, lw=lw)


def test_sampled_config_full_size_pregathered():
    prob = synth.sampled(seed=4)  # H40 N75776, the permuted importance-sampling workload
    idx, cnt, lw = gpu_index(prob)
    o, lse = _forward_pregathered(prob, idx, cnt, lw)
    status_ok()
    compare(prob, o, lse, idx, cnt, lw=lw, sel=sample_rows(prob, 3))
