"""GPU parity of the Scatter layer's geometry mode (INTRA, "Why Scatter Is
Uniform and Non-Contiguous"; "CQS-Aware Token-Sparse FlashAttention Kernel").

bsa_forward_scatter fetches each 128-position tile as one box of 128 tokens
at stride R.  It must give bsa_forward's result on the Scatter maps bit for
bit (the same tiles in the same order), and match the oracle, which reads
the maps from the definition in synth.scatter_map.
"""
import numpy as np
import pytest
import torch

import long_context_mask_gb300 as bsa
import oracle
import synth
from gpu_util import compare, status_ok

pytestmark = pytest.mark.gpu


def _problem(seed, H, N, D, R, density, H_kv=None):
    g = torch.Generator().manual_seed(seed)
    q = synth.normal_bf16(g, (1, H, N, D))
    hk = H if H_kv is None else H_kv
    k, v = (synth.normal_bf16(g, (1, hk, N, D)) for _ in range(2))
    nqb = N // 128
    rng = np.random.default_rng(seed)
    mask = (rng.random((H * nqb, nqb)) < density).astype(np.uint8)
    mask[np.arange(H * nqb), np.arange(H * nqb) % nqb] = 1
    mask[::5] = 0                                   # some empty rows
    m = synth.scatter_map(N, R)
    qmap = np.broadcast_to(m, (H, N)).copy()
    kvmap = np.broadcast_to(m, (hk, N)).copy()
    prob = synth.Problem("scatter-geo", 1, H, N, D, q, k, v, mask=mask, q_map=qmap, kv_map=kvmap,
                         H_kv=H_kv)
    return prob


def _lists(prob):
    idx, cnt, _ = oracle.index_mask(prob.mask)
    return torch.from_numpy(idx).cuda(), torch.from_numpy(cnt).cuda()


@pytest.mark.parametrize("N,R,D", [(2048, 16, 128), (4096, 8, 64), (4096, 32, 128), (1024, 1, 128)])
def test_scatter_geometry_matches_maps_and_oracle(N, R, D):
    prob = _problem(7 + R, 2, N, D, R, 0.3)
    idx, cnt = _lists(prob)
    q, k, v = prob.q.cuda(), prob.k.cuda(), prob.v.cuda()
    lw = torch.from_numpy(np.random.default_rng(3).normal(size=idx.shape).astype(np.float32)).cuda()
    o1, o2 = torch.empty_like(q), torch.empty_like(q)
    l1 = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    l2 = torch.empty_like(l1)
    qm = torch.from_numpy(prob.q_map).cuda()
    km = torch.from_numpy(prob.kv_map).cuda()
    bsa.forward(q, k, v, idx, cnt, o1, l1, log_w=lw, q_map=qm, kv_map=km)
    bsa.forward_scatter(q, k, v, R, idx, cnt, o2, l2, log_w=lw)
    torch.cuda.synchronize()
    status_ok()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    compare(prob, o2, l2, idx, cnt, lw=lw)


def test_scatter_geometry_grouped_heads_and_order():
    prob = _problem(21, 4, 2048, 128, 16, 0.4, H_kv=2)
    idx, cnt = _lists(prob)
    q, k, v = prob.q.cuda(), prob.k.cuda(), prob.v.cuda()
    o1, o2 = torch.empty_like(q), torch.empty_like(q)
    l1 = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    l2 = torch.empty_like(l1)
    qm = torch.from_numpy(prob.q_map).cuda()
    km = torch.from_numpy(prob.kv_map).cuda()
    bsa.forward_masked(q, k, v, idx, cnt, o1, l1, q_map=qm, kv_map=km)
    perm = torch.empty((4, prob.nqb), dtype=torch.int32, device="cuda")
    bsa.reorder_rows(cnt.view(4, -1), 5, perm)
    bsa.forward_scatter(q, k, v, 16, idx, cnt, o2, l2, row_perm=perm)
    torch.cuda.synchronize()
    status_ok()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    compare(prob, o2, l2, idx, cnt)


def test_scatter_layer_full_size():
    """The Scatter layer workload (B1 H24 N16384 D128, T = R = 128, one block
    per row) in the benchmark's launch configuration: bit-identical to the
    map path everywhere, against the oracle on sampled rows."""
    prob = synth.scatter()
    rows, nqb = prob.rows, prob.nqb
    idx = torch.from_numpy((np.arange(rows) % nqb).astype(np.int32)[:, None]).cuda()
    cnt = torch.ones(rows, dtype=torch.int32, device="cuda")
    q, k, v = prob.q.cuda(), prob.k.cuda(), prob.v.cuda()
    BH = prob.B * prob.H
    perm = torch.empty((BH, nqb), dtype=torch.int32, device="cuda")
    bsa.reorder_rows(cnt.view(BH, -1), bsa.resident_ctas(prob.D), perm)
    o1, o2 = torch.empty_like(q), torch.empty_like(q)
    l1 = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    l2 = torch.empty_like(l1)
    bsa.forward(q, k, v, idx, cnt, o1, l1, q_map=torch.from_numpy(prob.q_map).cuda(),
                kv_map=torch.from_numpy(prob.kv_map).cuda(), row_perm=perm)
    bsa.forward_scatter(q, k, v, 128, idx, cnt, o2, l2, row_perm=perm)
    torch.cuda.synchronize()
    status_ok()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    sel = np.array([0, 1, 77, nqb - 1, (BH - 1) * nqb, (BH - 1) * nqb + 64, BH * nqb - 1], np.int64)
    compare(prob, o2, l2, idx, cnt, sel=sel)
