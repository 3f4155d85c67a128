"""CRM rows, the CRM forward pass and eq. (7) upscaling on the GPU
(ScalingAttention sections 7.1-7.3) against the oracle and the list path."""
import numpy as np
import pytest
import torch

import long_context_mask_gb300 as bsa
import oracle
import synth
from gpu_util import DEV, compare, cuda, gpu_index, run_forward, status_ok

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    bsa.device_status()


def _crm(src, mode, p=0.0, extra_words=0):
    rows, nkb = src.shape
    nw = (nkb + 31) // 32 + extra_words
    words = torch.full((rows, nw), 123, dtype=torch.int32, device=DEV)
    bsa.build_crm(mode, cuda(src), words, p=p)
    status_ok()
    return words


@pytest.mark.parametrize("nkb", [1, 31, 32, 100, 256])
def test_crm_rows_bit_exact(nkb):
    g = np.random.default_rng(nkb)
    mask = (g.random((700, nkb)) < 0.3).astype(np.uint8)
    w = _crm(mask, bsa.IDX_MASK_U8, extra_words=1).cpu().numpy().view(np.uint32)
    ref = oracle.crm_rows(mask)
    np.testing.assert_array_equal(w[:, :ref.shape[1]], ref)
    assert np.all(w[:, ref.shape[1]:] == 0)
    T = g.random((700, nkb)).astype(np.float32)
    w = _crm(T, bsa.IDX_THRESHOLD_F32, p=0.2).cpu().numpy().view(np.uint32)
    np.testing.assert_array_equal(w, oracle.crm_rows(T, 0.2))


@pytest.mark.parametrize("D", [64, 128])
def test_crm_forward_small_all_rows_with_maps_and_order(D):
    prob = synth.tiny(seed=21, H=2, N=2048, D=D, density=0.3)
    g = np.random.default_rng(5)
    perm = np.stack([g.permutation(prob.N) for _ in range(2)]).astype(np.int32)
    prob.q_map, prob.kv_map = perm, perm
    words = _crm(prob.mask, bsa.IDX_MASK_U8)
    rp = cuda(np.stack([g.permutation(prob.nqb) for _ in range(2)]).astype(np.int32))
    q, k, v = cuda(prob.q), cuda(prob.k), cuda(prob.v)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=DEV)
    bsa.forward_crm(q, k, v, words, o, lse, q_map=cuda(perm), kv_map=cuda(perm), row_perm=rp)
    status_ok()
    idx, cnt, _ = gpu_index(prob)
    compare(prob, o, lse, idx, cnt)
    o2, l2 = run_forward(prob, idx, cnt)
    status_ok()
    assert torch.equal(o, o2) and torch.equal(lse, l2)   # same blocks, same order: same bits


def test_crm_forward_threshold_workload_equals_list_forward():
    prob = synth.threshold(seed=2)   # H12 N32768
    words = _crm(prob.T, bsa.IDX_THRESHOLD_F32, p=prob.p)
    q, k, v = cuda(prob.q), cuda(prob.k), cuda(prob.v)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=DEV)
    bsa.forward_crm(q, k, v, words, o, lse)
    idx, cnt, _ = gpu_index(prob)
    o2, l2 = run_forward(prob, idx, cnt, q=q, k=k, v=v)
    status_ok()
    assert torch.equal(o, o2) and torch.equal(lse, l2)


def test_crm_bits_beyond_the_last_block_are_flagged():
    prob = synth.tiny(seed=22, H=1, N=384, D=128, density=1.0)   # 3 blocks
    words = _crm(prob.mask, bsa.IDX_MASK_U8)
    words[0, 0] |= 1 << 5                                          # block 5 does not exist
    q, k, v = cuda(prob.q), cuda(prob.k), cuda(prob.v)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=DEV)
    bsa.forward_crm(q, k, v, words, o, lse)
    assert bsa.device_status() == 6


@pytest.mark.parametrize("shape", [((3, 7, 9), (3, 7, 9)), ((2, 30, 52), (2, 60, 104)),
                                   ((2, 21, 30), (2, 45, 80)), ((1, 5, 5), (1, 3, 4))])
def test_upscale_bit_exact(shape):
    (h, ub, vb), (_, ut, vt) = shape
    T = np.random.default_rng(ub * vb).random((h, ub, vb)).astype(np.float32)
    out = torch.empty((h, ut, vt), dtype=torch.float32, device=DEV)
    bsa.upscale_threshold(cuda(T), out)
    status_ok()
    np.testing.assert_array_equal(out.cpu().numpy(), oracle.upscale_threshold(T, ut, vt))
