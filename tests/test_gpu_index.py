"""GPU index lists, row reordering and block sampling: bit-exact vs the oracle."""
import numpy as np
import pytest
import torch

import long_context_mask_gb300 as bsa
import oracle
import synth
from gpu_util import DEV, cuda, status_ok

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    bsa.device_status()  # clear anything left by an earlier module


def _run_index(mode, src, max_kv, p=0.0, k_per_row=None, k_const=0):
    rows = src.shape[0]
    idx = torch.full((rows, max_kv), 7777, dtype=torch.int32, device=DEV)
    cnt = torch.full((rows,), 7777, dtype=torch.int32, device=DEV)
    bsa.build_index(mode, cuda(src), idx, cnt, p=p, k_per_row=cuda(k_per_row), k_const=k_const)
    return idx.cpu().numpy(), cnt.cpu().numpy()


@pytest.mark.parametrize("rows,nkb,density", [(32, 16, 0.25), (3001, 300, 0.3), (5, 1, 0.5),
                                              (64, 33, 1.0), (64, 70, 0.0)])
def test_mask_compaction_bit_exact(rows, nkb, density):
    g = np.random.default_rng(rows + nkb)
    mask = (g.random((rows, nkb)) < density).astype(np.uint8) * g.integers(1, 255, (rows, nkb)).astype(np.uint8)
    idx, cnt = _run_index(bsa.IDX_MASK_U8, mask, nkb)
    ridx, rcnt, ov = oracle.index_mask(mask)
    status_ok()
    assert ov == 0
    np.testing.assert_array_equal(cnt, rcnt)
    np.testing.assert_array_equal(idx, ridx)


def test_mask_overflow_truncates_and_reports():
    g = np.random.default_rng(3)
    mask = (g.random((500, 100)) < 0.5).astype(np.uint8)
    idx, cnt = _run_index(bsa.IDX_MASK_U8, mask, 40)
    ridx, rcnt, ov = oracle.index_mask(mask, max_kv=40)
    assert ov > 0
    assert bsa.device_status() == 3  # BSA_ERR_OVERFLOW
    np.testing.assert_array_equal(cnt, rcnt)
    np.testing.assert_array_equal(idx, ridx)
    status_ok()  # the read cleared it


def test_threshold_map_full_size_bit_exact():
    prob = synth.threshold(seed=2)  # H12 N32768: T [3072, 256], p = 0.15
    # fp32-boundary values: exactly p and its neighbours
    p32 = np.float32(prob.p)
    T = prob.T.copy()
    T[0, :3] = [p32, np.nextafter(p32, np.float32(1)), np.nextafter(p32, np.float32(0))]
    idx, cnt = _run_index(bsa.IDX_THRESHOLD_F32, T, T.shape[1], p=prob.p)
    ridx, rcnt, _ = oracle.index_threshold(T, prob.p)
    status_ok()
    np.testing.assert_array_equal(cnt, rcnt)
    np.testing.assert_array_equal(idx, ridx)


def test_topk_ties_signed_zero_and_edges():
    g = np.random.default_rng(11)
    rows, nkb = 2000, 77
    s = g.integers(-3, 4, (rows, nkb)).astype(np.float32)   # heavy ties
    s[::7] *= np.float32(-0.0)                               # signed zeros
    s[1::5] = g.standard_normal((len(s[1::5]), nkb)).astype(np.float32)
    k = g.integers(0, nkb + 5, rows).astype(np.int32)        # includes 0 and > nKB
    idx, cnt = _run_index(bsa.IDX_TOPK_F32, s, nkb, k_per_row=k)
    ridx, rcnt, _ = oracle.index_topk(s, k, max_kv=nkb)
    status_ok()
    np.testing.assert_array_equal(cnt, rcnt)
    np.testing.assert_array_equal(idx, ridx)


def test_topk_full_size_dynamic_and_sampled_configs():
    p5 = synth.dynamic(seed=5, H=4)   # 928 blocks per row, per-row k in [93, 185]
    kmax = int(p5.k_per_row.max())
    idx, cnt = _run_index(bsa.IDX_TOPK_F32, p5.scores, kmax, k_per_row=p5.k_per_row)
    ridx, rcnt, _ = oracle.index_topk(p5.scores, p5.k_per_row, max_kv=kmax)
    status_ok()
    np.testing.assert_array_equal(cnt, rcnt)
    np.testing.assert_array_equal(idx, ridx)
    g = torch.Generator().manual_seed(4)
    sc = torch.rand((40 * 592, 592), generator=g).numpy()
    idx, cnt = _run_index(bsa.IDX_TOPK_F32, sc, 16, k_const=16)
    ridx, rcnt, _ = oracle.index_topk(sc, 16, max_kv=16)
    status_ok()
    np.testing.assert_array_equal(idx, ridx)
    np.testing.assert_array_equal(cnt, rcnt)


@pytest.mark.parametrize("wave", [1, 3, 148, 152, 1000])
def test_reorder_bit_exact(wave):
    g = np.random.default_rng(wave)
    heads, nqb = 24, 928
    cnt = g.integers(93, 186, (heads, nqb)).astype(np.int32)
    order = np.stack([g.permutation(nqb) for _ in range(heads)]).astype(np.int32)
    for order_in in (None, order):
        perm = torch.empty((heads, nqb), dtype=torch.int32, device=DEV)
        bsa.reorder_rows(cuda(cnt), wave, perm, order_in=cuda(order_in))
        ref = oracle.reorder_rows(cnt, wave, order_in)
        status_ok()
        np.testing.assert_array_equal(perm.cpu().numpy(), ref)


def test_reorder_rejects_out_of_range_order():
    cnt = np.ones((1, 8), np.int32)
    order = np.arange(8, dtype=np.int32)
    order[3] = 99
    perm = torch.empty((1, 8), dtype=torch.int32, device=DEV)
    bsa.reorder_rows(cuda(cnt), 4, perm, order_in=cuda(order))
    assert bsa.device_status() == 6  # BSA_ERR_BOUNDS


def test_sampler_full_size_bit_exact():
    prob = synth.sampled(seed=4, H=40)
    rows = prob.rows
    ex_idx, ex_cnt, _ = oracle.index_topk(prob.scores, 16, max_kv=16)
    cap = 24
    idx = torch.empty((rows, cap), dtype=torch.int32, device=DEV)
    cnt = torch.empty(rows, dtype=torch.int32, device=DEV)
    lw = torch.empty((rows, cap), dtype=torch.float32, device=DEV)
    bsa.sample_blocks(cuda(prob.scores), cuda(ex_idx), cuda(ex_cnt), 8, cuda(prob.u), idx, cnt, lw)
    ridx, rcnt, rlw, ov = oracle.sample_blocks(prob.scores, ex_idx, ex_cnt, 8, prob.u, cap)
    status_ok()
    assert ov == 0 and np.all(rcnt == 24)
    np.testing.assert_array_equal(cnt.cpu().numpy(), rcnt)
    np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
    np.testing.assert_allclose(lw.cpu().numpy(), rlw, rtol=1e-6, atol=0)


def test_sampler_promotion_and_full_budget():
    g = np.random.default_rng(8)
    rows, nkb = 300, 40
    s = (g.random((rows, nkb)) + 0.01).astype(np.float32)
    s[:, 5] = 50.0   # capped at pi = 1 -> promoted
    s[:, 9] = 20.0
    ex = np.tile(np.array([[0, 1, 2]], np.int32), (rows, 1))
    ec = np.full(rows, 3, np.int32)
    u = g.random(rows)
    for m, cap in ((6, 10), (37, 40), (50, 40)):
        idx = torch.empty((rows, cap), dtype=torch.int32, device=DEV)
        cnt = torch.empty(rows, dtype=torch.int32, device=DEV)
        lw = torch.empty((rows, cap), dtype=torch.float32, device=DEV)
        bsa.sample_blocks(cuda(s), cuda(ex), cuda(ec), m, cuda(u), idx, cnt, lw)
        ridx, rcnt, rlw, ov = oracle.sample_blocks(s, ex, ec, m, u, cap)
        st = bsa.device_status()
        assert st == (3 if ov else 0)
        np.testing.assert_array_equal(cnt.cpu().numpy(), rcnt)
        np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
        np.testing.assert_allclose(lw.cpu().numpy(), rlw, rtol=1e-6, atol=0)
