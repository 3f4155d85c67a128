"""GPU spectral row order (WaveAlign section IV-C) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import long_context_mask_gb300 as bsa
import oracle
import synth
from gpu_util import DEV, cuda, gpu_index, status_ok

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    bsa.device_status()


def _planted(seed, heads, nqb, nkb, clusters):
    rng = np.random.default_rng(seed)
    mask = np.zeros((heads * nqb, nkb), np.uint8)
    lab = rng.integers(0, clusters, (heads, nqb))
    for h in range(heads):
        support = np.array_split(rng.permutation(nkb), clusters)
        for r in range(nqb):
            row = rng.random(nkb) < 0.02
            row[support[lab[h, r]]] |= rng.random(len(support[lab[h, r]])) < 0.6
            mask[h * nqb + r] = row
    return mask, lab


def _run(idx, cnt, nkb, x0, iters):
    heads, nqb = x0.shape[:2]
    order = torch.empty((heads, nqb), dtype=torch.int32, device=DEV)
    x_out = torch.empty((heads, nqb, 2), dtype=torch.float32, device=DEV)
    ang = torch.empty((heads, nqb), dtype=torch.float32, device=DEV)
    bsa.spectral_order(cuda(idx), cuda(cnt), nkb, cuda(x0.astype(np.float32)), order,
                       x_out=x_out, angle=ang, iters=iters)
    status_ok()
    return x_out.cpu().numpy(), ang.cpu().numpy(), order.cpu().numpy()


def _check(idx, cnt, nkb, x0, iters, x_tol=2e-3):
    X, ang, order = _run(idx, cnt, nkb, x0, iters)
    Xr, angr, orderr = oracle.spectral_order(idx, cnt, nkb, x0, iters)
    heads, nqb = x0.shape[:2]
    for h in range(heads):
        assert sorted(order[h]) == list(range(nqb))
        # the order is exactly the sort of the kernel's own angles (ties: lower row)
        key = np.lexsort((np.arange(nqb), ang[h]))
        assert np.array_equal(order[h], key)
        # the embedding matches the fp64 iteration (relative to the vectors' scale)
        scale = np.abs(Xr[h]).max()
        assert np.abs(X[h] - Xr[h]).max() <= x_tol * scale
        # the oracle's angles along the kernel's order only step back where the
        # two angles of a row disagree within the fp32 error
        d = np.diff(angr[h][order[h]])
        assert np.all(d >= -2e-3), d.min()


def test_planted_clusters_match_oracle():
    mask, _ = _planted(1, 3, 700, 600, 4)
    idx, cnt, _ = oracle.index_mask(mask)
    x0 = synth.spectral_start(3, 3, 700)
    _check(idx, cnt, 600, x0, iters=10)


def test_dynamic_workload_lists_match_oracle():
    prob = synth.dynamic(seed=5, H=2)      # 928 query blocks, top-k lists of 93..185
    idx_t, cnt_t, _ = gpu_index(prob)
    idx, cnt = idx_t.cpu().numpy(), cnt_t.cpu().numpy()
    ridx, rcnt, _ = oracle.index_topk(prob.scores, prob.k_per_row, max_kv=idx.shape[1])
    assert np.array_equal(idx, ridx)       # lists bit-exact first
    x0 = synth.spectral_start(4, 2, prob.nqb)
    _check(ridx, rcnt, prob.nqb, x0, iters=10)


def test_spectral_then_wave_sort_is_a_valid_schedule_and_result_is_unchanged():
    prob = synth.tiny(seed=12, H=2, N=4096, D=128, density=0.2)
    idx, cnt, _ = gpu_index(prob)
    x0 = torch.from_numpy(synth.spectral_start(5, 2, prob.nqb)).float().to(DEV)
    spec = torch.empty((2, prob.nqb), dtype=torch.int32, device=DEV)
    bsa.spectral_order(idx, cnt, prob.nqb, x0, spec, iters=8)
    rp = torch.empty_like(spec)
    bsa.reorder_rows(cnt.reshape(2, prob.nqb), 5, rp, order_in=spec)
    ref = oracle.reorder_rows(cnt.reshape(2, prob.nqb).cpu().numpy(), 5, spec.cpu().numpy())
    assert np.array_equal(rp.cpu().numpy(), ref)
    q, k, v = cuda(prob.q), cuda(prob.k), cuda(prob.v)
    o0, l0 = torch.empty_like(q), torch.empty(q.shape[:3], dtype=torch.float32, device=DEV)
    o1, l1 = torch.empty_like(q), torch.empty_like(l0)
    bsa.forward(q, k, v, idx, cnt, o0, l0)
    bsa.forward(q, k, v, idx, cnt, o1, l1, row_perm=rp)
    status_ok()
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
