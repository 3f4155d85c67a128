"""GPU block scores (mean-pooled / centroid) and the uniform sampler vs the oracle."""
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
    bsa.device_status()


def _gpu_scores(prob, mode, q_map=None, kv_map=None):
    out = torch.empty((prob.rows, prob.nqb), dtype=torch.float32, device=DEV)
    bsa.block_scores(cuda(prob.q), cuda(prob.k), out, q_map=cuda(q_map), kv_map=cuda(kv_map),
                     mode=mode)
    status_ok()
    return out.cpu().numpy().astype(np.float64)


def test_mean_pooled_scores_match_oracle_and_select_the_same_blocks():
    prob = synth.dynamic(seed=5, H=2)                # 928 blocks, clustered Q/K
    g = _gpu_scores(prob, bsa.SCORE_MEAN_DOT)
    r = oracle.block_scores(prob.q, prob.k)
    np.testing.assert_allclose(g, r, rtol=1e-5, atol=1e-4)
    # top-k on the two score sets: rows whose k-th / (k+1)-th oracle scores are
    # separated by more than the score error must select the same blocks
    k = prob.k_per_row
    gi, gc, _ = oracle.index_topk(g.astype(np.float32), k)
    ri, rc, _ = oracle.index_topk(r.astype(np.float32), k)
    srt = -np.sort(-r, axis=1)
    gap = srt[np.arange(len(k)), k - 1] - srt[np.arange(len(k)), k]
    err = np.abs(g - r).max()
    clear = gap > 2 * err + 1e-7     # no score error can reorder these rows' k-th boundary
    assert clear.mean() > 0.5
    assert np.array_equal(gi[clear], ri[clear]) and np.array_equal(gc, rc)


def test_centroid_scores_through_maps_match_oracle():
    prob = synth.sampled(seed=4, H=2)                # 592 blocks, random token permutation
    g = _gpu_scores(prob, bsa.SCORE_CENTROID_EXP, prob.q_map, prob.kv_map)
    r = oracle.block_scores(prob.q, prob.k, q_map=prob.q_map, kv_map=prob.kv_map, mode=1)
    np.testing.assert_allclose(g, r, rtol=1e-4, atol=0)
    assert np.all(g > 0)


def test_uniform_sampler_bit_exact():
    rows, nkb, m = 5000, 300, 7
    rng = np.random.default_rng(9)
    ex = np.sort(np.stack([rng.choice(nkb, 12, replace=False) for _ in range(rows)]), 1).astype(np.int32)
    ec = np.full(rows, 12, np.int32)
    u = rng.random(rows)
    cap = 12 + m
    idx = torch.empty((rows, cap), dtype=torch.int32, device=DEV)
    cnt = torch.empty(rows, dtype=torch.int32, device=DEV)
    lw = torch.empty((rows, cap), dtype=torch.float32, device=DEV)
    bsa.sample_blocks(None, cuda(ex), cuda(ec), m, cuda(u), idx, cnt, lw, nkb=nkb)
    ridx, rcnt, rlw, ov = oracle.sample_blocks(None, ex, ec, m, u, cap, nkb=nkb)
    status_ok()
    assert ov == 0 and np.all(rcnt == cap)
    np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
    np.testing.assert_array_equal(cnt.cpu().numpy(), rcnt)
    np.testing.assert_allclose(lw.cpu().numpy(), rlw, rtol=1e-6, atol=0)
