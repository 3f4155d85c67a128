"""The sampler's fp32 decisions against a plain fp64 evaluation (InstaGen
section 3.2.1: eq. (4) inclusion probabilities, systematic PPS).

The oracle (and the GPU sampler, bit for bit) take the draw in fp32: lambda,
pi and the running sums C.  The pages fix no precision.  This test evaluates
the same definition in fp64 on the permuted workload's rows and requires that
every row whose drawn set differs between the two precisions has a point
u + i within fp32 rounding of an interval edge C_j, i.e. that the two
readings part only where rounding decides.
"""
import numpy as np

import oracle
import synth


def _draw_fp64(s, exact, m, u):
    """Blocks drawn by eq. (4) + systematic PPS in fp64; also returns, per
    residual block in ascending order, C_j - u (the edge positions) and a
    bound on their fp32 rounding error."""
    nkb = s.shape[0]
    res = np.setdiff1d(np.arange(nkb), exact)
    sr = s[res].astype(np.float64)
    capped = np.zeros(res.shape[0], bool)
    while True:
        lam = (m - capped.sum()) / sr[~capped].sum()
        grow = (~capped) & (lam * sr >= 1.0)
        if not grow.any():
            break
        capped |= grow
    pi = np.where(capped, 1.0, lam * sr)
    free = ~capped
    c = np.cumsum(pi[free])
    m_free = m - int(capped.sum())
    pos = c - u
    prev = np.concatenate([[-u], pos[:-1]])
    drawn_free = np.flatnonzero(np.ceil(pos) > np.ceil(prev))[:m_free]
    drawn = np.concatenate([res[capped], res[free][drawn_free]])
    # fp32 rounding of the same sums: one ulp per term of C_j, plus lambda's and u's
    n = np.arange(1, c.shape[0] + 1)
    err = (n + 4) * np.spacing(np.float32(max(c[-1], 1.0))).astype(np.float64) + np.spacing(np.float32(1.0))
    return np.sort(drawn), pos, err


def test_fp32_and_fp64_draws_part_only_at_edges():
    prob = synth.sampled(seed=4, H=8)  # the permuted workload's rows (8 of its 40 heads)
    k_exact = prob.k_const
    ex_idx, ex_cnt, _ = oracle.index_topk(prob.scores, k_exact)
    idx, cnt, _, ov = oracle.sample_blocks(prob.scores, ex_idx, ex_cnt, prob.m_sample, prob.u,
                                           k_exact + prob.m_sample)
    assert ov == 0
    differ = 0
    for r in range(prob.rows):
        exact = ex_idx[r, :ex_cnt[r]]
        d64, pos, err = _draw_fp64(prob.scores[r], exact, prob.m_sample, float(prob.u[r]))
        d32 = np.setdiff1d(idx[r, :cnt[r]], exact)
        if np.array_equal(np.sort(d32), d64):
            continue
        differ += 1
        # some edge lies within its rounding error of an integer point
        dist = np.abs(pos - np.round(pos))
        assert (dist <= err).any(), (r, float(dist.min()), float(err.min()))
    # rounding decides rarely: a handful of rows at most
    assert differ <= max(2, prob.rows // 500), differ


def test_fp64_reference_is_the_definition_on_a_worked_row():
    """The fp64 helper on a small row worked by hand: scores 1..6 (blocks 0..5),
    no exact block, m = 2, u = 0.25: lambda = 2 / 21, C = (2, 6, 12, 20, 30,
    42) / 21; block j is drawn when a point u + i lies in (C_{j-1}, C_j]:
    0.25 in (C_0, C_1] = (0.095, 0.286] and 1.25 in (C_3, C_4] = (0.952,
    1.429], so blocks 1 and 4."""
    s = np.arange(1, 7, dtype=np.float32)
    drawn, pos, _ = _draw_fp64(s, np.array([], np.int64), 2, 0.25)
    assert drawn.tolist() == [1, 4]
    np.testing.assert_allclose(pos + 0.25, np.cumsum(np.arange(1, 7)) * 2 / 21)
