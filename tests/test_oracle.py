"""Pins for the fp64 oracle: checked against what the pages and the mathematics
fix, never against the oracle itself or the CUDA path.  CPU only."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).to(torch.bfloat16)


def _f64(t):
    return t.to(torch.float64).numpy()


def _all_blocks(rows, nb):
    idx = np.tile(np.arange(nb, dtype=np.int32), (rows, 1))
    return idx, np.full(rows, nb, np.int32)


def _by_token(O, L, tok, N):
    """Scatter oracle rows (one head) back to token order."""
    o = np.empty_like(O)
    lse = np.empty_like(L)
    o[tok] = O
    lse[tok] = L
    return o, lse


# --------------------------------------------------------------------------
# Dense softmax path: an all-ones mask is dense attention (InstaGen eq. 2),
# computed here separately in matrix form with numpy.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("D", [16, 64])
def test_all_ones_mask_is_dense_softmax_attention(D):
    B, H, N = 1, 2, 384
    q, k, v = (_bf16((B, H, N, D), s) for s in (1, 2, 3))
    nb = N // 128
    idx, cnt = _all_blocks(B * H * nb, nb)
    O, L, tok = oracle.attention(q, k, v, idx, cnt)
    for h in range(H):
        Q, K, V = _f64(q[0, h]), _f64(k[0, h]), _f64(v[0, h])
        logits = Q @ K.T / math.sqrt(D)
        mx = logits.max(1, keepdims=True)
        z = np.exp(logits - mx).sum(1, keepdims=True)
        ref_o = (np.exp(logits - mx) / z) @ V
        ref_l = (mx + np.log(z))[:, 0]
        sl = slice(h * N, (h + 1) * N)
        o, lse = _by_token(O[sl], L[sl], tok[sl], N)
        np.testing.assert_allclose(o, ref_o, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, ref_l, rtol=0, atol=1e-12)


def test_caller_scale_is_the_logit_factor():
    """A caller-given scale c replaces 1/sqrt(D): dense softmax(c Q K^T) V in
    matrix form; the default equals c = 1/sqrt(D) exactly."""
    B, H, N, D = 1, 1, 256, 32
    q, k, v = (_bf16((B, H, N, D), s) for s in (4, 5, 6))
    idx, cnt = _all_blocks(2, 2)
    Q, K, V = _f64(q[0, 0]), _f64(k[0, 0]), _f64(v[0, 0])
    for c in (0.05, 0.5):
        O, L, tok = oracle.attention(q, k, v, idx, cnt, scale=c)
        o, lse = _by_token(O, L, tok, N)
        logits = c * (Q @ K.T)
        mx = logits.max(1, keepdims=True)
        z = np.exp(logits - mx).sum(1, keepdims=True)
        np.testing.assert_allclose(o, (np.exp(logits - mx) / z) @ V, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, (mx + np.log(z))[:, 0], rtol=0, atol=1e-12)
    O0, L0, _ = oracle.attention(q, k, v, idx, cnt)
    O1, L1, _ = oracle.attention(q, k, v, idx, cnt, scale=1.0 / math.sqrt(D))
    assert np.array_equal(O0, O1) and np.array_equal(L0, L1)


def test_block_of_identical_keys_gives_its_value_exactly():
    """All 128 keys of the only listed block equal k and all values equal v:
    O = v and LSE = q.k*scale + ln 128 (closed form; fp64 rounding of the
    128 equal weights 1/128 is the only error)."""
    N, D = 256, 32
    q = _bf16((1, 1, N, D), 5)
    k = torch.zeros((1, 1, N, D), dtype=torch.bfloat16)
    v = torch.zeros((1, 1, N, D), dtype=torch.bfloat16)
    krow, vrow = _bf16((D,), 6), _bf16((D,), 7)
    k[0, 0, 128:] = krow
    v[0, 0, 128:] = vrow
    idx = np.array([[1], [1]], np.int32)
    cnt = np.array([1, 1], np.int32)
    O, L, tok = oracle.attention(q, k, v, idx, cnt)
    np.testing.assert_allclose(O, np.broadcast_to(_f64(vrow), O.shape), rtol=1e-14, atol=0)
    s = _f64(q[0, 0])[tok] @ _f64(krow) / math.sqrt(D)
    np.testing.assert_allclose(L, s + math.log(128), rtol=0, atol=1e-12)


def test_empty_list_gives_zero_output_and_minus_inf_lse():
    q, k, v = (_bf16((1, 1, 256, 16), s) for s in (1, 2, 3))
    idx = np.array([[0], [0]], np.int32)
    cnt = np.array([0, 1], np.int32)
    O, L, _ = oracle.attention(q, k, v, idx, cnt)
    assert np.all(O[:128] == 0) and np.all(np.isneginf(L[:128]))
    assert np.all(np.isfinite(L[128:]))


# --------------------------------------------------------------------------
# Log-weights (InstaGen Algorithm 1 step 14: softmax(l + log w)).
# --------------------------------------------------------------------------
def test_log_weights_zero_is_unweighted_and_constant_shifts_lse_only():
    p = synth.tiny(seed=11, H=2, N=512, D=32)
    idx, cnt, _ = oracle.index_mask(p.mask)
    O0, L0, _ = oracle.attention(p.q, p.k, p.v, idx, cnt)
    Oz, Lz, _ = oracle.attention(p.q, p.k, p.v, idx, cnt, log_w=np.zeros(idx.shape, np.float32))
    np.testing.assert_array_equal(Oz, O0)
    np.testing.assert_array_equal(Lz, L0)
    c = np.float32(1.75)
    Oc, Lc, _ = oracle.attention(p.q, p.k, p.v, idx, cnt, log_w=np.full(idx.shape, c, np.float32))
    np.testing.assert_allclose(Oc, O0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(Lc, L0 + float(c), rtol=0, atol=1e-12)


def test_log_weight_is_a_multiplicative_key_weight():
    """Weight w on one block equals repeating that block's keys w times
    (integer w = 2: list the block twice, unweighted)."""
    q, k, v = (_bf16((1, 1, 384, 16), s) for s in (21, 22, 23))
    idx_w = np.array([[0, 2]] * 3, np.int32)
    lw = np.array([[math.log(2.0), 0.0]] * 3, np.float32)
    cnt = np.full(3, 2, np.int32)
    Ow, Lw, _ = oracle.attention(q, k, v, idx_w, cnt, log_w=lw)
    idx_r = np.array([[0, 0, 2]] * 3, np.int32)
    Or, Lr, _ = oracle.attention(q, k, v, idx_r, np.full(3, 3, np.int32))
    # log(2) in fp32 is not exactly ln 2: allow its rounding (~1e-8 relative)
    np.testing.assert_allclose(Ow, Or, rtol=0, atol=1e-7)
    np.testing.assert_allclose(Lw, Lr, rtol=0, atol=1e-7)


# --------------------------------------------------------------------------
# Index maps and row permutation (INTRA CQS maps; WaveAlign: permuting query
# rows and mask rows, then restoring, leaves the result unchanged).
# --------------------------------------------------------------------------
def test_maps_equal_physically_gathered_tensors():
    B, H, N, D = 1, 2, 512, 32
    q, k, v = (_bf16((B, H, N, D), s) for s in (31, 32, 33))
    g = np.random.default_rng(0)
    qm = np.stack([g.permutation(N) for _ in range(H)]).astype(np.int32)
    km = np.stack([g.permutation(N) for _ in range(H)]).astype(np.int32)
    nb = N // 128
    mask = (g.random((H * nb, nb)) < 0.5).astype(np.uint8)
    mask[:, 0] = 1
    idx, cnt, _ = oracle.index_mask(mask)
    O, L, tok = oracle.attention(q, k, v, idx, cnt, q_map=qm, kv_map=km)
    qg = torch.stack([q[0, h][torch.from_numpy(qm[h]).long()] for h in range(H)])[None]
    kg = torch.stack([k[0, h][torch.from_numpy(km[h]).long()] for h in range(H)])[None]
    vg = torch.stack([v[0, h][torch.from_numpy(km[h]).long()] for h in range(H)])[None]
    Og, Lg, tokg = oracle.attention(qg, kg, vg, idx, cnt)
    for h in range(H):
        sl = slice(h * N, (h + 1) * N)
        o1, l1 = _by_token(O[sl], L[sl], tok[sl], N)
        # gathered row p is token qm[h][p]
        o2 = np.empty_like(o1)
        l2 = np.empty_like(l1)
        o2[qm[h][tokg[sl]]] = Og[sl]
        l2[qm[h][tokg[sl]]] = Lg[sl]
        np.testing.assert_array_equal(o1, o2)
        np.testing.assert_array_equal(l1, l2)


def test_permuting_query_blocks_and_mask_rows_then_restoring_is_identity():
    p = synth.tiny(seed=41, H=1, N=1024, D=32)
    nb = p.nqb
    idx, cnt, _ = oracle.index_mask(p.mask)
    O, L, tok = oracle.attention(p.q, p.k, p.v, idx, cnt)
    perm = np.random.default_rng(3).permutation(nb)
    # physically permute query blocks and the matching mask rows
    qp = p.q.reshape(1, 1, nb, 128, p.D)[:, :, torch.from_numpy(perm)].reshape(p.q.shape)
    idx_p, cnt_p = idx[perm], cnt[perm]
    Op, Lp, _ = oracle.attention(qp, p.k, p.v, idx_p, cnt_p)
    # restore: permuted block i holds original block perm[i]
    inv = np.empty(nb, np.int64)
    inv[perm] = np.arange(nb)
    Or = Op.reshape(nb, 128, p.D)[inv].reshape(O.shape)
    Lr = Lp.reshape(nb, 128)[inv].reshape(L.shape)
    np.testing.assert_array_equal(Or, O)
    np.testing.assert_array_equal(Lr, L)


# --------------------------------------------------------------------------
# Index lists.
# --------------------------------------------------------------------------
def test_topk_toy_example_from_the_page():
    lines = [l.split() for l in open(os.path.join(GOLD, "topk_toy_mcsparse.txt"))
             if l.strip() and not l.startswith("#")]
    scores = np.zeros((1, 8), np.float32)
    for l in lines:
        if l[0].isdigit():
            scores[0, int(l[0]) - 1] = float(l[1])
        elif l[0] == "k":
            k = int(l[1])
        elif l[0] == "expected":
            expected = [int(x) for x in l[1:]]
    idx, cnt, ov = oracle.index_topk(scores, k)
    assert ov == 0 and cnt[0] == k
    assert [int(x) + 1 for x in idx[0, :k]] == expected


def test_topk_matches_rank_counting_brute_force_with_ties():
    g = np.random.default_rng(7)
    for trial in range(200):
        nkb = int(g.integers(1, 40))
        s = g.integers(0, 5, size=(1, nkb)).astype(np.float32)  # many ties
        if trial % 3 == 0:
            s = -s
        k = int(g.integers(0, nkb + 3))
        idx, cnt, ov = oracle.index_topk(s, k, max_kv=nkb)
        # brute force: kb is kept iff fewer than k blocks beat it
        # (a higher score, or an equal score at a lower block index)
        keep = []
        for kb in range(nkb):
            beat = sum(1 for j in range(nkb)
                       if s[0, j] > s[0, kb] or (s[0, j] == s[0, kb] and j < kb))
            if beat < k:
                keep.append(kb)
        assert ov == 0
        assert cnt[0] == len(keep) and list(idx[0, :cnt[0]]) == keep


def test_threshold_is_inclusive_and_compared_in_fp32():
    p = 0.15  # fp64; the comparison uses fp32(0.15)
    p32 = np.float32(p)
    T = np.array([[p32, np.nextafter(p32, np.float32(1)), np.float32(0.0), np.float32(1.0),
                   np.nextafter(p32, np.float32(0))]], np.float32)
    idx, cnt, ov = oracle.index_threshold(T, p)
    assert ov == 0 and cnt[0] == 3 and list(idx[0, :3]) == [0, 2, 4]


def test_index_overflow_truncates_and_is_counted():
    mask = np.ones((3, 10), np.uint8)
    mask[1, 5:] = 0
    idx, cnt, ov = oracle.index_mask(mask, max_kv=6)
    assert ov == 2
    assert list(cnt) == [6, 5, 6]
    assert list(idx[0]) == [0, 1, 2, 3, 4, 5]
    assert list(idx[1]) == [0, 1, 2, 3, 4, -1]


# --------------------------------------------------------------------------
# Row reordering (WaveAlign stage 2).
# --------------------------------------------------------------------------
def test_reorder_hand_worked_example():
    vals = {}
    for l in open(os.path.join(GOLD, "reorder_stage2_example.txt")):
        if l.strip() and not l.startswith("#"):
            f = l.split()
            vals[f[0]] = [int(x) for x in f[1:]]
    perm = oracle.reorder_rows(np.array([vals["cnt"]], np.int32), vals["wave"][0])
    assert list(perm[0]) == vals["expected"]


@pytest.mark.parametrize("wave", [1, 5, 7, 64, 1000])
def test_reorder_properties(wave):
    g = np.random.default_rng(wave)
    heads, nqb = 3, 53
    cnt = g.integers(0, 9, size=(heads, nqb)).astype(np.int32)
    order = np.stack([g.permutation(nqb) for _ in range(heads)]).astype(np.int32)
    for order_in in (None, order):
        perm = oracle.reorder_rows(cnt, wave, order_in)
        base = np.tile(np.arange(nqb), (heads, 1)) if order_in is None else order_in
        for h in range(heads):
            assert sorted(perm[h]) == list(range(nqb))
            for b0 in range(0, nqb, wave):
                b = perm[h, b0:b0 + wave]
                src = list(base[h, b0:b0 + wave])
                assert sorted(b) == sorted(src)           # same rows stay in the wave
                c = cnt[h, b]
                assert np.all(c[:-1] >= c[1:])            # descending counts
                for i in range(len(b) - 1):               # ties keep input order
                    if c[i] == c[i + 1]:
                        assert src.index(b[i]) < src.index(b[i + 1])


# --------------------------------------------------------------------------
# Exact set + PPSWOR sample (InstaGen section 3.2.1).
# --------------------------------------------------------------------------
def _pi_by_bisection(s, m):
    """Independent solve of sum min(1, lam*s) = m by bisection."""
    lo, hi = 0.0, 1.0
    while np.minimum(1.0, hi * s).sum() < m:
        hi *= 2
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if np.minimum(1.0, mid * s).sum() < m:
            lo = mid
        else:
            hi = mid
    return np.minimum(1.0, hi * s)


def _sample_many(scores_row, exact, m, n_draws, seed):
    nkb = scores_row.shape[0]
    S = np.repeat(scores_row[None], n_draws, 0)
    ex = np.tile(np.array(exact, np.int32), (n_draws, 1)) if exact else np.zeros((n_draws, 1), np.int32)
    ec = np.full(n_draws, len(exact), np.int32)
    u = np.random.default_rng(seed).random(n_draws)
    return oracle.sample_blocks(S, ex, ec, m, u, max_kv=nkb)


def test_sample_size_inclusion_probabilities_and_promotion():
    g = np.random.default_rng(5)
    nkb, m = 40, 6
    s = g.random(nkb).astype(np.float32) + np.float32(0.01)
    s[7] = np.float32(30.0)  # large enough that its pi is capped at 1 (promoted)
    exact = [2, 11, 30]
    n = 40000
    idx, cnt, lw, ov = _sample_many(s, exact, m, n, 1)
    assert ov == 0
    assert np.all(cnt == len(exact) + m)  # exactly m drawn or promoted blocks per row
    resid = np.array([j for j in range(nkb) if j not in exact])
    pi = _pi_by_bisection(s[resid].astype(np.float64), m)
    assert pi[list(resid).index(7)] == 1.0
    freq = np.zeros(nkb)
    for r in range(n):
        freq[idx[r, :cnt[r]]] += 1
    freq /= n
    assert np.all(freq[exact] == 1.0) and freq[7] == 1.0
    # empirical inclusion frequency -> pi (4 sigma)
    sd = np.sqrt(pi * (1 - pi) / n) + 1e-12
    assert np.all(np.abs(freq[resid] - pi) <= 4 * sd + 1e-9)
    # weights: exact and promoted 0, sampled -log(pi)
    for r in range(50):
        for e in range(cnt[r]):
            j = idx[r, e]
            if j in exact or j == 7:
                assert lw[r, e] == 0.0
            else:
                assert lw[r, e] == pytest.approx(-math.log(pi[list(resid).index(j)]), rel=1e-6)


def _pps_cases():
    cases, cur = [], None
    for line in open(os.path.join(GOLD, "sampler_systematic_pps_example.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, _, rest = line.partition(" ")
        if key == "case":
            cur = {"name": rest}
            cases.append(cur)
        else:
            cur[key] = rest.split()
    return cases


@pytest.mark.parametrize("case", _pps_cases(), ids=lambda c: c["name"])
def test_sampler_hand_worked_draws(case):
    """Single rows worked by hand: which blocks the points u + i select, the
    capped block kept at weight 1, the whole residual kept when the budget
    covers it, and the uniform sampler."""
    from fractions import Fraction
    if "uniform" in case:
        scores, nkb = None, int(case["uniform"][0])
    else:
        scores = np.array([[float(x) for x in case["scores"]]], np.float32)
        nkb = scores.shape[1]
    exact = [int(x) for x in case.get("exact", [])]
    ex = np.array([exact or [0]], np.int32)
    ec = np.array([len(exact)], np.int32)
    u = np.array([float(case["u"][0])])
    idx, cnt, lw, ov = oracle.sample_blocks(scores, ex, ec, int(case["m"][0]), u, nkb, nkb=nkb)
    blocks = [int(x) for x in case["blocks"]]
    assert ov == 0 and cnt[0] == len(blocks)
    assert list(idx[0, :cnt[0]]) == blocks
    assert np.all(idx[0, cnt[0]:] == -1)
    for e, f in enumerate(case["pi"]):
        pi = Fraction(f)
        if pi == 1:
            assert lw[0, e] == 0.0
        else:
            assert lw[0, e] == pytest.approx(-math.log(float(pi)), rel=1e-6)


def test_horvitz_thompson_estimate_is_unbiased():
    g = np.random.default_rng(9)
    nkb, m = 30, 5
    s = (g.random(nkb) + 0.05).astype(np.float32)
    y = g.random(nkb) * (1 + 3 * s)  # roughly proportional to the score
    exact = [0, 4]
    n = 20000
    idx, cnt, lw, _ = _sample_many(s, exact, m, n, 2)
    est = np.array([np.sum(y[idx[r, :cnt[r]]] * np.exp(lw[r, :cnt[r]].astype(np.float64)))
                    for r in range(n)])
    sigma = est.std(ddof=1)
    assert abs(est.mean() - y.sum()) <= 4 * sigma / math.sqrt(n)


def test_sampled_attention_sums_are_unbiased():
    """exp(LSE) = z_hat and exp(LSE)*O = n_hat average to the dense z and n
    (InstaGen: E z_hat = z, E n_hat = n)."""
    N, D, nb = 1024, 16, 8
    q, k, v = (_bf16((1, 1, N, D), s) for s in (61, 62, 63))
    Od, Ld, tokd = oracle.attention(q, k, v, *_all_blocks(nb, nb), sel=np.array([0]))
    z = np.exp(Ld)
    nvec = z[:, None] * Od
    g = np.random.default_rng(4)
    s = (g.random(nb) + 0.1).astype(np.float32)
    n_draws = 3000
    S = np.repeat(s[None], n_draws, 0)
    u = g.random(n_draws)
    ex = np.zeros((n_draws, 1), np.int32)
    ec = np.ones(n_draws, np.int32)
    idx, cnt, lw, _ = oracle.sample_blocks(S, ex, ec, 3, u, max_kv=nb)
    zs = np.zeros((n_draws, 128))
    ns = np.zeros((n_draws, 128, D))
    for r in range(n_draws):
        # row r's list is used by query block 0 of a one-block query problem
        O, L, _ = oracle.attention(q, k, v, idx[r:r + 1], cnt[r:r + 1], log_w=lw[r:r + 1],
                                   sel=np.array([0]))
        zs[r] = np.exp(L)
        ns[r] = np.exp(L)[:, None] * O
    for x, ref in ((zs, z), (ns.reshape(n_draws, -1), nvec.reshape(-1))):
        mean, sd = x.mean(0), x.std(0, ddof=1)
        assert np.all(np.abs(mean - ref) <= 4.5 * sd / math.sqrt(n_draws) + 1e-9)


def test_full_budget_recovers_dense_attention():
    N, D, nb = 640, 16, 5
    q, k, v = (_bf16((1, 1, N, D), s) for s in (71, 72, 73))
    Od, Ld, _ = oracle.attention(q, k, v, *_all_blocks(nb, nb))
    s = np.random.default_rng(1).random((nb, nb)).astype(np.float32) + np.float32(0.1)
    ex = np.zeros((nb, 1), np.int32)
    ec = np.ones(nb, np.int32)
    idx, cnt, lw, _ = oracle.sample_blocks(s, ex, ec, nb - 1, np.full(nb, 0.5), max_kv=nb)
    assert np.all(cnt == nb) and np.all(lw == 0)
    O, L, _ = oracle.attention(q, k, v, idx, cnt, log_w=lw)
    np.testing.assert_allclose(O, Od, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L, Ld, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# Scatter / Gather structure (INTRA, Appendix D).
# --------------------------------------------------------------------------
@pytest.mark.parametrize("T", [8, 128])
def test_scatter_gather_overlap_and_two_layer_reachability(T):
    R = T
    N = T * R
    m = synth.scatter_map(N, R)
    assert sorted(m) == list(range(N))
    # Scatter group r = gathered positions r*T .. r*T+T-1 (one token per neighbourhood)
    scat = m.reshape(R, T)
    assert np.all(np.sort(scat // R, axis=1) == np.arange(T))
    assert np.all(scat % R == np.arange(R)[:, None])
    # Gather groups = neighbourhoods G_b = {b*R .. b*R+R-1}
    X = np.zeros((R, T), np.int64)
    for r in range(R):
        for tok in scat[r]:
            X[r, tok // R] += 1
    assert X.min() == T // R == 1 and X.max() == 1
    # two layers (Scatter then Gather) connect every source to every target
    A_s = np.zeros((N, N), bool)
    A_g = np.zeros((N, N), bool)
    if N <= 64 * 64:
        for r in range(R):
            A_s[np.ix_(scat[r], scat[r])] = True
        for b in range(T):
            A_g[b * R:(b + 1) * R, b * R:(b + 1) * R] = True
        reach = (A_g.astype(np.int64) @ A_s.astype(np.int64)) > 0
        assert reach.all()
        # Scatter keeps N^2 / R pairs
        assert A_s.sum() == N * N // R


# --------------------------------------------------------------------------
# Effective FLOP accounting (host logic of the product; pinned to the
# FLOP columns INTRA prints).
# --------------------------------------------------------------------------
def test_flop_formula_reproduces_printed_gflops():
    from long_context_mask_gb300 import dense_attention_flops
    for l in open(os.path.join(GOLD, "flops_intra_table1.txt")):
        if not l.strip() or l.startswith("#"):
            continue
        N, H, D, causal, groups, gf = l.split()
        f = dense_attention_flops(int(N), int(H), int(D), causal=bool(int(causal)))
        f /= int(groups)
        assert abs(f / 1e9 - float(gf)) <= 0.05, (l, f / 1e9)


# --------------------------------------------------------------------------
# Spectral row order (WaveAlign section IV-C): matrix-free centered subspace
# iteration, checked against numpy's SVD of the explicitly centered mask.
# --------------------------------------------------------------------------
def _lists_from_mask(mask):
    idx, cnt, _ = oracle.index_mask(mask)
    return idx, cnt


def _planted_mask(rng, heads, nqb, nkb, clusters, p_in=0.6, p_out=0.03):
    mask = np.zeros((heads, nqb, nkb), np.uint8)
    lab = np.zeros((heads, nqb), np.int64)
    for h in range(heads):
        cols = rng.permutation(nkb)
        support = np.array_split(cols, clusters)
        lab[h] = rng.integers(0, clusters, nqb)
        for r in range(nqb):
            row = rng.random(nkb) < p_out
            row[support[lab[h, r]]] |= rng.random(len(support[lab[h, r]])) < p_in
            row[r % nkb] = True
            mask[h, r] = row
    return mask, lab


def test_spectral_subspace_matches_svd_of_centered_mask():
    rng = np.random.default_rng(21)
    heads, nqb, nkb = 2, 96, 80
    mask, _ = _planted_mask(rng, heads, nqb, nkb, clusters=3)
    idx, cnt = _lists_from_mask(mask.reshape(heads * nqb, nkb))
    x0 = rng.standard_normal((heads, nqb, 2))
    X, ang, order = oracle.spectral_order(idx, cnt, nkb, x0, iters=300)
    for h in range(heads):
        A = mask[h].astype(np.float64)
        Ac = A - A.mean(0, keepdims=True)          # centered by the mean row
        U, S, _ = np.linalg.svd(Ac, full_matrices=False)
        assert S[1] > 1.05 * S[2]                  # a spectral gap to converge to
        cos = np.linalg.svd(U[:, :2].T @ X[h], compute_uv=False)
        assert cos.min() > 1 - 1e-8
        np.testing.assert_allclose(X[h].T @ X[h], np.eye(2), atol=1e-12)   # orthonormal
        np.testing.assert_allclose(X[h].sum(0), 0.0, atol=1e-9)            # orthogonal to 1


def test_spectral_order_groups_planted_clusters_and_is_a_permutation():
    rng = np.random.default_rng(5)
    heads, nqb, nkb = 3, 120, 100
    mask, lab = _planted_mask(rng, heads, nqb, nkb, clusters=3, p_in=0.7, p_out=0.01)
    idx, cnt = _lists_from_mask(mask.reshape(heads * nqb, nkb))
    x0 = rng.standard_normal((heads, nqb, 2))
    X, ang, order = oracle.spectral_order(idx, cnt, nkb, x0, iters=15)  # the page's 5-15
    for h in range(heads):
        assert sorted(order[h]) == list(range(nqb))
        seq = lab[h][order[h]]
        # each cluster occupies one circular run of the order
        changes = int(np.sum(seq != np.roll(seq, 1)))
        assert changes <= 3, (h, changes)
        assert np.all(np.diff(ang[h][order[h]]) >= 0)


def test_spectral_order_is_equivariant_under_row_relabelling():
    rng = np.random.default_rng(8)
    nqb, nkb = 64, 50
    mask, _ = _planted_mask(rng, 1, nqb, nkb, clusters=2)
    perm = rng.permutation(nqb)
    x0 = rng.standard_normal((1, nqb, 2))
    idx, cnt = _lists_from_mask(mask[0])
    X, ang, order = oracle.spectral_order(idx, cnt, nkb, x0, iters=10)
    idx_p, cnt_p = _lists_from_mask(mask[0][perm])
    Xp, angp, orderp = oracle.spectral_order(idx_p, cnt_p, nkb, x0[:, perm], iters=10)
    np.testing.assert_allclose(Xp[0], X[0][perm], atol=1e-10)
    np.testing.assert_allclose(angp[0], ang[0][perm], atol=1e-10)


def test_spectral_angle_and_ties_to_the_lower_row():
    """Identical mask rows get identical embeddings and angles; the order
    lists such rows by ascending query block.  The angle is the polar angle
    of the row's two coordinates, atan2(second, first)."""
    rng = np.random.default_rng(13)
    nqb, nkb = 40, 30
    mask, _ = _planted_mask(rng, 1, nqb, nkb, clusters=2)
    m = mask[0].copy()
    for dst, src in ((7, 3), (25, 3), (31, 12), (2, 12)):
        m[dst] = m[src]
    idx, cnt = _lists_from_mask(m)
    x0 = rng.standard_normal((1, nqb, 2))
    X, ang, order = oracle.spectral_order(idx, cnt, nkb, x0, iters=12)
    np.testing.assert_allclose(ang[0], np.arctan2(X[0][:, 1], X[0][:, 0]), rtol=0, atol=1e-12)
    assert ang[0][3] == ang[0][7] == ang[0][25] and ang[0][2] == ang[0][12] == ang[0][31]
    pos = {int(r): s for s, r in enumerate(order[0])}
    assert pos[3] < pos[7] < pos[25] and pos[2] < pos[12] < pos[31]
    assert [pos[r] for r in (3, 7, 25)] == list(range(pos[3], pos[3] + 3))


# --------------------------------------------------------------------------
# Block scores from block means (MC-Sparse mean-pooled score; InstaGen
# centroid score exp(q_g . k_c / sqrt d)).
# --------------------------------------------------------------------------
def test_block_scores_closed_form_for_constant_blocks_and_attention_logit():
    """Blocks whose 128 rows are all equal have means equal to that row, so the
    score is the scaled dot product; with one listed block of identical keys
    the attention oracle's LSE is that logit + ln 128 (an independent path)."""
    N, D = 384, 32
    rng = np.random.default_rng(3)
    a = torch.from_numpy(rng.standard_normal((3, D))).to(torch.bfloat16)
    b = torch.from_numpy(rng.standard_normal((3, D))).to(torch.bfloat16)
    q = a.repeat_interleave(128, 0)[None, None]
    k = b.repeat_interleave(128, 0)[None, None]
    S = oracle.block_scores(q, k)
    ref = _f64(a) @ _f64(b).T / math.sqrt(D)
    np.testing.assert_allclose(S, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(oracle.block_scores(q, k, mode=1), np.exp(ref), rtol=1e-12)
    v = torch.zeros_like(k)
    idx = np.array([[2], [0], [1]], np.int32)
    O, L, tok = oracle.attention(q, k, v, idx, np.ones(3, np.int32))
    for qb, kb in enumerate([2, 0, 1]):
        np.testing.assert_allclose(L[qb * 128:(qb + 1) * 128], S[qb, kb] + math.log(128), atol=1e-12)


def test_block_scores_ignore_order_inside_a_block_and_follow_maps():
    B, H, N, D = 1, 2, 512, 16
    q, k = _bf16((B, H, N, D), 41), _bf16((B, H, N, D), 42)
    rng = np.random.default_rng(4)
    # permuting tokens inside each block leaves the means, hence the scores, unchanged
    within = np.stack([np.concatenate([blk * 128 + rng.permutation(128) for blk in range(N // 128)])
                       for _ in range(H)]).astype(np.int32)
    np.testing.assert_allclose(oracle.block_scores(q, k, q_map=within, kv_map=within),
                               oracle.block_scores(q, k), rtol=0, atol=1e-12)
    # maps equal scoring the physically gathered tensors: query groups follow
    # q_map and key clusters kv_map, two independent maps
    perm = np.stack([rng.permutation(N) for _ in range(H)]).astype(np.int32)
    perm_k = np.stack([rng.permutation(N) for _ in range(H)]).astype(np.int32)
    qg = torch.stack([q[0, h][torch.from_numpy(perm[h]).long()] for h in range(H)])[None]
    kg = torch.stack([k[0, h][torch.from_numpy(perm_k[h]).long()] for h in range(H)])[None]
    np.testing.assert_allclose(oracle.block_scores(q, k, q_map=perm, kv_map=perm_k),
                               oracle.block_scores(qg, kg), rtol=0, atol=1e-12)


def test_uniform_sampler_inclusion_and_weights():
    """No scores: every residual block has pi = m / |R| (InstaGen Alg. 1 steps 6-8)."""
    nkb, m, n = 30, 4, 20000
    exact = [3, 17]
    ex = np.tile(np.array(exact, np.int32), (n, 1))
    ec = np.full(n, len(exact), np.int32)
    u = np.random.default_rng(6).random(n)
    idx, cnt, lw, ov = oracle.sample_blocks(None, ex, ec, m, u, max_kv=nkb, nkb=nkb)
    assert ov == 0 and np.all(cnt == len(exact) + m)
    pi = m / (nkb - len(exact))
    freq = np.zeros(nkb)
    for r in range(n):
        freq[idx[r, :cnt[r]]] += 1
    freq /= n
    resid = [j for j in range(nkb) if j not in exact]
    assert np.all(np.abs(freq[resid] - pi) <= 4 * math.sqrt(pi * (1 - pi) / n))
    drawn = ~np.isin(idx[:, :cnt[0]], exact)
    assert np.allclose(lw[:, :cnt[0]][drawn], -math.log(pi), rtol=1e-6)


# --------------------------------------------------------------------------
# CRM rows and eq. (7) upscaling (ScalingAttention sections 7.1-7.2).
# --------------------------------------------------------------------------
def test_crm_rows_encode_the_same_blocks_as_the_lists():
    g = np.random.default_rng(12)
    mask = (g.random((50, 75)) < 0.3).astype(np.uint8)
    words = oracle.crm_rows(mask)
    assert words.shape == (50, 3)
    idx, cnt, _ = oracle.index_mask(mask)
    for r in range(50):
        bits = [32 * w + i for w in range(3) for i in range(32) if (int(words[r, w]) >> i) & 1]
        assert bits == list(idx[r, :cnt[r]])
    T = g.random((50, 75)).astype(np.float32)
    np.testing.assert_array_equal(oracle.crm_rows(T, 0.4), oracle.crm_rows((T <= np.float32(0.4)).astype(np.uint8)))


def test_upscale_hand_worked_example():
    lines = [l.split() for l in open(os.path.join(GOLD, "upscale_eq7_example.txt"))
             if l.strip() and not l.startswith("#")]
    ub, vb = int(lines[0][1]), int(lines[0][2])
    base = np.array([[int(x) for x in l] for l in lines[1:1 + ub]], np.float32)
    ut, vt = int(lines[1 + ub][1]), int(lines[1 + ub][2])
    exp = np.array([[int(x) for x in l] for l in lines[3 + ub:3 + ub + ut]])
    # a 0/1 mask as a threshold map: active blocks get T = 0, others T = 1; keep T <= 0.5
    T = np.where(base > 0, 0.0, 1.0).astype(np.float32)[None]
    out = oracle.upscale_threshold(T, ut, vt)[0]
    np.testing.assert_array_equal((out <= 0.5).astype(int), exp)


def test_upscale_is_identity_at_scale_one_and_conservative_for_every_threshold():
    g = np.random.default_rng(13)
    T = g.random((2, 9, 11)).astype(np.float32)
    np.testing.assert_array_equal(oracle.upscale_threshold(T, 9, 11), T)
    out = oracle.upscale_threshold(T, 23, 30)
    for p in (0.1, 0.3, 0.7):
        # conservative: every target block whose nearest-lower base block is
        # active stays active; and never more active than the 2x2 neighbourhood
        for h in range(2):
            for u in range(23):
                for v in range(30):
                    i0, j0 = u * 9 // 23, v * 11 // 30
                    if T[h, i0, j0] <= p:
                        assert out[h, u, v] <= p
                    nb = T[h, i0:min(i0 + 2, 9), j0:min(j0 + 2, 11)]
                    assert out[h, u, v] >= nb.min()


# --------------------------------------------------------------------------
# Token masks and grouped key/value heads (INTRA: causal masking inside packed
# tiles, sliding windows with sinks, 32 query heads over 8 key/value heads).
# --------------------------------------------------------------------------
def _masked_dense(q, k, v, allowed):
    """Matrix-form softmax attention of one head over an explicit [N, N]
    boolean mask (rows: query tokens, columns: key tokens); fully masked rows
    give O = 0, LSE = -inf."""
    S = (q @ k.T) / math.sqrt(q.shape[1])
    S = np.where(allowed, S, -np.inf)
    mx = S.max(1, keepdims=True)
    safe = np.where(np.isfinite(mx), mx, 0.0)
    P = np.exp(S - safe)
    z = P.sum(1, keepdims=True)
    with np.errstate(invalid="ignore", divide="ignore"):
        O = np.where(z > 0, (P @ v) / np.where(z > 0, z, 1), 0.0)
        L = np.where(z[:, 0] > 0, np.log(np.where(z[:, 0] > 0, z[:, 0], 1)) + safe[:, 0], -np.inf)
    return O, L


def _allowed(N, causal=False, n_valid=0, window=0, sinks=0):
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    a = np.broadcast_to(j < (n_valid if n_valid > 0 else N), (N, N)).copy()
    if causal:
        a &= j <= i
    if window > 0:
        a &= (j > i - window) | (j < sinks)
    return a


@pytest.mark.parametrize("kw", [dict(causal=True), dict(causal=True, window=100, sinks=16),
                                dict(n_valid=300), dict(causal=True, n_valid=333)])
def test_token_mask_all_blocks_equals_matrix_form(kw):
    N, D, nb = 384, 16, 3
    q, k, v = (_bf16((1, 1, N, D), s) for s in (81, 82, 83))
    O, L, tok = oracle.attention(q, k, v, *_all_blocks(nb, nb), **kw)
    o, lse = _by_token(O, L, tok, N)
    Oref, Lref = _masked_dense(_f64(q[0, 0]), _f64(k[0, 0]), _f64(v[0, 0]), _allowed(N, **kw))
    np.testing.assert_allclose(o, Oref, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(Lref))
    fin = np.isfinite(Lref)
    np.testing.assert_allclose(lse[fin], Lref[fin], rtol=0, atol=1e-12)


def test_causal_mask_is_on_original_tokens_under_maps():
    """With every block listed the kept set is every key whatever the maps, so
    causal attention through arbitrary maps equals plain causal attention."""
    N, D, nb = 384, 16, 3
    q, k, v = (_bf16((1, 1, N, D), s) for s in (84, 85, 86))
    g = np.random.default_rng(8)
    qm, km = (g.permutation(N).astype(np.int32)[None] for _ in range(2))
    O, L, tok = oracle.attention(q, k, v, *_all_blocks(nb, nb), q_map=qm, kv_map=km, causal=True)
    o, lse = _by_token(O, L, tok, N)
    Oref, Lref = _masked_dense(_f64(q[0, 0]), _f64(k[0, 0]), _f64(v[0, 0]), _allowed(N, causal=True))
    np.testing.assert_allclose(o, Oref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, Lref, rtol=0, atol=1e-12)


def test_fully_masked_row_is_empty():
    N, D = 384, 16
    q, k, v = (_bf16((1, 1, N, D), s) for s in (87, 88, 89))
    idx = np.array([[2], [2], [1]], np.int32)  # blocks 0, 1 list only a later block
    cnt = np.ones(3, np.int32)
    O, L, tok = oracle.attention(q, k, v, idx, cnt, causal=True)
    assert np.all(np.isneginf(L[:256])) and np.all(O[:256] == 0)
    assert np.all(np.isfinite(L[256:]))


def test_grouped_heads_equal_repeated_heads_and_matrix_form():
    B, H, H_kv, N, D, nb = 2, 4, 2, 256, 16, 2
    q = _bf16((B, H, N, D), 90)
    k, v = _bf16((B, H_kv, N, D), 91), _bf16((B, H_kv, N, D), 92)
    idx, cnt = _all_blocks(B * H * nb, nb)
    O, L, tok = oracle.attention(q, k, v, idx, cnt, causal=True)
    rep = lambda t: t.repeat_interleave(H // H_kv, dim=1)  # noqa: E731
    O2, L2, _ = oracle.attention(q, rep(k), rep(v), idx, cnt, causal=True)
    np.testing.assert_array_equal(O, O2)
    np.testing.assert_array_equal(L, L2)
    # query head 3 of batch 1 reads key/value head 1 of batch 1
    bh = 1 * H + 3
    rows = slice(bh * nb * 128, (bh + 1) * nb * 128)
    o, lse = _by_token(O[rows], L[rows], tok[rows], N)
    Oref, Lref = _masked_dense(_f64(q[1, 3]), _f64(k[1, 1]), _f64(v[1, 1]), _allowed(N, causal=True))
    np.testing.assert_allclose(o, Oref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, Lref, rtol=0, atol=1e-12)
