"""GPU parity on every row of the small and mid-size workloads, on the
benchmarked dynamic path with pooled scores, and for the documented options
that the other files do not run (a caller-given logit scale, the Gather 0
layer without quadrant masks, packed key tiles over a map longer than N).

Expected values come from the oracle alone: its own index lists, block
scores and Gather 0 key sets.  Tolerances are those of gpu_util.compare
(O max-abs 1e-2, mean-relative 5e-3, LSE 1e-3).
"""
import numpy as np
import pytest
import torch

import long_context_mask_gb300 as bsa
import oracle
import synth
from gpu_util import DEV, LSE_MAX_ABS, O_MAX_ABS, O_MEAN_REL, compare, cuda, run_forward, status_ok

pytestmark = pytest.mark.gpu


def _oracle_lists(prob):
    if prob.diag_list:
        idx, cnt = synth.diag_lists(prob.rows, prob.nqb)
    elif prob.mask is not None:
        idx, cnt, _ = oracle.index_mask(prob.mask)
    else:
        idx, cnt, _ = oracle.index_threshold(prob.T, prob.p)
    return torch.from_numpy(np.ascontiguousarray(idx)).to(DEV), torch.from_numpy(cnt).to(DEV)


def _rows_of_heads(prob, heads):
    return np.concatenate([np.arange(h * prob.nqb, (h + 1) * prob.nqb) for h in heads]).astype(np.int64)


# ------------------------------------------------------------ every row of configs 2 and 3
def test_scatter_layer_every_row_maps_and_geometry():
    """Scatter layer (B1 H24 N16384 D128, T = R = 128): the map path and the
    geometry path, every row of every head against the oracle."""
    prob = synth.scatter(seed=3, layer="scatter")
    idx, cnt = _oracle_lists(prob)
    q, k, v = cuda(prob.q), cuda(prob.k), cuda(prob.v)
    o1, l1 = run_forward(prob, idx, cnt, q=q, k=k, v=v)
    o2, l2 = torch.empty_like(q), torch.empty_like(l1)
    bsa.forward_scatter(q, k, v, 128, idx, cnt, o2, l2)
    torch.cuda.synchronize()
    status_ok()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    compare(prob, o2, l2, idx, cnt)


def test_gather_layer_every_row():
    """Gather layer (the neighbourhoods, no maps): every row of every head."""
    prob = synth.scatter(seed=3, layer="gather")
    idx, cnt = _oracle_lists(prob)
    o, lse = run_forward(prob, idx, cnt)
    status_ok()
    compare(prob, o, lse, idx, cnt)


def test_threshold_workload_two_full_heads():
    """Threshold-map workload (B1 H12 N32768 D128, p = 0.15) with the lists the
    oracle builds: every query block of the first and the last head."""
    prob = synth.threshold(seed=2)
    idx, cnt = _oracle_lists(prob)
    o, lse = run_forward(prob, idx, cnt)
    status_ok()
    compare(prob, o, lse, idx, cnt, sel=_rows_of_heads(prob, [0, prob.B * prob.H - 1]))


# ------------------------------------------------------------ the benchmarked dynamic path
def test_dynamic_workload_pooled_scores_end_to_end():
    """B1 H24 N118784 D128: block scores from Q/K (mean-pooled), per-row top-k,
    the guard's row order and the forward, as the benchmark runs them.  The
    oracle scores the blocks itself in fp64: its top-k lists must equal the
    GPU's on every row whose k-th and (k+1)-th oracle scores are further apart
    than the fp32 score error, and O / LSE must match the oracle (on its own
    lists) on sampled query blocks of the first and last head whose lists
    agree."""
    prob = synth.dynamic(seed=5)
    heads, nqb = prob.B * prob.H, prob.nqb
    q, k, v = cuda(prob.q), cuda(prob.k), cuda(prob.v)
    scores = torch.empty((prob.rows, nqb), dtype=torch.float32, device=DEV)
    ws = torch.empty(bsa.load_library().bsa_block_scores_workspace_size(prob.B, prob.H, prob.N, prob.D),
                     dtype=torch.uint8, device=DEV)
    bsa.block_scores(q, k, scores, workspace=ws)
    kpr = cuda(prob.k_per_row)
    max_kv = int(prob.k_per_row.max())
    idx = torch.empty((prob.rows, max_kv), dtype=torch.int32, device=DEV)
    cnt = torch.empty(prob.rows, dtype=torch.int32, device=DEV)
    bsa.build_index(bsa.IDX_TOPK_F32, scores, idx, cnt, k_per_row=kpr)
    listed = int(cnt.sum().item())
    g = bsa.reorder_guard(heads=heads, nqb=nqb, nkb=nqb, D=prob.D, listed_blocks=listed)
    perm = None
    if g["order"] != "input":
        perm = torch.empty((heads, nqb), dtype=torch.int32, device=DEV)
        bsa.reorder_rows(cnt.view(heads, nqb), bsa.resident_ctas(prob.D), perm)
    o, lse = run_forward(prob, idx, cnt, row_perm=perm, q=q, k=k, v=v)
    status_ok()

    ref_scores = oracle.block_scores(prob.q, prob.k)
    o_idx, o_cnt, _ = oracle.index_topk(ref_scores.astype(np.float32), prob.k_per_row)
    g_idx, g_cnt = idx.cpu().numpy(), cnt.cpu().numpy()
    srt = -np.sort(-ref_scores, axis=1)
    kk = prob.k_per_row.astype(np.int64)
    gap = srt[np.arange(prob.rows), kk - 1] - srt[np.arange(prob.rows), np.minimum(kk, nqb - 1)]
    err = 1e-5 * np.abs(ref_scores).max(axis=1) + 1e-6  # fp32 block means and dot products
    clear = gap > 2 * err
    assert clear.mean() > 0.9
    same = np.array([np.array_equal(g_idx[r, :g_cnt[r]], o_idx[r, :o_cnt[r]]) for r in range(prob.rows)])
    assert same[clear].all(), int((~same[clear]).sum())
    rng = np.random.default_rng(5)
    sel = []
    for h in (0, heads - 1):
        cand = np.flatnonzero(same[h * nqb:(h + 1) * nqb]) + h * nqb
        sel += sorted(rng.choice(cand, 6, replace=False).tolist())
    compare(prob, o, lse, torch.from_numpy(o_idx).to(DEV), torch.from_numpy(o_cnt).to(DEV),
            sel=np.array(sel, np.int64))


# ------------------------------------------------------------ a caller-given logit scale
@pytest.mark.parametrize("scale", [0.05, 0.3])
def test_caller_scale_forward_and_masked(scale):
    """At D = 64, scale 0.3 (2.4 times 1/sqrt(D)) makes each row's softmax peak
    on a few keys, so O sits near single rows of V (|v| up to about 4.5) where
    bf16's half-ulp reaches 2^-7: the few-key bound applies there (it is below
    1e-2 only for |O| < 2)."""
    prob = synth.tiny(seed=61, H=2, N=2048, D=64, density=0.4)
    idx, cnt = _oracle_lists(prob)
    q, k, v = cuda(prob.q), cuda(prob.k), cuda(prob.v)
    o, lse = torch.empty_like(q), torch.empty(q.shape[:3], dtype=torch.float32, device=DEV)
    bsa.forward(q, k, v, idx, cnt, o, lse, scale=scale)
    o2, l2 = torch.empty_like(o), torch.empty_like(lse)
    bsa.forward_masked(q, k, v, idx, cnt, o2, l2, causal=True, scale=scale)
    torch.cuda.synchronize()
    status_ok()
    # the oracle with the same logit factor (InstaGen eq. (1) with the scale supplied)
    O, L, tok = oracle.attention(prob.q, prob.k, prob.v, idx.cpu().numpy(), cnt.cpu().numpy(), scale=scale)
    _check_all(prob, o, lse, O, L, tok, few_keys=scale > 0.2)
    O, L, tok = oracle.attention(prob.q, prob.k, prob.v, idx.cpu().numpy(), cnt.cpu().numpy(), scale=scale,
                                 causal=True)
    _check_all(prob, o2, l2, O, L, tok, few_keys=True)


def _check_all(prob, o, lse, O, L, tok, few_keys=False):
    """All rows (oracle order: query block by query block)."""
    bh = np.repeat(np.arange(prob.rows) // prob.nqb, 128)
    flat = bh * prob.N + tok
    og = o.reshape(-1, prob.D)[torch.from_numpy(flat).to(o.device)].float().cpu().numpy()
    lg = lse.reshape(-1)[torch.from_numpy(flat).to(o.device)].cpu().numpy().astype(np.float64)
    diff = np.abs(og - O)
    bound = 3 * 2.0 ** -8 * float(prob.v.float().abs().max()) if few_keys else O_MAX_ABS
    assert diff.max() <= bound, diff.max()
    assert diff.sum() / np.abs(O).sum() <= O_MEAN_REL
    assert np.array_equal(np.isneginf(lg), np.isneginf(L))
    fin = np.isfinite(L)
    assert np.abs(lg[fin] - L[fin]).max() <= LSE_MAX_ABS


def test_caller_scale_gather0():
    img_h, img_w, n_text, groups = 32, 48, 256, 4
    prob = synth.image_gather0(seed=62, B=1, H=2, img_h=img_h, img_w=img_w, n_text=n_text, groups=groups,
                               D=128)
    _, _, idx, cnt, qm = bsa.gather0_layout(img_h, img_w, n_text, groups, 2)
    q, k, v = cuda(prob.q), cuda(prob.k), cuda(prob.v)
    o, lse = torch.empty_like(q), torch.empty(q.shape[:3], dtype=torch.float32, device=DEV)
    bsa.forward_gather0(q, k, v, img_h, img_w, n_text, groups, idx, cnt, o, lse, quad_mask=qm, scale=0.1)
    torch.cuda.synchronize()
    status_ok()
    O_ref, L_ref = oracle.gather0_attention(prob.q, prob.k, prob.v, img_h, img_w, n_text, groups, scale=0.1)
    _compare_tokens(o, lse, O_ref, L_ref, [0, 1], np.arange(prob.N))


def _compare_tokens(o, lse, O_ref, L_ref, heads, toks):
    og = o.float().cpu().numpy().reshape(-1, o.shape[2], o.shape[3])
    lg = lse.cpu().numpy().reshape(-1, lse.shape[2])
    num = den = 0.0
    for hi, bh in enumerate(heads):
        d = np.abs(og[bh, toks] - O_ref[hi, toks])
        assert d.max() <= O_MAX_ABS, d.max()
        num += d.sum()
        den += np.abs(O_ref[hi, toks]).sum()
        assert np.abs(lg[bh, toks] - L_ref[hi, toks]).max() <= LSE_MAX_ABS
    assert num / den <= O_MEAN_REL


# ------------------------------------------------------------ no quadrant masks
def _tile_keys(img_h, img_w, n_text, groups):
    """Per query tile of the Gather 0 layout, its query tokens and the keys of
    its listed tiles, each tile's tokens once per tile (a token held by two
    listed tiles counts twice).  With no quadrant mask every row of a tile
    sees all of them.  The windows come from the oracle's definition of each
    CQS; which bands a tile pair lists is the layout's documented rule: the two
    8-row bands of each patch's 16-row window, a band both windows share
    listed once.  Text tiles list the text tiles and their groups' tiles."""
    sets = oracle.gather0_sets(img_h, img_w, n_text, groups)
    pw = img_w // 8
    n_img = img_h * img_w // 64
    text = np.arange(n_text, dtype=np.int32)
    tiles = []
    for t in range(n_text // 128):
        qt = np.arange(128 * t, 128 * t + 128, dtype=np.int32)
        per = n_text // groups
        gs = sorted({int(i) // per for i in qt})
        group_keys = [sets[n_img + g][1][sets[n_img + g][1] >= n_text] for g in gs]
        tiles.append((qt, np.concatenate([text] + group_keys)))
    for s in range(img_h // 16):
        for c in range(pw):
            a, b = sets[(2 * s) * pw + c], sets[(2 * s + 1) * pw + c]
            tops, left = set(), None
            for qs, ks in (a, b):
                img = ks[ks >= n_text] - n_text
                top = int((img // img_w).min())
                left = int((img % img_w).min())
                tops |= {top, top + 8}
            bands = [n_text + (y + i) * img_w + left + j for y in sorted(tops) for i in range(8) for j in range(16)]
            tiles.append((np.concatenate([a[0], b[0]]), np.concatenate([text, np.array(bands, np.int32)])))
    return tiles


@pytest.mark.parametrize("img_h,img_w,n_text,groups", [(32, 32, 128, 2), (48, 16, 256, 2), (16, 24, 0, 1)])
def test_gather0_and_packed_without_quadrant_masks(img_h, img_w, n_text, groups):
    """bsa_forward_gather0 with quad_mask = NULL and bsa_forward_packed without a
    quadrant mask over the layout's map (N_kv > N): each query tile attends to
    every key of its listed tiles (a token two listed tiles hold counts
    twice)."""
    H = 2
    prob = synth.image_gather0(seed=63 + img_w, B=1, H=H, img_h=img_h, img_w=img_w, n_text=n_text,
                               groups=groups, D=128)
    q_map, kv_map, idx, cnt, _ = bsa.gather0_layout(img_h, img_w, n_text, groups, H)
    assert kv_map.shape[1] > prob.N
    q, k, v = cuda(prob.q), cuda(prob.k), cuda(prob.v)
    o1, l1 = torch.empty_like(q), torch.empty(q.shape[:3], dtype=torch.float32, device=DEV)
    o2, l2 = torch.empty_like(o1), torch.empty_like(l1)
    bsa.forward_gather0(q, k, v, img_h, img_w, n_text, groups, idx, cnt, o1, l1, quad_mask=None)
    bsa.forward_packed(q, k, v, idx, cnt, kv_map, o2, l2, quad_mask=None, q_map=q_map)
    torch.cuda.synchronize()
    status_ok()
    # the same softmax arithmetic on the same tiles (boxes of the image, or rows
    # copied through the map): bit for bit, and against the oracle
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    _check_tiles(prob, o1, l1, H, img_h, img_w, n_text, groups)


def _check_tiles(prob, o1, l1, H, img_h, img_w, n_text, groups):
    og = o1.float().cpu().numpy().reshape(H, prob.N, prob.D)
    lg = l1.cpu().numpy().reshape(H, prob.N)
    num = den = 0.0
    for bh in range(H):
        for qt, kt in _tile_keys(img_h, img_w, n_text, groups):
            O, L = oracle.attention_set(prob.q, prob.k, prob.v, bh, qt, kt)
            d = np.abs(og[bh, qt] - O)
            assert d.max() <= O_MAX_ABS, d.max()
            assert np.abs(lg[bh, qt] - L).max() <= LSE_MAX_ABS
            num += d.sum()
            den += np.abs(O).sum()
    assert num / den <= O_MEAN_REL
