"""GPU parity of the INTRA Gather 0 image layer (appendix "Sparse Pattern
Index Function", Gather 0; text queries as in "Mapping Back to INTRA").

The layout call builds maps, lists and quadrant masks on the GPU; the
packed forward runs them.  The oracle computes the layer from its
definition (per CQS: the query patch, the clamped 16 x 16 window and the
text keys), sharing nothing with the layout:
  * the key set each query sees through the layout equals the oracle's set
    exactly (integer parity, every query of the first and last head);
  * O / LSE match the oracle within the float bar, on every row of small
    images and on sampled CQS of the FLUX.1-dev shape.
"""
import numpy as np
import pytest
import torch

import long_context_mask_gb300 as bsa
import oracle
import synth
from gpu_util import LSE_MAX_ABS, O_MAX_ABS, O_MEAN_REL, status_ok

pytestmark = pytest.mark.gpu

# img_h, img_w, n_text, groups
SHAPES = [
    (32, 32, 128, 2),    # 2 text groups of 64: two groups per text tile
    (16, 24, 0, 1),      # one row of tile pairs (windows equal), no text
    (48, 16, 256, 2),    # one group per text tile; edge and interior pairs
    (64, 32, 256, 8),    # 32 text queries per group: one group per quadrant
]


def _layout(img_h, img_w, n_text, groups, heads):
    out = bsa.gather0_layout(img_h, img_w, n_text, groups, heads)
    torch.cuda.synchronize()
    status_ok()
    return out


@pytest.mark.parametrize("img_h,img_w,n_text,groups", SHAPES + [(128, 128, 512, 8)])
def test_layout_key_sets_match_definition(img_h, img_w, n_text, groups):
    heads = 3
    q_map, kv_map, idx, cnt, qm = (t.cpu().numpy() for t in _layout(img_h, img_w, n_text, groups, heads))
    N = n_text + img_h * img_w
    nqb = N // 128
    expected = {}
    for qt, kt in oracle.gather0_sets(img_h, img_w, n_text, groups):
        ks = np.sort(kt)
        for t in qt:
            expected[int(t)] = ks
    assert len(expected) == N
    for h in range(heads):
        assert np.array_equal(np.sort(q_map[h]), np.arange(N))        # a permutation
        assert np.array_equal(q_map[h], q_map[0]) and np.array_equal(kv_map[h], kv_map[0])
    assert kv_map.min() >= 0 and kv_map.max() < N
    for h in (0, heads - 1):
        for qb in range(nqb):
            row = h * nqb + qb
            n = int(cnt[row])
            assert np.all(idx[row, n:] == 0) and np.all(qm[row, n:] == 0)
            for quad in range(4):
                tiles = [int(t) for t, m in zip(idx[row, :n], qm[row, :n]) if (m >> quad) & 1]
                keys = np.sort(np.concatenate([kv_map[h, 128 * t: 128 * t + 128] for t in tiles]))
                for r in range(32 * quad, 32 * quad + 32):
                    tok = int(q_map[h, qb * 128 + r])
                    assert np.array_equal(keys, expected[tok]), (h, qb, r, tok)


def _check(o, lse, O_ref, L_ref, heads, rows):
    """Compare the GPU rows `rows` (token ids) of flat heads `heads`."""
    D = o.shape[-1]
    og = o.reshape(-1, o.shape[2], D)[heads][:, rows].float().cpu().numpy()
    lg = lse.reshape(-1, lse.shape[2])[heads][:, rows].cpu().numpy().astype(np.float64)
    Oo, Lo = O_ref[:, rows], L_ref[:, rows]
    assert np.isfinite(Lo).all()
    diff = np.abs(og - Oo)
    max_abs = float(diff.max())
    mean_rel = float(diff.sum() / np.abs(Oo).sum())
    lse_abs = float(np.abs(lg - Lo).max())
    assert max_abs <= O_MAX_ABS, f"O max-abs {max_abs}"
    assert mean_rel <= O_MEAN_REL, f"O mean-rel {mean_rel}"
    assert lse_abs <= LSE_MAX_ABS, f"LSE max-abs {lse_abs}"
    return max_abs, mean_rel, lse_abs


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("img_h,img_w,n_text,groups", SHAPES)
def test_forward_small_all_rows(img_h, img_w, n_text, groups, D):
    prob = synth.image_gather0(seed=20 + img_w, B=1, H=2, img_h=img_h, img_w=img_w, n_text=n_text,
                               groups=groups, D=D)
    q_map, kv_map, idx, cnt, qm = _layout(img_h, img_w, n_text, groups, prob.B * prob.H)
    q, k, v = (t.cuda() for t in (prob.q, prob.k, prob.v))
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    bsa.forward_packed(q, k, v, idx, cnt, kv_map, o, lse, quad_mask=qm, q_map=q_map)
    torch.cuda.synchronize()
    status_ok()
    O_ref, L_ref = oracle.gather0_attention(prob.q, prob.k, prob.v, img_h, img_w, n_text, groups)
    _check(o, lse, O_ref, L_ref, [0, 1], np.arange(prob.N))


def test_forward_grouped_heads_and_row_order():
    """Grouped key/value heads (4 query heads over 2) with the first B*H_kv
    copies of kv_map; any row order gives bit-identical output."""
    img_h, img_w, n_text, groups = 32, 32, 128, 2
    prob = synth.image_gather0(seed=31, B=1, H=4, img_h=img_h, img_w=img_w, n_text=n_text,
                               groups=groups, D=128)
    k_h, v_h = prob.k[:, :2].contiguous(), prob.v[:, :2].contiguous()
    q_map, kv_map, idx, cnt, qm = _layout(img_h, img_w, n_text, groups, 4)
    q, k, v = prob.q.cuda(), k_h.cuda(), v_h.cuda()
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    bsa.forward_packed(q, k, v, idx, cnt, kv_map[:2].contiguous(), o, lse, quad_mask=qm, q_map=q_map)
    perm = torch.empty((4, prob.N // 128), dtype=torch.int32, device=q.device)
    bsa.reorder_rows(cnt.view(4, -1), 7, perm)
    o2, lse2 = torch.empty_like(o), torch.empty_like(lse)
    bsa.forward_packed(q, k, v, idx, cnt, kv_map[:2].contiguous(), o2, lse2, quad_mask=qm, q_map=q_map,
                       row_perm=perm)
    torch.cuda.synchronize()
    status_ok()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    O_ref, L_ref = oracle.gather0_attention(prob.q, k_h, v_h, img_h, img_w, n_text, groups)
    _check(o, lse, O_ref, L_ref, [0, 1, 2, 3], np.arange(prob.N))


def test_forward_flux_shape_sampled():
    """FLUX.1-dev shape (512 text tokens, 128 x 128 image, 24 heads, D 128)
    in the launch configuration the benchmark times, against the oracle on
    sampled CQS: corner, edge and interior patches and two text groups, on
    the first and last head."""
    prob = synth.image_gather0()
    img_h, img_w, n_text, groups = prob.img_h, prob.img_w, prob.n_text, prob.groups
    BH = prob.B * prob.H
    q_map, kv_map, idx, cnt, qm = _layout(img_h, img_w, n_text, groups, BH)
    perm = torch.empty((BH, prob.N // 128), dtype=torch.int32, device="cuda")
    bsa.reorder_rows(cnt.view(BH, -1), bsa.resident_ctas(prob.D), perm)
    q, k, v = (t.cuda() for t in (prob.q, prob.k, prob.v))
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    bsa.forward_packed(q, k, v, idx, cnt, kv_map, o, lse, quad_mask=qm, q_map=q_map, row_perm=perm)
    torch.cuda.synchronize()
    status_ok()
    n_img = img_h * img_w // 64
    pw = img_w // 8
    sets = [0, pw - 1, pw + 1, n_img // 2 + 3, n_img - pw, n_img - 1, n_img, n_img + groups - 1]
    heads = [0, BH - 1]
    O_ref, L_ref = oracle.gather0_attention(prob.q, prob.k, prob.v, img_h, img_w, n_text, groups,
                                            heads=heads, sets=sets)
    all_sets = oracle.gather0_sets(img_h, img_w, n_text, groups)
    rows = np.concatenate([all_sets[s][0] for s in sets])
    _check(o, lse, O_ref, L_ref, heads, rows)


def _run_both(prob, heads_kv=None, row_perm=True):
    """The packed forward on the layout's maps and the geometry-mode forward
    on the same lists; returns both results and the inputs used."""
    img_h, img_w, n_text, groups = prob.img_h, prob.img_w, prob.n_text, prob.groups
    BH = prob.B * prob.H
    k_h = prob.k if heads_kv is None else prob.k[:, :heads_kv].contiguous()
    v_h = prob.v if heads_kv is None else prob.v[:, :heads_kv].contiguous()
    q_map, kv_map, idx, cnt, qm = _layout(img_h, img_w, n_text, groups, BH)
    perm = None
    if row_perm:
        perm = torch.empty((BH, prob.N // 128), dtype=torch.int32, device="cuda")
        bsa.reorder_rows(cnt.view(BH, -1), bsa.resident_ctas(prob.D), perm)
    q, k, v = prob.q.cuda(), k_h.cuda(), v_h.cuda()
    kvh = k.shape[0] * k.shape[1]
    o1, o2 = torch.empty_like(q), torch.empty_like(q)
    l1 = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    l2 = torch.empty_like(l1)
    bsa.forward_packed(q, k, v, idx, cnt, kv_map[:kvh].contiguous(), o1, l1, quad_mask=qm, q_map=q_map,
                       row_perm=perm)
    bsa.forward_gather0(q, k, v, img_h, img_w, n_text, groups, idx, cnt, o2, l2, quad_mask=qm,
                        row_perm=perm)
    torch.cuda.synchronize()
    status_ok()
    return (o1, l1), (o2, l2), (k_h, v_h)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("img_h,img_w,n_text,groups", SHAPES)
def test_geometry_mode_small(img_h, img_w, n_text, groups, D):
    """Tiles fetched as boxes of the image give the packed path's result bit
    for bit, and match the oracle on every row."""
    prob = synth.image_gather0(seed=40 + img_h, B=1, H=2, img_h=img_h, img_w=img_w, n_text=n_text,
                               groups=groups, D=D)
    (o1, l1), (o2, l2), _ = _run_both(prob, row_perm=False)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    O_ref, L_ref = oracle.gather0_attention(prob.q, prob.k, prob.v, img_h, img_w, n_text, groups)
    _check(o2, l2, O_ref, L_ref, [0, 1], np.arange(prob.N))


def test_geometry_mode_grouped_heads():
    prob = synth.image_gather0(seed=41, B=2, H=4, img_h=48, img_w=16, n_text=256, groups=2, D=128)
    (o1, l1), (o2, l2), (k_h, v_h) = _run_both(prob, heads_kv=2)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    O_ref, L_ref = oracle.gather0_attention(prob.q, k_h, v_h, prob.img_h, prob.img_w, prob.n_text,
                                            prob.groups)
    _check(o2, l2, O_ref, L_ref, list(range(8)), np.arange(prob.N))


def test_geometry_mode_flux_shape():
    """The benchmark's launch configuration (FLUX.1-dev shape, reordered rows):
    bit-identical to the packed path everywhere, and against the oracle on
    sampled CQS of the first and last head."""
    prob = synth.image_gather0()
    (o1, l1), (o2, l2), _ = _run_both(prob)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    img_h, img_w, n_text, groups = prob.img_h, prob.img_w, prob.n_text, prob.groups
    n_img = img_h * img_w // 64
    pw = img_w // 8
    sets = [0, pw, 2 * pw + 5, n_img // 3, n_img - pw - 1, n_img - 1, n_img + 1, n_img + groups - 2]
    heads = [0, prob.B * prob.H - 1]
    O_ref, L_ref = oracle.gather0_attention(prob.q, prob.k, prob.v, img_h, img_w, n_text, groups,
                                            heads=heads, sets=sets)
    all_sets = oracle.gather0_sets(img_h, img_w, n_text, groups)
    rows = np.concatenate([all_sets[s][0] for s in sets])
    _check(o2, l2, O_ref, L_ref, heads, rows)


def _sweep_shapes():
    import test_gather0_shapes
    return test_gather0_shapes.SHAPES


@pytest.mark.parametrize("img_h,img_w,n_text,groups", _sweep_shapes())
def test_layout_key_sets_sweep(img_h, img_w, n_text, groups):
    """The GPU layout over 30 seeded image shapes: every query sees exactly
    the oracle's key set (one head; heads are identical copies)."""
    q_map, kv_map, idx, cnt, qm = (t.cpu().numpy() for t in _layout(img_h, img_w, n_text, groups, 1))
    N = n_text + img_h * img_w
    expected = {}
    for qt, kt in oracle.gather0_sets(img_h, img_w, n_text, groups):
        ks = np.sort(kt)
        for t in qt:
            expected[int(t)] = ks
    assert np.array_equal(np.sort(q_map[0]), np.arange(N))
    for qb in range(N // 128):
        n = int(cnt[qb])
        for quad in range(4):
            tiles = [int(t) for t, m in zip(idx[qb, :n], qm[qb, :n]) if (m >> quad) & 1]
            keys = np.sort(np.concatenate([kv_map[0, 128 * t: 128 * t + 128] for t in tiles]))
            toks = q_map[0, qb * 128 + 32 * quad: qb * 128 + 32 * quad + 32]
            for tok in toks:
                assert np.array_equal(keys, expected[int(tok)])
