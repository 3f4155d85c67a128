"""Pins of the Gather 0 oracle (INTRA, appendix "Sparse Pattern Index
Function", Gather 0; "Mapping Back to INTRA" for the text tokens).

Each check compares the oracle with something other than itself: a
hand-worked table of window corners, geometric properties of the windows,
the whole-image special case (dense attention) and a masked
scaled-dot-product attention whose mask is built from a different
description of the window (the in-image 16-row / 16-column span nearest to
the patch centre).
"""
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "gather0_windows.txt")


def _golden_rows():
    rows = []
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        rows.append(tuple(int(x) for x in line.split()))
    return rows


def _pix(tok, n_text, img_w):
    u = np.asarray(tok, np.int64) - n_text
    return u // img_w, u % img_w


@pytest.mark.parametrize("row", _golden_rows())
def test_window_corners_hand_worked(row):
    img_h, img_w, i, r, c, r0, c0, first, last = row
    qt, kt = oracle.gather0_sets(img_h, img_w, 0, 1)[i]
    qy, qx = _pix(qt, 0, img_w)
    assert qy.min() == 8 * r and qx.min() == 8 * c
    assert kt.min() == first and kt.max() == last
    ky, kx = _pix(kt, 0, img_w)
    box = {(y, x) for y in range(r0, r0 + 16) for x in range(c0, c0 + 16)}
    assert set(zip(ky.tolist(), kx.tolist())) == box


@pytest.mark.parametrize("img_h,img_w,n_text,groups", [(32, 32, 0, 1), (64, 48, 128, 2), (16, 24, 0, 1),
                                                       (48, 16, 256, 8), (16, 16, 128, 4)])
def test_window_geometry(img_h, img_w, n_text, groups):
    sets = oracle.gather0_sets(img_h, img_w, n_text, groups)
    hw = img_h * img_w
    n_img = hw // 64
    assert len(sets) == n_img + (groups if n_text else 0)
    seen_q = np.zeros(n_text + hw, np.int64)
    for qt, kt in sets[:n_img]:
        seen_q[qt] += 1
        assert len(qt) == 64 and len(kt) == n_text + 256
        # text keys first, each once
        assert np.array_equal(kt[:n_text], np.arange(n_text))
        img = kt[n_text:]
        assert len(np.unique(img)) == 256 and img.min() >= n_text and img.max() < n_text + hw
        qy, qx = _pix(qt, n_text, img_w)
        ky, kx = _pix(img, n_text, img_w)
        # the queries are one aligned 8 x 8 patch
        assert qy.max() - qy.min() == 7 and qx.max() - qx.min() == 7
        assert qy.min() % 8 == 0 and qx.min() % 8 == 0
        assert len(set(zip(qy.tolist(), qx.tolist()))) == 64
        # the keys are one 16 x 16 box inside the image that holds the patch
        assert ky.max() - ky.min() == 15 and kx.max() - kx.min() == 15
        assert ky.min() <= qy.min() and ky.max() >= qy.max()
        assert kx.min() <= qx.min() and kx.max() >= qx.max()
        # centred on the patch, unless that would leave the image: then it
        # touches the edge it was shifted away from
        for lo_q, hi_q, lo_k, hi_k, ext in ((qy.min(), qy.max(), ky.min(), ky.max(), img_h),
                                            (qx.min(), qx.max(), kx.min(), kx.max(), img_w)):
            if lo_q - 4 >= 0 and hi_q + 4 <= ext - 1:
                assert lo_k == lo_q - 4 and hi_k == hi_q + 4
            else:
                assert lo_k == 0 or hi_k == ext - 1
    for g, (qt, kt) in enumerate(sets[n_img:]):
        seen_q[qt] += 1
        per = n_text // groups
        assert np.array_equal(qt, np.arange(g * per, (g + 1) * per))
        assert np.array_equal(kt[:n_text], np.arange(n_text))
        img = kt[n_text:] - n_text
        assert len(img) == hw // groups and len(np.unique(img)) == len(img)
        assert np.all(img % groups == g)
    # every query token belongs to exactly one set
    assert np.all(seen_q == 1)


def _sdpa_ref(q, k, v, allowed):
    """Masked softmax attention by torch's scaled_dot_product_attention in
    fp64 (a library routine), LSE by torch.logsumexp."""
    qf, kf, vf = (t.to(torch.float64) for t in (q, k, v))
    mask = torch.from_numpy(allowed)
    O = torch.nn.functional.scaled_dot_product_attention(qf, kf, vf, attn_mask=mask)
    s = (qf @ kf.transpose(-1, -2)) / (q.shape[-1] ** 0.5)
    s = s.masked_fill(~mask, float("-inf"))
    return O.numpy(), torch.logsumexp(s, dim=-1).numpy()


def _allowed_nearest_span(img_h, img_w, n_text, groups):
    """Visibility built from a second description of the pattern: a query's
    key rows are the 16 consecutive in-image rows whose centre lies nearest to
    the centre of the query's 8-row patch (likewise columns); all text keys
    are visible; a text query sees the image tokens whose index is congruent
    to its Scatter group modulo the group count."""
    N = n_text + img_h * img_w

    def span(p, ext):
        centre = 8 * (p // 8) + 3.5
        starts = np.arange(0, ext - 15)
        a = starts[np.argmin(np.abs(starts + 7.5 - centre))]
        return a, a + 16

    allowed = np.zeros((N, N), bool)
    allowed[:, :n_text] = True
    for i in range(n_text, N):
        y, x = divmod(i - n_text, img_w)
        y0, y1 = span(y, img_h)
        x0, x1 = span(x, img_w)
        for ky in range(y0, y1):
            allowed[i, n_text + ky * img_w + x0: n_text + ky * img_w + x1] = True
    if n_text:
        per = n_text // groups
        img_idx = np.arange(img_h * img_w)
        for i in range(n_text):
            allowed[i, n_text + img_idx[img_idx % groups == i // per]] = True
    return allowed


@pytest.mark.parametrize("img_h,img_w,n_text,groups", [(16, 16, 0, 1), (16, 16, 128, 2), (32, 24, 128, 4)])
def test_attention_against_masked_sdpa(img_h, img_w, n_text, groups):
    N = n_text + img_h * img_w
    g = torch.Generator().manual_seed(11)
    q, k, v = (synth.normal_bf16(g, (1, 2, N, 64)) for _ in range(3))
    O, L = oracle.gather0_attention(q, k, v, img_h, img_w, n_text, groups)
    allowed = _allowed_nearest_span(img_h, img_w, n_text, groups)
    if img_h == 16 and img_w == 16:
        # the window is the whole image: every image query is dense attention
        assert allowed[n_text:].all()
    O_ref, L_ref = _sdpa_ref(q, k, v, allowed)
    np.testing.assert_allclose(O, O_ref[0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(L, L_ref[0], rtol=0, atol=1e-12)


def test_attention_grouped_heads_and_subsets():
    """Grouped key/value heads read head h / (H/H_kv); a subset of heads and
    sets fills only those rows."""
    img_h, img_w, n_text, groups = 16, 16, 128, 2
    N = n_text + img_h * img_w
    g = torch.Generator().manual_seed(12)
    q = synth.normal_bf16(g, (1, 4, N, 64))
    k, v = (synth.normal_bf16(g, (1, 2, N, 64)) for _ in range(2))
    O, L = oracle.gather0_attention(q, k, v, img_h, img_w, n_text, groups, heads=[3], sets=[1])
    allowed = _allowed_nearest_span(img_h, img_w, n_text, groups)
    O_ref, L_ref = _sdpa_ref(q[:, 3:4], k[:, 1:2], v[:, 1:2], allowed)
    qt, _ = oracle.gather0_sets(img_h, img_w, n_text, groups)[1]
    np.testing.assert_allclose(O[0, qt], O_ref[0, 0, qt], rtol=0, atol=1e-12)
    np.testing.assert_allclose(L[0, qt], L_ref[0, 0, qt], rtol=0, atol=1e-12)
    others = np.setdiff1d(np.arange(N), qt)
    assert np.isnan(L[0, others]).all()
