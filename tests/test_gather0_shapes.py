"""Gather 0 over a seeded sweep of image shapes (no GPU).

The oracle's sets (INTRA, appendix "Sparse Pattern Index Function",
Gather 0) are checked against geometric facts on every shape, and the
library's host-side sizes (bsa_gather0_sizes) against a brute-force count
of the layout the header describes: two patches per 128-row query tile,
their windows' distinct 8-row bands, text tiles in front, Scatter-group
tiles for the text queries.
"""
import ctypes

import numpy as np
import pytest

import oracle
from long_context_mask_gb300 import build as bsa_build
from long_context_mask_gb300.binding import load_library


@pytest.fixture(scope="module")
def lib():
    bsa_build.build()
    return load_library()


def _shapes(count=30, seed=7):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < count:
        h = int(rng.choice([16, 32, 48, 64]))
        w = int(rng.choice([16, 24, 32, 40, 48, 56, 64]))
        nt = int(rng.choice([0, 128, 256, 384]))
        hw = h * w
        gs = [g for g in (1, 2, 4, 8) if nt and nt % g == 0 and (nt // g) % 32 == 0 and hw % g == 0
              and (hw // g) % 128 == 0]
        if nt and not gs:
            continue
        g = int(rng.choice(gs)) if nt else 1
        out.append((h, w, nt, g))
    return out


SHAPES = _shapes()


@pytest.mark.parametrize("h,w,nt,g", SHAPES)
def test_oracle_sets_geometry(h, w, nt, g):
    sets = oracle.gather0_sets(h, w, nt, g)
    hw = h * w
    seen = np.zeros(nt + hw, np.int64)
    for qt, kt in sets[: hw // 64]:
        seen[qt] += 1
        img = kt[nt:] - nt
        ky, kx = img // w, img % w
        qy, qx = (qt - nt) // w, (qt - nt) % w
        # a 16 x 16 box inside the image holding the 8 x 8 patch, text keys first
        assert np.array_equal(kt[:nt], np.arange(nt))
        assert len(set(img.tolist())) == 256
        assert ky.min() >= 0 and ky.max() < h and kx.min() >= 0 and kx.max() < w
        assert ky.max() - ky.min() == 15 and kx.max() - kx.min() == 15
        assert ky.min() <= qy.min() and ky.max() >= qy.max() and kx.min() <= qx.min() and kx.max() >= qx.max()
        # no window closer to the patch centre fits inside the image
        for lo, ext, c in ((ky.min(), h, qy.min() + 3.5), (kx.min(), w, qx.min() + 3.5)):
            best = min(range(0, ext - 15), key=lambda a: abs(a + 7.5 - c))
            assert lo == best
    for qt, kt in sets[hw // 64:]:
        seen[qt] += 1
    assert np.all(seen == 1)


def _sizes_brute(h, w, nt, g):
    """N, N_kv and the list capacity, by enumerating the layout."""
    hw = h * w
    clamp = lambda x, lo, hi: max(lo, min(hi, x))  # noqa: E731
    need = 0
    for s in range(h // 16):
        ra, rb = clamp(16 * s - 4, 0, h - 16), clamp(16 * s + 4, 0, h - 16)
        need = max(need, len({ra, ra + 8, rb, rb + 8}))
    if nt:
        per, G = nt // g, hw // g // 128
        for t in range(nt // 128):
            groups = {(128 * t + 32 * q) // per for q in range(4)}
            need = max(need, len(groups) * G)
    return nt + hw, nt + 4 * hw + (hw if nt else 0), nt // 128 + need


@pytest.mark.parametrize("h,w,nt,g", SHAPES)
def test_library_sizes_match_layout(lib, h, w, nt, g):
    i32 = ctypes.c_int32
    N, N_kv, mk = i32(0), i32(0), i32(0)
    assert lib.bsa_gather0_sizes(h, w, nt, g, ctypes.byref(N), ctypes.byref(N_kv), ctypes.byref(mk)) == 0
    assert (N.value, N_kv.value, mk.value) == _sizes_brute(h, w, nt, g)
