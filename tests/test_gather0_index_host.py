"""The forward kernel's Gather 0 and Scatter index functions on the host (no GPU).

``csrc/bsa_gather0.cuh`` holds the integer index functions that the layout
kernel and the geometry-mode forward use to turn a tile position into the
tokens it holds.  ``g0_index_host.cpp`` compiles that header unchanged for
the host, and this file checks the functions against the oracle's Gather 0
sets (INTRA, appendix "Sparse Pattern Index Function") over a seeded sweep
of image shapes, many more than the GPU tests run:
  * the query map is a permutation with text first, and each 64-row half of
    a query tile holds one oracle patch;
  * the bands of each tile pair are distinct and ascending, and each
    patch's window is exactly the bands that start at its top row or 8 rows
    below;
  * an unused band slot repeats band 0;
  * the Scatter-group key tiles hold each group's image tokens;
  * the Scatter layer's map is the gathered order of the Scatter groups.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
P32 = ctypes.POINTER(ctypes.c_int32)


@pytest.fixture(scope="module")
def g0(tmp_path_factory):
    so = str(tmp_path_factory.mktemp("g0") / "libg0host.so")
    subprocess.run(["g++", "-O1", "-std=c++17", "-fPIC", "-shared",
                    "-I", os.path.join(ROOT, "long_context_mask_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "g0_index_host.cpp"), "-o", so], check=True)
    return ctypes.CDLL(so)


def _arr(n):
    a = np.zeros(n, np.int32)
    return a, a.ctypes.data_as(P32)


def _shapes(count=200, seed=11):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < count:
        h = 16 * int(rng.integers(1, 9))
        w = 8 * int(rng.integers(2, 17))
        if (h * w) % 128:
            continue
        nt = 128 * int(rng.integers(0, 5))
        hw = h * w
        gs = [g for g in (1, 2, 4, 8) if nt and (nt // g) % 32 == 0 and hw % g == 0 and (hw // g) % 128 == 0]
        if nt and not gs:
            continue
        out.append((h, w, nt, int(rng.choice(gs)) if nt else 1))
    return out


SHAPES = _shapes()


def _pixels(tok, nt, w):
    u = np.asarray(tok, np.int64) - nt
    return set(zip((u // w).tolist(), (u % w).tolist()))


@pytest.mark.parametrize("h,w,nt,groups", SHAPES)
def test_index_functions_match_oracle_sets(g0, h, w, nt, groups):
    hw = h * w
    N, N_kv = nt + hw, nt + 4 * hw + (hw if nt else 0)
    pw, P = w // 8, hw // 128
    q, qp = _arr(N)
    g0.g0_query_tokens(h, w, nt, groups, N, N_kv, qp)
    k, kp = _arr(N_kv)
    g0.g0_key_tokens(h, w, nt, groups, N, N_kv, kp)
    y0, y0p = _arr(4 * P)
    cnt, cntp = _arr(P)
    c0, c0p = _arr(P)
    ra, rap = _arr(P)
    rb, rbp = _arr(P)
    g0.g0_pair_bands(h, w, nt, groups, N, N_kv, y0p, cntp, c0p, rap, rbp)
    y0 = y0.reshape(P, 4)

    sets = oracle.gather0_sets(h, w, nt, groups)
    assert np.array_equal(np.sort(q), np.arange(N)) and np.array_equal(q[:nt], np.arange(nt))
    assert np.array_equal(k[:nt], np.arange(nt))
    for i in range(hw // 64):
        qt, kt = sets[i]
        r, c = divmod(i, pw)
        p, half = (r // 2) * pw + c, r % 2
        rows = q[nt + 128 * p + 64 * half: nt + 128 * p + 64 * half + 64]
        assert set(rows.tolist()) == set(qt.tolist())
        win = _pixels(kt[nt:], nt, w)
        top = min(y for y, _ in win)
        assert (ra[p] if half == 0 else rb[p]) == top and c0[p] == min(x for _, x in win)
        n = cnt[p]
        bands = y0[p, :n]
        assert np.all(np.diff(bands) > 0) and set(bands.tolist()) == {ra[p], ra[p] + 8, rb[p], rb[p] + 8}
        seen = set()
        for u in range(4):
            tile = k[nt + 128 * (4 * p + u): nt + 128 * (4 * p + u + 1)]
            if u >= n:  # an unused slot repeats band 0
                assert np.array_equal(tile, k[nt + 128 * 4 * p: nt + 128 * (4 * p + 1)])
                continue
            pix = _pixels(tile, nt, w)
            assert pix == {(bands[u] + a, c0[p] + b) for a in range(8) for b in range(16)}
            if bands[u] in (top, top + 8):
                seen |= pix
        assert seen == win
    if nt:
        per_group = hw // groups
        for g in range(groups):
            qt, kt = sets[hw // 64 + g]
            tiles = k[nt + 4 * hw + g * per_group: nt + 4 * hw + (g + 1) * per_group]
            assert set(tiles.tolist()) == set(kt[nt:].tolist())


@pytest.mark.parametrize("N,R", [(1024, 1), (2048, 16), (4096, 8), (4096, 32), (16384, 128), (16384, 64)])
def test_scatter_map_is_the_gathered_group_order(g0, N, R):
    q, qp = _arr(N)
    g0.scatter_query_tokens(N, R, qp)
    assert np.array_equal(q, synth.scatter_map(N, R))
    T = N // R
    # position p = r*T + t holds token t*R + r: group r is contiguous, tokens at stride R
    for r in (0, R // 2, R - 1):
        assert np.array_equal(q[r * T:(r + 1) * T], np.arange(T) * R + r)
