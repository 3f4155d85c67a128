// Index functions of the INTRA Gather 0 image layer and of the Scatter layer,
// shared by the layout kernel (bsa_gather.cu) and the forward kernel's
// geometry mode (bsa_attn.cu).
//
// INTRA, appendix "Sparse Pattern Index Function", Gather 0: an 8 x 8 patch of
// image queries attends to the 16 x 16 window centred on it, shifted inward
// at the image edges, and to every text key; text queries attend to every
// text key and to their Scatter group's image tokens ("Mapping Back to
// INTRA").  The sequence is nt text tokens, then the h x w image row-major.
//
// Layout: query tile nt/128 + s*(w/8) + c holds patch (2s, c) in rows 0..63
// and patch (2s+1, c) in rows 64..127.  Key tiles: the text tiles; then four
// slots per query tile pair for its windows' 8-row x 16-column bands (the band
// the two windows share stored once); then the Scatter groups, 128 tokens per
// tile.
//
// Scatter layer (INTRA, "Why Scatter Is Uniform and Non-Contiguous"): N = R*T
// tokens, token (t, r) = t*R + r; group S_r = {(t, r) : t} in gathered order,
// position p = r*T + t.  A 128-position tile is 128 tokens at stride R, and
// the same geometry serves queries and keys.  It is described here with no
// text and no image: every key tile is a group tile.
#pragma once

#include <stdint.h>

namespace bsa {
namespace g0 {

struct Geom {
    int32_t h, w, nt, groups;
    int32_t hw, pw;     // image tokens; patch columns (w / 8)
    int32_t nT, P, G;   // text tiles; query tile pairs; key tiles per Scatter group
    int32_t per;        // text queries per Scatter group
    int32_t N, N_kv, nQB;
    int32_t scatter;    // 1: the Scatter layer (groups = R, hw = N, no text, no image)
};

inline Geom make(int32_t h, int32_t w, int32_t nt, int32_t groups, int32_t N, int32_t N_kv) {
    Geom g;
    g.h = h;
    g.w = w;
    g.nt = nt;
    g.groups = nt > 0 ? groups : 1;
    g.hw = h * w;
    g.pw = w / 8;
    g.nT = nt / 128;
    g.P = g.hw / 128;
    g.G = g.hw / g.groups / 128;
    g.per = nt > 0 ? nt / g.groups : 1;
    g.N = N;
    g.N_kv = N_kv;
    g.nQB = N / 128;
    g.scatter = 0;
    return g;
}

inline Geom make_scatter(int32_t N, int32_t R) {
    Geom g;
    g.h = g.w = g.nt = 0;
    g.groups = R;
    g.hw = N;
    g.pw = 1;
    g.nT = 0;
    g.P = 0;
    g.G = N / R / 128;
    g.per = 1;
    g.N = N;
    g.N_kv = N;
    g.nQB = N / 128;
    g.scatter = 1;
    return g;
}

__device__ __forceinline__ int32_t clampi(int32_t x, int32_t lo, int32_t hi) {
    return x < lo ? lo : (x > hi ? hi : x);
}

// Key bands of query tile pair p: top rows y0[0..cnt) ascending, the shared
// left column c0, and the window tops ra (upper patch) and rb (lower patch).
// Clamping is monotone and moves no value further than its argument moves,
// so 0 <= rb - ra <= 8: equal windows give the bands {ra, ra+8}, windows 8
// rows apart share the middle band, {ra, ra+8, ra+16}, and otherwise the
// four bands interleave, {ra, rb, ra+8, rb+8}.
__device__ __forceinline__ int pair_bands(const Geom& g, int32_t p, int32_t (&y0)[4], int32_t& c0,
                                          int32_t& ra, int32_t& rb) {
    const int32_t s = p / g.pw, c = p % g.pw;
    ra = clampi(16 * s - 4, 0, g.h - 16);
    rb = clampi(16 * s + 4, 0, g.h - 16);
    c0 = clampi(8 * c - 4, 0, g.w - 16);
    const int cnt = rb == ra ? 2 : (rb == ra + 8 ? 3 : 4);
    y0[0] = ra;
    y0[1] = cnt == 4 ? rb : ra + 8;
    y0[2] = cnt == 4 ? ra + 8 : ra + 16;
    y0[3] = rb + 8;
    return cnt;
}

// Top row of band slot u of pair p (an unused slot repeats band 0) and the
// band's left column.
__device__ __forceinline__ int32_t band_top(const Geom& g, int32_t p, int32_t u, int32_t& c0) {
    int32_t y0[4], ra, rb;
    const int cnt = pair_bands(g, p, y0, c0, ra, rb);
    return u >= cnt ? y0[0] : (u == 0 ? y0[0] : (u == 1 ? y0[1] : (u == 2 ? y0[2] : y0[3])));
}

// Original token of query position pos (the query map).
__device__ __forceinline__ int32_t query_token(const Geom& g, int32_t pos) {
    if (g.scatter) {
        const int32_t T = g.hw / g.groups;
        return (pos % T) * g.groups + pos / T;
    }
    if (pos < g.nt) return pos;
    const int32_t u = pos - g.nt, p = u / 128, i = u % 128;
    const int32_t s = p / g.pw, c = p % g.pw;
    const int32_t y = 16 * s + 8 * (i / 64) + (i % 64) / 8, x = 8 * c + i % 8;
    return g.nt + y * g.w + x;
}

// Original token of packed key position pos (the key/value map).
__device__ __forceinline__ int32_t key_token(const Geom& g, int32_t pos) {
    if (pos < g.nt) return pos;
    const int32_t u = pos - g.nt;
    if (u < 4 * g.hw) {
        const int32_t slot = u / 128, e = u % 128;
        int32_t c0;
        const int32_t yk = band_top(g, slot / 4, slot % 4, c0);
        return g.nt + (yk + e / 16) * g.w + c0 + e % 16;
    }
    const int32_t v = u - 4 * g.hw, per_group = g.hw / g.groups;
    return g.nt + (v % per_group) * g.groups + v / per_group;
}

}  // namespace g0
}  // namespace bsa
