// Host build of the Gather 0 / Scatter index functions (bsa_gather0.cuh) for
// the CPU tests.  The header is plain integer arithmetic; here the CUDA
// function qualifiers are defined away and the functions run on the host,
// unchanged, over whole index ranges.
#define __device__
#define __forceinline__ inline
#include "bsa_gather0.cuh"

using namespace bsa::g0;

extern "C" {

// Query map of the Gather 0 layout: out[pos] = original token, pos in [0, N).
void g0_query_tokens(int32_t h, int32_t w, int32_t nt, int32_t groups, int32_t N, int32_t N_kv,
                     int32_t* out) {
    const Geom g = make(h, w, nt, groups, N, N_kv);
    for (int32_t pos = 0; pos < N; ++pos) out[pos] = query_token(g, pos);
}

// Key/value map of the packed key tiles: out[pos] = original token, pos in [0, N_kv).
void g0_key_tokens(int32_t h, int32_t w, int32_t nt, int32_t groups, int32_t N, int32_t N_kv,
                   int32_t* out) {
    const Geom g = make(h, w, nt, groups, N, N_kv);
    for (int32_t pos = 0; pos < N_kv; ++pos) out[pos] = key_token(g, pos);
}

// Bands of every query tile pair: y0 [P, 4], cnt, c0, ra, rb [P].
void g0_pair_bands(int32_t h, int32_t w, int32_t nt, int32_t groups, int32_t N, int32_t N_kv,
                   int32_t* y0, int32_t* cnt, int32_t* c0, int32_t* ra, int32_t* rb) {
    const Geom g = make(h, w, nt, groups, N, N_kv);
    for (int32_t p = 0; p < g.P; ++p) {
        int32_t y[4];
        cnt[p] = pair_bands(g, p, y, c0[p], ra[p], rb[p]);
        for (int u = 0; u < 4; ++u) y0[4 * p + u] = y[u];
    }
}

// Query (= key) map of the Scatter layer of N tokens in groups of stride R.
void scatter_query_tokens(int32_t N, int32_t R, int32_t* out) {
    const Geom g = make_scatter(N, R);
    for (int32_t pos = 0; pos < N; ++pos) out[pos] = query_token(g, pos);
}

}  // extern "C"
