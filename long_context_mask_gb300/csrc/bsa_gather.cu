// Token rows permuted into gathered order in HBM (bsa_gather_rows), and the
// maps / lists / quadrant masks of the INTRA Gather 0 image layer
// (bsa_gather0_layout).
//
// Gathered rows:
// InstaGen, section 3.3 / Introduction: permuted block-sparse attention
// stores every token cluster as a contiguous block; INTRA, "CQS-Aware
// Token-Sparse FlashAttention Kernel": the gathered order is given by an
// index map per head.  dst[bh][p] = src[bh][map[bh][p]].
//
// HBM-bound copy: every source row is read once (a random 2D-byte row) and
// every destination row written once, contiguously.  A warp handles 32
// consecutive destination rows per step: one coalesced load of their 32 map
// entries, then 16-byte copies in which the lanes covering one row read
// consecutive chunks of it (whole 128-byte lines), all loads of the step in
// flight before the first store.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "bsa_internal.h"

namespace bsa {
namespace {

constexpr int kGatherThreads = 256;

template <int D>
__global__ void __launch_bounds__(kGatherThreads) k_gather_rows(const uint4* __restrict__ src,
                                                               const int32_t* __restrict__ map,
                                                               int64_t total_rows, int32_t N,
                                                               uint4* __restrict__ dst, int32_t* status) {
    constexpr int kChunks = D / 8;              // 16-byte chunks per row
    constexpr int kRowsPerCopy = 32 / kChunks;  // rows covered by one warp-wide copy
    constexpr int kCopies = 32 / kRowsPerCopy;  // copies per 32-row step
    const int lane = threadIdx.x & 31;
    const int sub = lane / kChunks, chunk = lane % kChunks;
    const int64_t warps = (int64_t)gridDim.x * (kGatherThreads / 32);
    for (int64_t w = (int64_t)blockIdx.x * (kGatherThreads / 32) + (threadIdx.x >> 5); w * 32 < total_rows;
         w += warps) {
        const int64_t r0 = w * 32;
        // lane l resolves destination row r0 + l to its source row
        long long src_row = -1;
        if (r0 + lane < total_rows) {
            const int64_t r = r0 + lane;
            const int32_t tok = map[r];
            if (tok >= 0 && tok < N) src_row = (r / N) * N + tok;
            else atomicCAS(status, 0, BSA_ERR_BOUNDS);
        }
        uint4 v[kCopies];
#pragma unroll
        for (int k = 0; k < kCopies; ++k) {
            const long long sr = __shfl_sync(0xffffffffu, src_row, k * kRowsPerCopy + sub);
            v[k] = sr >= 0 ? __ldg(src + sr * kChunks + chunk) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int k = 0; k < kCopies; ++k) {
            const int64_t r = r0 + k * kRowsPerCopy + sub;
            if (r < total_rows) dst[r * kChunks + chunk] = v[k];
        }
    }
}

// ---------------------------------------------------------------- Gather 0
// INTRA, appendix "Sparse Pattern Index Function", Gather 0: an 8 x 8 patch of
// image queries attends to the 16 x 16 window centred on it, shifted inward
// at the image edges, and to every text key; text queries attend to every
// text key and to their Scatter group's image tokens ("Mapping Back to
// INTRA").  Two vertically adjacent patches share one 128-row query tile;
// their windows are stored as 8-row x 16-column key bands (the band the two
// windows share is stored once) and each listed band carries the 32-row
// quadrants that see it.

constexpr int kLayoutThreads = 256;

struct G0 {
    int32_t h, w, nt, groups;
    int32_t hw, pw;     // image tokens; patch columns (w / 8)
    int32_t nT, P, G;   // text tiles; query tile pairs; key tiles per Scatter group
    int32_t per;        // text queries per Scatter group
    int32_t N, N_kv, nQB;
};

__device__ __forceinline__ int32_t clampi(int32_t x, int32_t lo, int32_t hi) {
    return x < lo ? lo : (x > hi ? hi : x);
}

// Key bands of query tile pair p: top rows y0[0..cnt) ascending, the shared
// left column c0, and the window tops ra (upper patch) and rb (lower patch).
__device__ int pair_bands(const G0& g, int32_t p, int32_t (&y0)[4], int32_t& c0, int32_t& ra,
                          int32_t& rb) {
    const int32_t s = p / g.pw, c = p % g.pw;
    ra = clampi(16 * s - 4, 0, g.h - 16);
    rb = clampi(16 * s + 4, 0, g.h - 16);
    c0 = clampi(8 * c - 4, 0, g.w - 16);
    const int32_t cand[4] = {ra, ra + 8, rb, rb + 8};
    int cnt = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        // insert cand[i] into the sorted prefix unless present
        bool dup = false;
        for (int j = 0; j < cnt; ++j) dup |= y0[j] == cand[i];
        if (dup) continue;
        int j = cnt++;
        while (j > 0 && y0[j - 1] > cand[i]) {
            y0[j] = y0[j - 1];
            --j;
        }
        y0[j] = cand[i];
    }
    return cnt;
}

__device__ int32_t g0_query_token(const G0& g, int32_t pos) {
    if (pos < g.nt) return pos;
    const int32_t u = pos - g.nt, p = u / 128, i = u % 128;
    const int32_t s = p / g.pw, c = p % g.pw;
    const int32_t y = 16 * s + 8 * (i / 64) + (i % 64) / 8, x = 8 * c + i % 8;
    return g.nt + y * g.w + x;
}

__device__ int32_t g0_key_token(const G0& g, int32_t pos) {
    if (pos < g.nt) return pos;
    const int32_t u = pos - g.nt;
    if (u < 4 * g.hw) {
        const int32_t slot = u / 128, e = u % 128;
        int32_t y0[4] = {0, 0, 0, 0}, c0, ra, rb;
        const int cnt = pair_bands(g, slot / 4, y0, c0, ra, rb);
        int k = slot % 4;
        k = k < cnt ? k : 0;  // unused slot: a copy of the first band (never listed)
        int32_t yk = y0[0];
#pragma unroll
        for (int i = 1; i < 4; ++i) yk = i == k ? y0[i] : yk;
        return g.nt + (yk + e / 16) * g.w + c0 + e % 16;
    }
    const int32_t v = u - 4 * g.hw, per_group = g.hw / g.groups;
    return g.nt + (v % per_group) * g.groups + v / per_group;
}

__global__ void __launch_bounds__(kLayoutThreads) k_gather0_layout(G0 g, int32_t* __restrict__ q_map,
                                                                   int32_t* __restrict__ kv_map,
                                                                   int32_t* __restrict__ kv_idx,
                                                                   int32_t* __restrict__ kv_cnt,
                                                                   uint8_t* __restrict__ quad_mask,
                                                                   int32_t max_kv) {
    const int64_t h = blockIdx.y;
    const int64_t per_head = (int64_t)g.N + g.N_kv + g.nQB;
    for (int64_t e = (int64_t)blockIdx.x * kLayoutThreads + threadIdx.x; e < per_head;
         e += (int64_t)gridDim.x * kLayoutThreads) {
        if (e < g.N) {
            q_map[h * g.N + e] = g0_query_token(g, (int32_t)e);
            continue;
        }
        if (e < (int64_t)g.N + g.N_kv) {
            const int32_t pos = (int32_t)(e - g.N);
            kv_map[h * g.N_kv + pos] = g0_key_token(g, pos);
            continue;
        }
        // one query tile's list
        const int32_t qb = (int32_t)(e - g.N - g.N_kv);
        const int64_t row = h * g.nQB + qb;
        int32_t* idx = kv_idx + row * max_kv;
        uint8_t* qm = quad_mask + row * max_kv;
        int32_t n = 0;
        for (int32_t t = 0; t < g.nT; ++t, ++n) {  // text keys: every row
            idx[n] = t;
            qm[n] = 0xF;
        }
        if (qb < g.nT) {
            // text queries: the Scatter group of each quadrant, groups in order
            const int32_t scatter_tile0 = g.nT + 4 * g.P;
            int32_t prev = -1;
            for (int qd = 0; qd < 4; ++qd) {
                const int32_t grp = (128 * qb + 32 * qd) / g.per;
                if (grp == prev) continue;
                prev = grp;
                uint8_t bits = 0;
                for (int qq = qd; qq < 4; ++qq)
                    if ((128 * qb + 32 * qq) / g.per == grp) bits |= (uint8_t)(1u << qq);
                for (int32_t u = 0; u < g.G; ++u, ++n) {
                    idx[n] = scatter_tile0 + grp * g.G + u;
                    qm[n] = bits;
                }
            }
        } else {
            const int32_t p = qb - g.nT;
            int32_t y0[4] = {0, 0, 0, 0}, c0, ra, rb;
            const int cnt = pair_bands(g, p, y0, c0, ra, rb);
            for (int u = 0; u < cnt; ++u, ++n) {
                idx[n] = g.nT + 4 * p + u;
                const bool upper = y0[u] == ra || y0[u] == ra + 8;
                const bool lower = y0[u] == rb || y0[u] == rb + 8;
                qm[n] = (uint8_t)((upper ? 0x3u : 0u) | (lower ? 0xCu : 0u));
            }
        }
        kv_cnt[row] = n;
        for (int32_t j = n; j < max_kv; ++j) {
            idx[j] = 0;
            qm[j] = 0;
        }
    }
}

}  // namespace

bool gather0_geometry(int32_t img_h, int32_t img_w, int32_t n_text, int32_t groups, Gather0Geom* out) {
    if (img_h < 16 || img_h > 4096 || (img_h % 16) != 0 || img_w < 16 || img_w > 4096 || (img_w % 8) != 0)
        return false;
    if (n_text < 0 || n_text > (1 << 20) || (n_text % 128) != 0) return false;
    const int64_t hw = (int64_t)img_h * img_w;
    if (n_text > 0) {
        if (groups < 1 || (n_text % groups) != 0 || ((n_text / groups) % 32) != 0 || (hw % groups) != 0 ||
            ((hw / groups) % 128) != 0)
            return false;
    }
    const int64_t N = n_text + hw, N_kv = n_text + 4 * hw + (n_text > 0 ? hw : 0);
    if (N > (1 << 24) || N_kv > (1 << 26)) return false;
    const int32_t nT = n_text / 128;
    int32_t need = img_h > 16 ? 4 : 2;  // window bands of a tile pair
    if (n_text > 0) {
        const int32_t per = n_text / groups, G = (int32_t)(hw / groups / 128);
        for (int32_t t = 0; t < nT; ++t) {
            int32_t distinct = 0, prev = -1;
            for (int qd = 0; qd < 4; ++qd) {
                const int32_t grp = (128 * t + 32 * qd) / per;
                if (grp != prev) ++distinct;
                prev = grp;
            }
            need = need > distinct * G ? need : distinct * G;
        }
    }
    out->img_h = img_h;
    out->img_w = img_w;
    out->n_text = n_text;
    out->groups = n_text > 0 ? groups : 1;
    out->N = (int32_t)N;
    out->N_kv = (int32_t)N_kv;
    out->max_kv = nT + need;
    return true;
}

cudaError_t launch_gather0_layout(const Gather0Geom& geo, int64_t heads, int32_t* q_map, int32_t* kv_map,
                                  int32_t* kv_idx, int32_t* kv_cnt, uint8_t* quad_mask, int32_t max_kv,
                                  cudaStream_t stream) {
    G0 g;
    g.h = geo.img_h;
    g.w = geo.img_w;
    g.nt = geo.n_text;
    g.groups = geo.groups;
    g.hw = geo.img_h * geo.img_w;
    g.pw = geo.img_w / 8;
    g.nT = geo.n_text / 128;
    g.P = g.hw / 128;
    g.G = g.hw / g.groups / 128;
    g.per = geo.n_text > 0 ? geo.n_text / geo.groups : 1;
    g.N = geo.N;
    g.N_kv = geo.N_kv;
    g.nQB = geo.N / 128;
    const int64_t per_head = (int64_t)g.N + g.N_kv + g.nQB;
    const int64_t want = (per_head + kLayoutThreads - 1) / kLayoutThreads;
    const unsigned gx = (unsigned)(want < 4096 ? want : 4096);
    k_gather0_layout<<<dim3(gx, (unsigned)heads), kLayoutThreads, 0, stream>>>(g, q_map, kv_map, kv_idx,
                                                                                kv_cnt, quad_mask, max_kv);
    return cudaGetLastError();
}

cudaError_t launch_gather_rows(const void* src, const int32_t* map, int64_t heads, int32_t N,
                               int32_t D, void* dst, int32_t* status, cudaStream_t stream) {
    const int64_t total_rows = heads * (int64_t)N;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int64_t steps = (total_rows + 31) / 32;
    const int64_t want = (steps + kGatherThreads / 32 - 1) / (kGatherThreads / 32);
    const int64_t cap = (int64_t)sms * 8;  // 8 resident blocks of 256 threads per SM
    const unsigned grid = (unsigned)(want < cap ? want : cap);
    if (D == 128)
        k_gather_rows<128><<<grid, kGatherThreads, 0, stream>>>(static_cast<const uint4*>(src), map,
                                                                 total_rows, N, static_cast<uint4*>(dst), status);
    else
        k_gather_rows<64><<<grid, kGatherThreads, 0, stream>>>(static_cast<const uint4*>(src), map,
                                                                total_rows, N, static_cast<uint4*>(dst), status);
    return cudaGetLastError();
}

}  // namespace bsa
