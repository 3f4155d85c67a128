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

#include "bsa_gather0.cuh"
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
// Maps, lists and quadrant masks of the INTRA Gather 0 layer; the index
// functions are in bsa_gather0.cuh.  Two vertically adjacent patches share
// one 128-row query tile; each listed window band carries the 32-row
// quadrants that see it.

constexpr int kLayoutThreads = 256;
using g0::Geom;

__global__ void __launch_bounds__(kLayoutThreads) k_gather0_layout(Geom g, int32_t* __restrict__ q_map,
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
            q_map[h * g.N + e] = g0::query_token(g, (int32_t)e);
            continue;
        }
        if (e < (int64_t)g.N + g.N_kv) {
            const int32_t pos = (int32_t)(e - g.N);
            kv_map[h * g.N_kv + pos] = g0::key_token(g, pos);
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
            const int cnt = g0::pair_bands(g, p, y0, c0, ra, rb);
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
    const Geom g = g0::make(geo.img_h, geo.img_w, geo.n_text, geo.groups, geo.N, geo.N_kv);
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
