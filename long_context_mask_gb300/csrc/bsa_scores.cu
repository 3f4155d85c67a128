// Block scores from block means: the scoring step in front of top-k block
// selection and importance sampling.
//
// MC-Sparse, "The MC-Sparse Architecture": block-sparse attention keeps, per
// query block, the KV blocks with the highest mean-pooled similarity.
// InstaGen, Algorithm 1 step 2 and section 3.3: the centroid score
// s_gc = exp(q_g . k_c / sqrt d) of a query group and a key cluster.  With
// the tokens gathered through q_map / kv_map, a group or cluster is a
// 128-token block of the gathered order.
//
//   k_block_means   one thread block per (head, block, tensor): the fp32 mean
//                   of the block's 128 rows (gathered through the map), read
//                   with 16-byte loads; written to the caller's workspace.
//   k_block_scores  per head, a 128 x 128 tile of  mean(Q_u) . mean(K_v) * scale
//                   (or its exponential) per thread block, 8 x 8 outputs per
//                   thread from shared-memory stages of the two mean matrices.
// The work is a read of Q and K (HBM-bound) and a small fp32 product.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "bsa_internal.h"

namespace bsa {
namespace {


// One thread block (128 threads) per (head, block, tensor).  D / 8 threads
// cover a row with 16-byte loads (8 columns each) and 128 / (D / 8) rows are
// read per pass, so every thread's loads are independent; the row groups'
// partial sums meet in shared memory.  D is a multiple of 8, at most 256.
constexpr int kMeanThreads = 128;
__global__ void __launch_bounds__(kMeanThreads) k_block_means(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k, int32_t N, int32_t D,
    const int32_t* __restrict__ q_map, const int32_t* __restrict__ kv_map, float* __restrict__ means,
    int64_t per_tensor, int32_t* status) {
    __shared__ float part[kMeanThreads * 8];  // [row group][column]
    const int32_t b = blockIdx.x;
    const int64_t bh = blockIdx.y;
    const int which = blockIdx.z;  // 0: Q, 1: K
    const __nv_bfloat16* x = which ? k : q;
    const int32_t* map = which ? kv_map : q_map;
    const int32_t nb = N / kBlock;
    const int lanes_per_row = D / 8;                   // 16-byte chunks per row
    const int groups = kMeanThreads / lanes_per_row;   // rows read per pass
    const int chunk = threadIdx.x % lanes_per_row, grp = threadIdx.x / lanes_per_row;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (grp < groups) {
        for (int32_t t = grp; t < kBlock; t += groups) {
            const int32_t p = b * kBlock + t;
            int32_t i = map ? map[bh * N + p] : p;
            if (i < 0 || i >= N) {
                if (chunk == 0) atomicCAS(status, 0, BSA_ERR_BOUNDS);
                i = 0;
            }
            const uint4 v = *reinterpret_cast<const uint4*>(x + (bh * N + i) * D + chunk * 8);
            const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = __bfloat1622float2(h[e]);
                acc[2 * e] += f.x;
                acc[2 * e + 1] += f.y;
            }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) part[grp * D + chunk * 8 + e] = acc[e];
    }
    __syncthreads();
    for (int32_t d = threadIdx.x; d < D; d += kMeanThreads) {
        float sum = 0.f;
        for (int g = 0; g < groups; ++g) sum += part[g * D + d];
        means[which * per_tensor + (bh * nb + b) * D + d] = sum * (1.0f / kBlock);
    }
}

// One thread block (256 threads) per 128 x 128 tile of one head's score
// matrix.  Per step the block stages 16 columns of the two mean matrices in
// shared memory, transposed (column k of the means is row k of the stage);
// thread (ty, tx) accumulates rows 8 ty .. 8 ty + 7 against columns
// tx + 16 j (j < 8): two 16-byte loads of its rows and eight 4-byte loads of
// its columns per 64 FMAs, and its stores along a row are consecutive across
// the warp's threads.
constexpr int kScoreTile = 128;
constexpr int kScoreK = 16;
__global__ void __launch_bounds__(256) k_block_scores(const float* __restrict__ means,
                                                      int64_t per_tensor, int32_t nb, int32_t D,
                                                      float scale, int32_t mode,
                                                      float* __restrict__ scores) {
    __shared__ __align__(16) float as[kScoreK][kScoreTile + 4];
    __shared__ __align__(16) float bs[kScoreK][kScoreTile + 4];
    const int64_t bh = blockIdx.z;
    const int32_t u0 = blockIdx.y * kScoreTile, v0 = blockIdx.x * kScoreTile;
    const float* qm = means + bh * nb * (int64_t)D;
    const float* km = means + per_tensor + bh * nb * (int64_t)D;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    // staging: thread t copies row t / 2, columns 8 (t % 2) .. + 7 of each tile
    const int sr = threadIdx.x >> 1, sc = (threadIdx.x & 1) * 8;
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
    for (int32_t d0 = 0; d0 < D; d0 += kScoreK) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int32_t d = d0 + sc + j;
            as[sc + j][sr] = (u0 + sr < nb && d < D) ? qm[(int64_t)(u0 + sr) * D + d] : 0.f;
            bs[sc + j][sr] = (v0 + sr < nb && d < D) ? km[(int64_t)(v0 + sr) * D + d] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int c = 0; c < kScoreK; ++c) {
            const float4 a0 = *reinterpret_cast<const float4*>(&as[c][ty * 8]);
            const float4 a1 = *reinterpret_cast<const float4*>(&as[c][ty * 8 + 4]);
            const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            float bv[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) bv[j] = bs[c][tx + 16 * j];
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], bv[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int32_t u = u0 + ty * 8 + i;
        if (u >= nb) continue;
        float* row = scores + (bh * nb + u) * (int64_t)nb;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int32_t v = v0 + tx + 16 * j;
            if (v < nb) {
                const float sv = acc[i][j] * scale;
                row[v] = mode == 1 ? expf(sv) : sv;
            }
        }
    }
}

}  // namespace

size_t block_scores_workspace_bytes(int64_t BH, int32_t N, int32_t D) {
    return (size_t)2 * BH * (N / kBlock) * (size_t)D * sizeof(float);
}

cudaError_t launch_block_scores(const void* q, const void* k, int32_t B, int32_t H, int32_t N,
                                int32_t D, const int32_t* q_map, const int32_t* kv_map, float scale,
                                int32_t mode, float* workspace, float* scores, int32_t* status,
                                cudaStream_t stream) {
    const int64_t BH = (int64_t)B * H;
    const int32_t nb = N / kBlock;
    const int64_t per_tensor = BH * nb * (int64_t)D;
    k_block_means<<<dim3((unsigned)nb, (unsigned)BH, 2), kMeanThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k), N, D, q_map,
        kv_map, workspace, per_tensor, status);
    const unsigned tiles = (unsigned)((nb + kScoreTile - 1) / kScoreTile);
    const float sc = scale > 0.f ? scale : 1.0f / sqrtf((float)D);
    k_block_scores<<<dim3(tiles, tiles, (unsigned)BH), 256, 0, stream>>>(workspace, per_tensor, nb, D,
                                                                         sc, mode, scores);
    return cudaGetLastError();
}

}  // namespace bsa
