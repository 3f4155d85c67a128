// Spectral row order (WaveAlign section IV-C, "SVD-Based Global Spatial
// Ordering"): per head, the rank-2 embedding of the centered block mask by
// matrix-free subspace iteration, and the rows sorted by polar angle.
//
// One thread block of 1024 threads per head.  The mask is the index lists
// (row r = query block, column c = KV block); it is never formed.  With mu the
// mean row (column means of the mask) and X the nQB x 2 iterate:
//     Z = A^T X - mu (1^T X)         one warp per row scatters X[r] into Z
//                                    with shared-memory atomics
//     Y = A Z   - 1 (mu^T Z)         one warp per row gathers Z over its list
//     X = Gram-Schmidt(Y)            block reductions
// Then theta_r = atan2(X[r][1], X[r][0]) and a bitonic sort of
// (order-preserving key of theta, row) gives the order, ties to the lower
// row.  fp32 throughout; the order is meant as an input to the NNZ-guided
// wave sort (bsa_reorder_rows), where only its coarse grouping matters.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "bsa_internal.h"

namespace bsa {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) red[w] = v;
    __syncthreads();
    float t = l < kWarps ? red[l] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    return t;  // every thread gets the total
}

__device__ void gram_schmidt(float2* X, int32_t n, float* red) {
    float a = 0.f;
    for (int32_t r = threadIdx.x; r < n; r += kThreads) a += X[r].x * X[r].x;
    const float n0 = sqrtf(block_sum(a, red));
    const float i0 = n0 > 0.f ? 1.0f / n0 : 0.f;
    float d = 0.f;
    for (int32_t r = threadIdx.x; r < n; r += kThreads) {
        X[r].x *= i0;
        d += X[r].x * X[r].y;
    }
    d = block_sum(d, red);
    float b = 0.f;
    for (int32_t r = threadIdx.x; r < n; r += kThreads) {
        X[r].y -= d * X[r].x;
        b += X[r].y * X[r].y;
    }
    const float n1 = sqrtf(block_sum(b, red));
    const float i1 = n1 > 0.f ? 1.0f / n1 : 0.f;
    for (int32_t r = threadIdx.x; r < n; r += kThreads) X[r].y *= i1;
    __syncthreads();
}

__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t b = __float_as_uint(f);
    if (b == 0x80000000u) b = 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// dynamic smem: X [nQB] float2 | Z [nKB] float2 | mu [nKB] float | keys [P2] u64
__global__ void __launch_bounds__(kThreads) k_spectral_order(
    const int32_t* __restrict__ kv_idx, const int32_t* __restrict__ kv_cnt, int32_t max_kv,
    int32_t nQB, int32_t nKB, int32_t iters, int32_t p2, const float* __restrict__ x0,
    float* __restrict__ x_out, float* __restrict__ angle, int32_t* __restrict__ order,
    int32_t* status) {
    extern __shared__ __align__(16) uint8_t sm[];
    __shared__ float red[kWarps];
    float2* X = reinterpret_cast<float2*>(sm);
    float2* Z = X + nQB;
    float* mu = reinterpret_cast<float*>(Z + nKB);
    uint64_t* keys = reinterpret_cast<uint64_t*>(sm + (((size_t)nQB * 8 + (size_t)nKB * 12 + 15) & ~(size_t)15));
    const int64_t h = blockIdx.x;
    const int32_t* idx = kv_idx + h * nQB * (int64_t)max_kv;
    const int32_t* cnt = kv_cnt + h * nQB;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    for (int32_t c = threadIdx.x; c < nKB; c += kThreads) mu[c] = 0.f;
    for (int32_t r = threadIdx.x; r < nQB; r += kThreads)
        X[r] = make_float2(x0[(h * nQB + r) * 2], x0[(h * nQB + r) * 2 + 1]);
    __syncthreads();
    // mu = column means of the mask
    for (int32_t r = warp; r < nQB; r += kWarps) {
        int32_t n = cnt[r];
        n = n < 0 ? 0 : (n > max_kv ? max_kv : n);
        for (int32_t e = lane; e < n; e += 32) {
            const int32_t c = idx[r * (int64_t)max_kv + e];
            if (c >= 0 && c < nKB) atomicAdd(&mu[c], 1.0f);
            else atomicCAS(status, 0, BSA_ERR_BOUNDS);
        }
    }
    __syncthreads();
    const float inv_n = 1.0f / (float)nQB;
    for (int32_t c = threadIdx.x; c < nKB; c += kThreads) mu[c] *= inv_n;
    gram_schmidt(X, nQB, red);

    for (int32_t it = 0; it < iters; ++it) {
        float a0 = 0.f, a1 = 0.f;
        for (int32_t r = threadIdx.x; r < nQB; r += kThreads) {
            a0 += X[r].x;
            a1 += X[r].y;
        }
        const float s0 = block_sum(a0, red);
        const float s1 = block_sum(a1, red);
        for (int32_t c = threadIdx.x; c < nKB; c += kThreads) Z[c] = make_float2(0.f, 0.f);
        __syncthreads();
        for (int32_t r = warp; r < nQB; r += kWarps) {  // Z = A^T X
            int32_t n = cnt[r];
            n = n < 0 ? 0 : (n > max_kv ? max_kv : n);
            const float2 x = X[r];
            for (int32_t e = lane; e < n; e += 32) {
                const int32_t c = idx[r * (int64_t)max_kv + e];
                if (c >= 0 && c < nKB) {
                    atomicAdd(&Z[c].x, x.x);
                    atomicAdd(&Z[c].y, x.y);
                }
            }
        }
        __syncthreads();
        float b0 = 0.f, b1 = 0.f;
        for (int32_t c = threadIdx.x; c < nKB; c += kThreads) {  // centering, then mu^T Z
            float2 z = Z[c];
            z.x -= mu[c] * s0;
            z.y -= mu[c] * s1;
            Z[c] = z;
            b0 += mu[c] * z.x;
            b1 += mu[c] * z.y;
        }
        const float m0 = block_sum(b0, red);
        const float m1 = block_sum(b1, red);
        for (int32_t r = warp; r < nQB; r += kWarps) {  // X = A Z - 1 (mu^T Z)
            int32_t n = cnt[r];
            n = n < 0 ? 0 : (n > max_kv ? max_kv : n);
            float y0 = 0.f, y1 = 0.f;
            for (int32_t e = lane; e < n; e += 32) {
                const int32_t c = idx[r * (int64_t)max_kv + e];
                if (c >= 0 && c < nKB) {
                    y0 += Z[c].x;
                    y1 += Z[c].y;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                y0 += __shfl_xor_sync(0xffffffffu, y0, o);
                y1 += __shfl_xor_sync(0xffffffffu, y1, o);
            }
            if (lane == 0) X[r] = make_float2(y0 - m0, y1 - m1);
        }
        __syncthreads();
        gram_schmidt(X, nQB, red);
    }

    // polar angle and sort
    for (int32_t r = threadIdx.x; r < p2; r += kThreads) {
        if (r < nQB) {
            const float th = atan2f(X[r].y, X[r].x);
            if (angle) angle[h * nQB + r] = th;
            if (x_out) {
                x_out[(h * nQB + r) * 2] = X[r].x;
                x_out[(h * nQB + r) * 2 + 1] = X[r].y;
            }
            keys[r] = ((uint64_t)order_key(th) << 32) | (uint32_t)r;
        } else {
            keys[r] = ~0ull;  // padding sorts last
        }
    }
    __syncthreads();
    for (int32_t k = 2; k <= p2; k <<= 1) {
        for (int32_t j = k >> 1; j > 0; j >>= 1) {
            for (int32_t i = threadIdx.x; i < p2; i += kThreads) {
                const int32_t l = i ^ j;
                if (l > i) {
                    const uint64_t a = keys[i], b = keys[l];
                    const bool up = (i & k) == 0;
                    if ((a > b) == up) {
                        keys[i] = b;
                        keys[l] = a;
                    }
                }
            }
            __syncthreads();
        }
    }
    for (int32_t s = threadIdx.x; s < nQB; s += kThreads)
        order[h * nQB + s] = (int32_t)(keys[s] & 0xffffffffu);
}

}  // namespace

size_t spectral_order_smem(int32_t nQB, int32_t nKB, int32_t* p2_out) {
    int32_t p2 = 1;
    while (p2 < nQB) p2 <<= 1;
    if (p2_out) *p2_out = p2;
    return (((size_t)nQB * 8 + (size_t)nKB * 12 + 15) & ~(size_t)15) + (size_t)p2 * 8;
}

cudaError_t launch_spectral_order(const int32_t* kv_idx, const int32_t* kv_cnt, int32_t max_kv,
                                  int64_t heads, int32_t nQB, int32_t nKB, int32_t iters,
                                  const float* x0, float* x_out, float* angle, int32_t* order,
                                  int32_t* status, cudaStream_t stream) {
    if (heads == 0) return cudaSuccess;
    int32_t p2 = 0;
    const size_t smem = spectral_order_smem(nQB, nKB, &p2);
    cudaError_t e = cudaFuncSetAttribute(k_spectral_order, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    k_spectral_order<<<(unsigned)heads, kThreads, smem, stream>>>(kv_idx, kv_cnt, max_kv, nQB, nKB,
                                                                  iters, p2, x0, x_out, angle,
                                                                  order, status);
    return cudaGetLastError();
}

}  // namespace bsa
