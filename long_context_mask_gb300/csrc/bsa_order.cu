// Spectral row order (WaveAlign section IV-C, "SVD-Based Global Spatial
// Ordering"): per head, the rank-2 embedding of the centered block mask by
// matrix-free subspace iteration, and the rows sorted by polar angle.
//
// The mask is the index lists (row r = query block, column c = KV block); it
// is never formed.  With mu the mean row (column means of the mask), each
// iteration is
//     Z = A^T X - mu (1^T X)            k_spec_scatter + k_spec_center
//     Y = A Z   - 1 (mu^T Z)            k_spec_gather
//     X = Gram-Schmidt(Y)               folded into the next read of Y
// spread over the whole GPU: one warp per query block, fp32 atomics into a
// caller-provided workspace for Z and the per-head scalars.  X is never
// stored: with the five sums of Y (sum y0, sum y1, |y0|^2, y0.y1, |y1|^2) the
// Gram-Schmidt step is applied on the fly wherever X is read.  A last kernel
// (one block per head) turns X into polar angles and bitonic-sorts
// (order-preserving key of the angle, row), ties to the lower row.
//
// fp32 atomics make the embedding's last bits depend on execution order; the
// order is meant as an input to the NNZ-guided wave sort (bsa_reorder_rows),
// where only its coarse grouping matters.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "bsa_internal.h"

namespace bsa {
namespace {

constexpr int kRowWarps = 8;  // query blocks per thread block in the row kernels
constexpr int kSortThreads = 1024;
constexpr int kScatterWarps = 16;       // shared-memory scatter: warps per block
constexpr int kScatterRows = 64;        // query blocks per block (4 per warp)
constexpr int kScatterSmemMax = 96 * 1024;

// Workspace layout per head (floats): mu[nKB] | Z[2 nKB] | Zc[2 nKB] | Y[2 nQB] | S[2][8]
// S[k]: 0 sum y0, 1 sum y1, 2 |y0|^2, 3 y0.y1, 4 |y1|^2, 5 m0, 6 m1 (k = iteration parity)
struct Ws {
    float* mu;
    float2* Z;
    float2* Zc;
    float2* Y;
    float* S;
};

__host__ __device__ __forceinline__ size_t ws_floats_per_head(int32_t nQB, int32_t nKB) {
    return (size_t)5 * nKB + (size_t)2 * nQB + 16;
}

__device__ __forceinline__ Ws ws_of(float* base, int64_t h, int32_t nQB, int32_t nKB) {
    float* p = base + h * ws_floats_per_head(nQB, nKB);
    Ws w;
    w.mu = p;
    w.Z = reinterpret_cast<float2*>(p + nKB);
    w.Zc = reinterpret_cast<float2*>(p + 3 * (size_t)nKB);
    w.Y = reinterpret_cast<float2*>(p + 5 * (size_t)nKB);
    w.S = p + 5 * (size_t)nKB + 2 * (size_t)nQB;
    return w;
}

// Gram-Schmidt of Y from its sums: x0 = y0 / n0, x1 = (y1 - a y0) / n1 with
// a = (y0.y1) / n0^2 and n1^2 = |y1|^2 - (y0.y1)^2 / n0^2.
struct GS {
    float i0, a, i1;
};
__device__ __forceinline__ GS gs_of(const float* S) {
    const float n00 = S[2], d = S[3], n11 = S[4];
    GS g;
    g.i0 = n00 > 0.f ? rsqrtf(n00) : 0.f;
    g.a = n00 > 0.f ? d / n00 : 0.f;
    const float r = n11 - g.a * d;
    g.i1 = r > 0.f ? rsqrtf(r) : 0.f;
    return g;
}
__device__ __forceinline__ float2 gs_apply(const GS& g, float2 y) {
    return make_float2(y.x * g.i0, (y.y - g.a * y.x) * g.i1);
}

__device__ __forceinline__ int32_t row_len(const int32_t* cnt, int32_t r, int32_t max_kv) {
    const int32_t n = cnt[r];
    return n < 0 ? 0 : (n > max_kv ? max_kv : n);
}

// Block-wide reduction of 5 partial sums into S (atomics, one per block).
__device__ __forceinline__ void add_stats(float (&v)[5], float* S) {
    __shared__ float red[kRowWarps][5];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 0; k < 5; ++k)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v[k] += __shfl_xor_sync(0xffffffffu, v[k], o);
    if (lane == 0)
#pragma unroll
        for (int k = 0; k < 5; ++k) red[warp][k] = v[k];
    __syncthreads();
    if (threadIdx.x < 5) {
        float t = 0.f;
        for (int w = 0; w < kRowWarps; ++w) t += red[w][threadIdx.x];
        atomicAdd(&S[threadIdx.x], t);
    }
}

__global__ void k_spec_zero(float* ws, size_t n) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        ws[i] = 0.f;
}

// Y = x0, the sums of Y into S[0], and the column counts of the mask into mu.
__global__ void __launch_bounds__(kRowWarps * 32) k_spec_init(
    const int32_t* __restrict__ kv_idx, const int32_t* __restrict__ kv_cnt, int32_t max_kv,
    int32_t nQB, int32_t nKB, const float* __restrict__ x0, float* ws, int32_t* status) {
    const int64_t h = blockIdx.y;
    Ws w = ws_of(ws, h, nQB, nKB);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int32_t r = blockIdx.x * kRowWarps + warp;
    float v[5] = {0.f, 0.f, 0.f, 0.f, 0.f};
    if (r < nQB) {
        const int64_t row = h * nQB + r;
        const int32_t n = row_len(kv_cnt, (int32_t)row, max_kv);
        const int32_t* list = kv_idx + row * max_kv;
        for (int32_t e = lane; e < n; e += 32) {
            const int32_t c = list[e];
            if (c >= 0 && c < nKB) atomicAdd(&w.mu[c], 1.0f);
            else atomicCAS(status, 0, BSA_ERR_BOUNDS);
        }
        if (lane == 0) {
            const float2 y = make_float2(x0[row * 2], x0[row * 2 + 1]);
            w.Y[r] = y;
            v[0] = y.x;
            v[1] = y.y;
            v[2] = y.x * y.x;
            v[3] = y.x * y.y;
            v[4] = y.y * y.y;
        }
    }
    add_stats(v, w.S);
}

// Z += A^T X (X from Y and S[par]); the first block of each head clears the
// m slot of this iteration.
__global__ void __launch_bounds__(kRowWarps * 32) k_spec_scatter(
    const int32_t* __restrict__ kv_idx, const int32_t* __restrict__ kv_cnt, int32_t max_kv,
    int32_t nQB, int32_t nKB, int32_t par, float* ws) {
    const int64_t h = blockIdx.y;
    Ws w = ws_of(ws, h, nQB, nKB);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int32_t r = blockIdx.x * kRowWarps + warp;
    float* S = w.S + 8 * par;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        S[5] = 0.f;
        S[6] = 0.f;
    }
    if (r >= nQB) return;
    const GS g = gs_of(S);
    const float2 x = gs_apply(g, w.Y[r]);
    const int64_t row = h * nQB + r;
    const int32_t n = row_len(kv_cnt, (int32_t)row, max_kv);
    const int32_t* list = kv_idx + row * max_kv;
    for (int32_t e = lane; e < n; e += 32) {
        const int32_t c = list[e];
        if (c >= 0 && c < nKB) {
            atomicAdd(&w.Z[c].x, x.x);
            atomicAdd(&w.Z[c].y, x.y);
        }
    }
}

// The same with Z first accumulated in shared memory by kScatterRows query
// blocks, then added to the workspace with one atomic per column (used when
// 8 nKB bytes fit in shared memory).
__global__ void __launch_bounds__(kScatterWarps * 32) k_spec_scatter_smem(
    const int32_t* __restrict__ kv_idx, const int32_t* __restrict__ kv_cnt, int32_t max_kv,
    int32_t nQB, int32_t nKB, int32_t par, float* ws) {
    extern __shared__ float2 zs[];
    const int64_t h = blockIdx.y;
    Ws w = ws_of(ws, h, nQB, nKB);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float* S = w.S + 8 * par;
    for (int32_t c = threadIdx.x; c < nKB; c += blockDim.x) zs[c] = make_float2(0.f, 0.f);
    const GS g = gs_of(S);
    __syncthreads();
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        S[5] = 0.f;
        S[6] = 0.f;
    }
    const int32_t r0 = blockIdx.x * kScatterRows;
    for (int32_t r = r0 + warp; r < r0 + kScatterRows && r < nQB; r += kScatterWarps) {
        const float2 x = gs_apply(g, w.Y[r]);
        const int64_t row = h * nQB + r;
        const int32_t n = row_len(kv_cnt, (int32_t)row, max_kv);
        const int32_t* list = kv_idx + row * max_kv;
        for (int32_t e = lane; e < n; e += 32) {
            const int32_t c = list[e];
            if (c >= 0 && c < nKB) {
                atomicAdd(&zs[c].x, x.x);
                atomicAdd(&zs[c].y, x.y);
            }
        }
    }
    __syncthreads();
    for (int32_t c = threadIdx.x; c < nKB; c += blockDim.x) {
        const float2 z = zs[c];
        if (z.x != 0.f || z.y != 0.f) {
            atomicAdd(&w.Z[c].x, z.x);
            atomicAdd(&w.Z[c].y, z.y);
        }
    }
}

// Zc = Z - mu (1^T X), Z = 0, m = mu^T Zc into S[par]; the first block of
// each head clears the sums of the next Y (S[par ^ 1]).
__global__ void __launch_bounds__(256) k_spec_center(int32_t nQB, int32_t nKB, int32_t par, float* ws) {
    __shared__ float red[8][2];
    const int64_t h = blockIdx.y;
    Ws w = ws_of(ws, h, nQB, nKB);
    float* S = w.S + 8 * par;
    const GS g = gs_of(S);
    const float s0 = S[0] * g.i0;                   // 1^T x0
    const float s1 = (S[1] - g.a * S[0]) * g.i1;    // 1^T x1
    const float inv_n = 1.0f / (float)nQB;
    float m0 = 0.f, m1 = 0.f;
    const int32_t c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c < nKB) {
        const float mu = w.mu[c] * inv_n;
        const float2 z = w.Z[c];
        const float2 zc = make_float2(z.x - mu * s0, z.y - mu * s1);
        w.Zc[c] = zc;
        w.Z[c] = make_float2(0.f, 0.f);
        m0 = mu * zc.x;
        m1 = mu * zc.y;
    }
    if (blockIdx.x == 0 && threadIdx.x < 5) w.S[8 * (par ^ 1) + threadIdx.x] = 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        m0 += __shfl_xor_sync(0xffffffffu, m0, o);
        m1 += __shfl_xor_sync(0xffffffffu, m1, o);
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        red[warp][0] = m0;
        red[warp][1] = m1;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float t0 = 0.f, t1 = 0.f;
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) {
            t0 += red[i][0];
            t1 += red[i][1];
        }
        atomicAdd(&S[5], t0);
        atomicAdd(&S[6], t1);
    }
}

// Y = A Zc - 1 (mu^T Zc), and the sums of the new Y into S[par ^ 1].
__global__ void __launch_bounds__(kRowWarps * 32) k_spec_gather(
    const int32_t* __restrict__ kv_idx, const int32_t* __restrict__ kv_cnt, int32_t max_kv,
    int32_t nQB, int32_t nKB, int32_t par, float* ws) {
    const int64_t h = blockIdx.y;
    Ws w = ws_of(ws, h, nQB, nKB);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int32_t r = blockIdx.x * kRowWarps + warp;
    const float m0 = w.S[8 * par + 5], m1 = w.S[8 * par + 6];
    float v[5] = {0.f, 0.f, 0.f, 0.f, 0.f};
    if (r < nQB) {
        const int64_t row = h * nQB + r;
        const int32_t n = row_len(kv_cnt, (int32_t)row, max_kv);
        const int32_t* list = kv_idx + row * max_kv;
        float y0 = 0.f, y1 = 0.f;
        for (int32_t e = lane; e < n; e += 32) {
            const int32_t c = list[e];
            if (c >= 0 && c < nKB) {
                const float2 z = w.Zc[c];
                y0 += z.x;
                y1 += z.y;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            y0 += __shfl_xor_sync(0xffffffffu, y0, o);
            y1 += __shfl_xor_sync(0xffffffffu, y1, o);
        }
        if (lane == 0) {
            const float2 y = make_float2(y0 - m0, y1 - m1);
            w.Y[r] = y;
            v[0] = y.x;
            v[1] = y.y;
            v[2] = y.x * y.x;
            v[3] = y.x * y.y;
            v[4] = y.y * y.y;
        }
    }
    add_stats(v, w.S + 8 * (par ^ 1));
}

__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t b = __float_as_uint(f);
    if (b == 0x80000000u) b = 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// X from Y and S[par], polar angles, bitonic sort; one block per head.
// dynamic smem: keys [p2] u64
__global__ void __launch_bounds__(kSortThreads) k_spec_sort(int32_t nQB, int32_t nKB, int32_t par,
                                                            int32_t p2, const float* ws,
                                                            float* __restrict__ x_out,
                                                            float* __restrict__ angle,
                                                            int32_t* __restrict__ order) {
    extern __shared__ uint64_t keys[];
    const int64_t h = blockIdx.x;
    Ws w = ws_of(const_cast<float*>(ws), h, nQB, nKB);
    const GS g = gs_of(w.S + 8 * par);
    for (int32_t r = threadIdx.x; r < p2; r += kSortThreads) {
        if (r < nQB) {
            const float2 x = gs_apply(g, w.Y[r]);
            const float th = atan2f(x.y, x.x);
            if (angle) angle[h * nQB + r] = th;
            if (x_out) {
                x_out[(h * nQB + r) * 2] = x.x;
                x_out[(h * nQB + r) * 2 + 1] = x.y;
            }
            keys[r] = ((uint64_t)order_key(th) << 32) | (uint32_t)r;
        } else {
            keys[r] = ~0ull;  // padding sorts last
        }
    }
    __syncthreads();
    for (int32_t k = 2; k <= p2; k <<= 1) {
        for (int32_t j = k >> 1; j > 0; j >>= 1) {
            for (int32_t i = threadIdx.x; i < p2; i += kSortThreads) {
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
    for (int32_t s = threadIdx.x; s < nQB; s += kSortThreads)
        order[h * nQB + s] = (int32_t)(keys[s] & 0xffffffffu);
}

}  // namespace

cudaError_t load_spectral_kernels() {
    // querying a kernel's attributes loads its module when modules load lazily
    cudaFuncAttributes fa;
    const void* fns[] = {(const void*)k_spec_zero,   (const void*)k_spec_init,   (const void*)k_spec_scatter,
                         (const void*)k_spec_scatter_smem, (const void*)k_spec_center,
                         (const void*)k_spec_gather, (const void*)k_spec_sort};
    for (const void* f : fns) {
        const cudaError_t e = cudaFuncGetAttributes(&fa, f);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

size_t spectral_order_workspace_bytes(int64_t heads, int32_t nQB, int32_t nKB) {
    return (size_t)heads * ws_floats_per_head(nQB, nKB) * sizeof(float);
}

cudaError_t launch_spectral_order(const int32_t* kv_idx, const int32_t* kv_cnt, int32_t max_kv,
                                  int64_t heads, int32_t nQB, int32_t nKB, int32_t iters,
                                  const float* x0, float* workspace, float* x_out, float* angle,
                                  int32_t* order, int32_t* status, cudaStream_t stream) {
    if (heads == 0) return cudaSuccess;
    int32_t p2 = 1;
    while (p2 < nQB) p2 <<= 1;
    const size_t sort_smem = (size_t)p2 * sizeof(uint64_t);
    cudaError_t e = cudaFuncSetAttribute(k_spec_sort, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)sort_smem);
    if (e != cudaSuccess) return e;
    const size_t n_ws = (size_t)heads * ws_floats_per_head(nQB, nKB);
    const dim3 rows_grid((unsigned)((nQB + kRowWarps - 1) / kRowWarps), (unsigned)heads);
    const dim3 cols_grid((unsigned)((nKB + 255) / 256), (unsigned)heads);
    k_spec_zero<<<(unsigned)((n_ws + 1023) / 1024 < 4096 ? (n_ws + 1023) / 1024 : 4096), 1024, 0, stream>>>(
        workspace, n_ws);
    k_spec_init<<<rows_grid, kRowWarps * 32, 0, stream>>>(kv_idx, kv_cnt, max_kv, nQB, nKB, x0,
                                                          workspace, status);
    const size_t zs_bytes = (size_t)nKB * sizeof(float2);
    const bool smem_scatter = zs_bytes <= (size_t)kScatterSmemMax;
    if (smem_scatter) {
        e = cudaFuncSetAttribute(k_spec_scatter_smem, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)zs_bytes);
        if (e != cudaSuccess) return e;
    }
    const dim3 scat_grid((unsigned)((nQB + kScatterRows - 1) / kScatterRows), (unsigned)heads);
    int32_t par = 0;
    for (int32_t it = 0; it < iters; ++it, par ^= 1) {
        if (smem_scatter)
            k_spec_scatter_smem<<<scat_grid, kScatterWarps * 32, zs_bytes, stream>>>(
                kv_idx, kv_cnt, max_kv, nQB, nKB, par, workspace);
        else
            k_spec_scatter<<<rows_grid, kRowWarps * 32, 0, stream>>>(kv_idx, kv_cnt, max_kv, nQB,
                                                                     nKB, par, workspace);
        k_spec_center<<<cols_grid, 256, 0, stream>>>(nQB, nKB, par, workspace);
        k_spec_gather<<<rows_grid, kRowWarps * 32, 0, stream>>>(kv_idx, kv_cnt, max_kv, nQB, nKB,
                                                                par, workspace);
    }
    k_spec_sort<<<(unsigned)heads, kSortThreads, sort_smem, stream>>>(nQB, nKB, par, p2, workspace,
                                                                      x_out, angle, order);
    return cudaGetLastError();
}

}  // namespace bsa
