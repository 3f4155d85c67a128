// Index-list construction, row reordering and block sampling kernels.
//
//  * Predicate compaction (mask / threshold map -> ascending KV-block lists):
//    one warp per row; each 32-block chunk is one __ballot_sync word, and a
//    block's slot is its prefix popcount.  ScalingAttention, section 5.2
//    eq. (2) (M_p = I(T <= p)) and section 7.2 (a 32-block bitmask word per
//    load); WaveAlign, "B. Sparse Attention for Long-Video Generation".
//  * Top-k (MC-Sparse, "The MC-Sparse Architecture"; InstaGen 3.2.1): one
//    warp per row, a 1-bit-per-pass radix select of the k-th largest
//    order-preserving key, ties resolved toward the lower block index with a
//    ballot scan, then the same ballot compaction.
//  * Row reordering (WaveAlign section IV-D): one thread block per
//    (head, bucket of W slots); each row's slot in its bucket is its rank
//    under (count descending, input position ascending).
//  * Block sampling (InstaGen section 3.2.1 eq. (4), systematic PPS,
//    Algorithm 1 step 13): one thread per row, fp32, fixed summation order,
//    explicit round-to-nearest arithmetic (never fused).
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "bsa_internal.h"

namespace bsa {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ void raise_status(int32_t* status, int32_t code) {
    atomicCAS(status, 0, code);
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// ------------------------------------------------------------ compaction
template <int MODE>
__device__ __forceinline__ bool keep_block(const void* src, int64_t off, float p) {
    if (MODE == BSA_IDX_MASK_U8) return static_cast<const uint8_t*>(src)[off] != 0;
    return static_cast<const float*>(src)[off] <= p;
}

template <int MODE>
__global__ void __launch_bounds__(256) k_index_predicate(const void* __restrict__ src, int64_t rows,
                                                         int32_t nKB, float p,
                                                         int32_t* __restrict__ kv_idx,
                                                         int32_t* __restrict__ kv_cnt,
                                                         int32_t max_kv, int32_t* status) {
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const int64_t base_in = row * (int64_t)nKB;
    int32_t* out = kv_idx + row * (int64_t)max_kv;
    int32_t n = 0;
    for (int32_t c = 0; c < nKB; c += 32) {
        const int32_t kb = c + lane;
        const bool keep = kb < nKB && keep_block<MODE>(src, base_in + kb, p);
        const uint32_t word = __ballot_sync(kFull, keep);
        const int32_t pos = n + __popc(word & lanemask_lt());
        if (keep && pos < max_kv) out[pos] = kb;
        n += __popc(word);
    }
    const int32_t kept = n < max_kv ? n : max_kv;
    for (int32_t e = kept + lane; e < max_kv; e += 32) out[e] = -1;
    if (lane == 0) {
        kv_cnt[row] = kept;
        if (n > max_kv) raise_status(status, BSA_ERR_OVERFLOW);
    }
}

// ------------------------------------------------------------ CRM rows
// The ballot word of each 32-block chunk is the row's CRM word (ScalingAttention
// section 7.2): one warp per row, lane 0 stores the word.
template <int MODE>
__global__ void __launch_bounds__(256) k_crm_rows(const void* __restrict__ src, int64_t rows,
                                                  int32_t nKB, float p, uint32_t* __restrict__ words,
                                                  int32_t n_words) {
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const int64_t base_in = row * (int64_t)nKB;
    for (int32_t w = 0; w < n_words; ++w) {
        const int32_t kb = 32 * w + lane;
        const bool keep = kb < nKB && keep_block<MODE>(src, base_in + kb, p);
        const uint32_t word = __ballot_sync(kFull, keep);
        if (lane == 0) words[row * (int64_t)n_words + w] = word;
    }
}

// ------------------------------------------------------------ eq. (7) upscaling
// Target (u, v) samples base (u Ub / Ut, v Vb / Vt); the lower neighbour always
// has a nonzero bilinear weight, the upper one only when the coordinate is
// fractional (integer test).  The ceiling rule on every mask M_p = I(T <= p)
// is the minimum of T over the neighbours with nonzero weight.
__global__ void k_upscale_threshold(const float* __restrict__ T, int32_t Ub, int32_t Vb, int32_t Ut,
                                    int32_t Vt, float* __restrict__ out) {
    const int64_t h = blockIdx.z;
    const int32_t u = blockIdx.y;
    const int32_t v = blockIdx.x * blockDim.x + threadIdx.x;
    if (v >= Vt) return;
    const int64_t xu = (int64_t)u * Ub, yv = (int64_t)v * Vb;
    const int32_t i0 = (int32_t)(xu / Ut), j0 = (int32_t)(yv / Vt);
    const int32_t i1 = (xu % Ut != 0 && i0 + 1 < Ub) ? i0 + 1 : i0;
    const int32_t j1 = (yv % Vt != 0 && j0 + 1 < Vb) ? j0 + 1 : j0;
    const float* b = T + h * (int64_t)Ub * Vb;
    const float m = fminf(fminf(b[(int64_t)i0 * Vb + j0], b[(int64_t)i0 * Vb + j1]),
                          fminf(b[(int64_t)i1 * Vb + j0], b[(int64_t)i1 * Vb + j1]));
    out[(h * Ut + u) * (int64_t)Vt + v] = m;
}

// ------------------------------------------------------------ top-k
// Order-preserving map fp32 -> uint32 (larger float -> larger key); -0 == +0.
__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t b = __float_as_uint(f);
    if (b == 0x80000000u) b = 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// kRegs > 0: the row (nKB <= 32 * kRegs) is read once into registers, lane l
// holding blocks l, l + 32, ...; kRegs = 0: every pass re-reads it (through L1).
template <int kRegs>
__global__ void __launch_bounds__(256) k_index_topk(const float* __restrict__ scores, int64_t rows,
                                                    int32_t nKB, const int32_t* __restrict__ k_per_row,
                                                    int32_t k_const, int32_t* __restrict__ kv_idx,
                                                    int32_t* __restrict__ kv_cnt, int32_t max_kv,
                                                    int32_t* status) {
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const float* s = scores + row * (int64_t)nKB;
    int32_t* out = kv_idx + row * (int64_t)max_kv;
    int32_t k = k_per_row ? k_per_row[row] : k_const;
    k = k < 0 ? 0 : (k > nKB ? nKB : k);
    // keys of blocks lane + 32 i; 0 past the end (0 is below every candidate,
    // which has a bit set, and the selection checks the bound)
    uint32_t key[kRegs > 0 ? kRegs : 1];
    if constexpr (kRegs > 0) {
#pragma unroll
        for (int i = 0; i < kRegs; ++i) {
            const int32_t kb = lane + 32 * i;
            key[i] = kb < nKB ? order_key(s[kb]) : 0u;
        }
    }

    int32_t n = 0;
    if (k > 0) {
        // Largest key value T with #{key >= T} >= k, one bit per pass.
        uint32_t T = 0;
        for (int bit = 31; bit >= 0; --bit) {
            const uint32_t cand = T | (1u << bit);
            int32_t c = 0;
            if constexpr (kRegs > 0) {
#pragma unroll
                for (int i = 0; i < kRegs; ++i) c += key[i] >= cand;
            } else {
                for (int32_t kb = lane; kb < nKB; kb += 32) c += order_key(s[kb]) >= cand;
            }
            if (__reduce_add_sync(kFull, c) >= k) T = cand;
        }
        int32_t gt = 0;
        if constexpr (kRegs > 0) {
#pragma unroll
            for (int i = 0; i < kRegs; ++i) gt += key[i] > T;
        } else {
            for (int32_t kb = lane; kb < nKB; kb += 32) gt += order_key(s[kb]) > T;
        }
        gt = __reduce_add_sync(kFull, gt);
        const int32_t need_eq = k - gt;  // >= 1: equal keys taken from the lowest block up
        int32_t eq_seen = 0;
        // blocks c .. c + 31 (this lane: c + lane, key kk), selected in
        // ascending block order; ties resolved by the ballot of equal keys
        auto pick = [&](int32_t c, uint32_t kk) {
            const int32_t kb = c + lane;
            const bool eq = kb < nKB && kk == T;
            const uint32_t eq_word = __ballot_sync(kFull, eq);
            const bool sel = kb < nKB && (kk > T || (eq && eq_seen + __popc(eq_word & lanemask_lt()) < need_eq));
            eq_seen += __popc(eq_word);
            const uint32_t word = __ballot_sync(kFull, sel);
            const int32_t pos = n + __popc(word & lanemask_lt());
            if (sel && pos < max_kv) out[pos] = kb;
            n += __popc(word);
        };
        if constexpr (kRegs > 0) {
#pragma unroll
            for (int i = 0; i < kRegs; ++i)
                if (32 * i < nKB) pick(32 * i, key[i]);
        } else {
            for (int32_t c = 0; c < nKB; c += 32) pick(c, c + lane < nKB ? order_key(s[c + lane]) : 0u);
        }
    }
    const int32_t kept = n < max_kv ? n : max_kv;
    for (int32_t e = kept + lane; e < max_kv; e += 32) out[e] = -1;
    if (lane == 0) {
        kv_cnt[row] = kept;
        if (n > max_kv) raise_status(status, BSA_ERR_OVERFLOW);
    }
}

// ------------------------------------------------------------ reorder
// grid: (buckets per head, heads); dynamic smem: 2 * W int32.
__global__ void __launch_bounds__(256) k_reorder_rows(const int32_t* __restrict__ kv_cnt,
                                                      const int32_t* __restrict__ order_in,
                                                      int32_t nQB, int32_t wave,
                                                      int32_t* __restrict__ row_perm,
                                                      int32_t* status) {
    extern __shared__ int32_t sm[];
    const int64_t h = blockIdx.y;
    const int32_t b0 = blockIdx.x * wave;
    const int32_t len = min(wave, nQB - b0);
    int32_t* s_qb = sm;
    int32_t* s_cnt = sm + wave;
    for (int32_t i = threadIdx.x; i < len; i += blockDim.x) {
        int32_t qb = order_in ? order_in[h * nQB + b0 + i] : b0 + i;
        if (qb < 0 || qb >= nQB) {
            raise_status(status, BSA_ERR_BOUNDS);
            qb = 0;
        }
        s_qb[i] = qb;
        s_cnt[i] = kv_cnt[h * nQB + qb];
    }
    __syncthreads();
    for (int32_t i = threadIdx.x; i < len; i += blockDim.x) {
        const int32_t ci = s_cnt[i];
        int32_t rank = 0;
        for (int32_t j = 0; j < len; ++j) {
            const int32_t cj = s_cnt[j];
            rank += (cj > ci) | ((cj == ci) & (j < i));
        }
        row_perm[h * nQB + b0 + rank] = s_qb[i];
    }
}

// ------------------------------------------------------------ sampling
constexpr int kMaxSampleKB = 4096;
constexpr int kWords = kMaxSampleKB / 32;


// One thread per row, 64 rows per block.  The scores are read in 32 x 32 tiles
// per warp (coalesced) and each lane then walks its own row in ascending block
// order: the sums must run in that order, one row per thread, to match the
// oracle bit for bit.  The exact / promoted set of each row is a bitset in
// shared memory (word w of thread t at w * 64 + t: conflict-free).
constexpr int kSampleThreads = 64;
static_assert(kSampleThreads == kSampleRowsPerBlock, "the host bounds rows by this launch shape");

__global__ void __launch_bounds__(kSampleThreads) k_sample_blocks(
    const float* __restrict__ scores, int64_t rows, int32_t nKB, const int32_t* __restrict__ exact_idx,
    const int32_t* __restrict__ exact_cnt, int32_t exact_stride, int32_t m,
    const double* __restrict__ u, int32_t* __restrict__ kv_idx, int32_t* __restrict__ kv_cnt,
    float* __restrict__ log_w, int32_t max_kv, int32_t* status) {
    __shared__ float tile[kSampleThreads / 32][32][33];
    __shared__ uint32_t taken_s[kWords * kSampleThreads];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t row0 = (int64_t)blockIdx.x * kSampleThreads;
    const int64_t row = row0 + tid;
    const bool active = row < rows;
    const int32_t nw = (nKB + 31) >> 5;
    auto taken = [&](int32_t kb) -> bool { return (taken_s[(kb >> 5) * kSampleThreads + tid] >> (kb & 31)) & 1u; };
    auto take = [&](int32_t kb) { taken_s[(kb >> 5) * kSampleThreads + tid] |= 1u << (kb & 31); };
    for (int32_t w = 0; w < nw; ++w) taken_s[w * kSampleThreads + tid] = 0u;
    int32_t n_res = nKB;
    if (active) {
        const int32_t ec = exact_cnt[row];
        for (int32_t e = 0; e < ec; ++e) {
            const int32_t kb = exact_idx[row * (int64_t)exact_stride + e];
            if (kb < 0 || kb >= nKB) {
                raise_status(status, BSA_ERR_BOUNDS);
                continue;
            }
            if (!taken(kb)) {
                take(kb);
                --n_res;
            }
        }
    }
    // Columns c0 .. c0 + 31 of this warp's 32 rows into its tile (1 for the
    // uniform sampler); lane l then reads its row from tile[warp][l][*].
    // The next chunk's 32 loads are issued before the current chunk is
    // processed (one chunk in flight in registers), so their latency overlaps
    // the sequential per-row work.
    float pre[32];
    auto fetch = [&](int32_t c0) {
        const int32_t c = c0 + lane;
#pragma unroll
        for (int rr = 0; rr < 32; ++rr) {
            const int64_t rw = row0 + warp * 32 + rr;
            pre[rr] = (scores != nullptr && rw < rows && c < nKB) ? __ldg(scores + rw * nKB + c) : 1.0f;
        }
    };
    auto load_tile = [&](int32_t c0) {  // chunk c0 (already fetched) into the tile; fetch the next
        __syncwarp();
#pragma unroll
        for (int rr = 0; rr < 32; ++rr) tile[warp][rr][lane] = pre[rr];
        __syncwarp();
        fetch(c0 + 32 < nKB ? c0 + 32 : 0);  // wraps to the start for the next pass
    };
    fetch(0);

    // fp32 throughout, IEEE round-to-nearest without contraction, sums in
    // ascending block order: these values decide which blocks are drawn
    const bool all_promoted = n_res <= m;  // the budget covers the residual: pi = 1 everywhere
    float lambda = 0.0f;
    int32_t n_cap = 0;
    bool iterate = active && !all_promoted;
    // eq. (4): cap at 1 and renormalise until the capped set is stable
    while (__any_sync(0xffffffffu, iterate)) {
        float sum = 0.0f, smax = 0.0f;
        for (int32_t c0 = 0; c0 < nKB; c0 += 32) {
            load_tile(c0);
            if (iterate) {
                // skipped blocks add +0 (x + 0 = x exactly), past-the-end columns too
                const uint32_t tw = taken_s[(c0 >> 5) * kSampleThreads + tid];
                const int32_t cn = nKB - c0 < 32 ? nKB - c0 : 32;
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const bool skip = c >= cn || ((tw >> c) & 1u);
                    const float x = skip ? 0.0f : tile[warp][lane][c];
                    sum = __fadd_rn(sum, x);
                    smax = fmaxf(smax, x);
                }
            }
        }
        if (iterate) {
            lambda = __fdiv_rn((float)(m - n_cap), sum);
            // rounding is monotone: if the largest score stays below 1, all do
            if (__fmul_rn(lambda, smax) < 1.0f) iterate = false;
        }
        if (!__any_sync(0xffffffffu, iterate)) break;
        bool grew = false;
        for (int32_t c0 = 0; c0 < nKB; c0 += 32) {
            load_tile(c0);
            if (iterate) {
                const int32_t cn = nKB - c0 < 32 ? nKB - c0 : 32;
                for (int32_t c = 0; c < cn; ++c) {
                    if (!taken(c0 + c) && __fmul_rn(lambda, tile[warp][lane][c]) >= 1.0f) {
                        take(c0 + c);
                        ++n_cap;
                        grew = true;
                    }
                }
            }
        }
        if (!grew) iterate = false;
    }

    // Systematic PPS over the uncapped residual in ascending block order,
    // merged with the exact and promoted blocks into the output list.
    const int32_t m_rest = m - n_cap;
    const float ur = active ? __double2float_rn(u[row]) : 0.0f;
    float C = 0.0f;
    int32_t nd = 0, n = 0, total = 0;
    int32_t* out = kv_idx + row * (int64_t)max_kv;
    float* lw = log_w + row * (int64_t)max_kv;
    auto emit = [&](int32_t kb, float w) {
        if (n < max_kv) {
            out[n] = kb;
            lw[n] = w;
            ++n;
        }
        ++total;
    };
    for (int32_t c0 = 0; c0 < nKB; c0 += 32) {
        load_tile(c0);
        if (!active) continue;
        const int32_t cn = nKB - c0 < 32 ? nKB - c0 : 32;
        const uint32_t tw = all_promoted ? ~0u : taken_s[(c0 >> 5) * kSampleThreads + tid];
#pragma unroll 8
        for (int32_t c = 0; c < cn; ++c) {
            const int32_t kb = c0 + c;
            if ((tw >> c) & 1u) {
                emit(kb, 0.0f);
                continue;
            }
            if (nd < m_rest) {
                const float pj = __fmul_rn(lambda, tile[warp][lane][c]);
                const float C_prev = C;
                C = __fadd_rn(C, pj);
                if (ceilf(__fsub_rn(C, ur)) > ceilf(__fsub_rn(C_prev, ur))) {
                    // drawn: log-weight -log(pi) (fp32 log; fp64 issue is slow here)
                    emit(kb, -logf(pj));
                    ++nd;
                }
            }
        }
    }
    if (!active) return;
    for (int32_t e = n; e < max_kv; ++e) {
        out[e] = -1;
        lw[e] = 0.0f;
    }
    kv_cnt[row] = n;
    if (total > max_kv) raise_status(status, BSA_ERR_OVERFLOW);
}

}  // namespace

cudaError_t launch_index_predicate(bsa_idx_mode mode, const void* src, int64_t rows, int32_t nKB,
                                   float p, int32_t* kv_idx, int32_t* kv_cnt, int32_t max_kv,
                                   int32_t* status, cudaStream_t stream) {
    if (rows == 0) return cudaSuccess;
    const int warps = kListRowsPerBlock;
    const dim3 grid((unsigned)((rows + warps - 1) / warps));
    if (mode == BSA_IDX_MASK_U8)
        k_index_predicate<BSA_IDX_MASK_U8><<<grid, warps * 32, 0, stream>>>(src, rows, nKB, p, kv_idx,
                                                                           kv_cnt, max_kv, status);
    else
        k_index_predicate<BSA_IDX_THRESHOLD_F32><<<grid, warps * 32, 0, stream>>>(
            src, rows, nKB, p, kv_idx, kv_cnt, max_kv, status);
    return cudaGetLastError();
}

cudaError_t launch_crm_rows(bsa_idx_mode mode, const void* src, int64_t rows, int32_t nKB, float p,
                            uint32_t* words, int32_t n_words, cudaStream_t stream) {
    if (rows == 0) return cudaSuccess;
    const dim3 grid((unsigned)((rows + kListRowsPerBlock - 1) / kListRowsPerBlock));
    if (mode == BSA_IDX_MASK_U8)
        k_crm_rows<BSA_IDX_MASK_U8><<<grid, kListRowsPerBlock * 32, 0, stream>>>(src, rows, nKB, p, words, n_words);
    else
        k_crm_rows<BSA_IDX_THRESHOLD_F32><<<grid, kListRowsPerBlock * 32, 0, stream>>>(src, rows, nKB, p, words, n_words);
    return cudaGetLastError();
}

cudaError_t launch_upscale_threshold(const float* T, int64_t heads, int32_t Ub, int32_t Vb,
                                     int32_t Ut, int32_t Vt, float* out, cudaStream_t stream) {
    if (heads == 0) return cudaSuccess;
    const dim3 grid((unsigned)((Vt + 127) / 128), (unsigned)Ut, (unsigned)heads);
    k_upscale_threshold<<<grid, 128, 0, stream>>>(T, Ub, Vb, Ut, Vt, out);
    return cudaGetLastError();
}

cudaError_t launch_index_topk(const float* scores, int64_t rows, int32_t nKB,
                              const int32_t* k_per_row, int32_t k_const, int32_t* kv_idx,
                              int32_t* kv_cnt, int32_t max_kv, int32_t* status,
                              cudaStream_t stream) {
    if (rows == 0) return cudaSuccess;
    const int warps = kListRowsPerBlock;
    const dim3 grid((unsigned)((rows + warps - 1) / warps));
    if (nKB <= 32 * 32)
        k_index_topk<32><<<grid, warps * 32, 0, stream>>>(scores, rows, nKB, k_per_row, k_const, kv_idx,
                                                          kv_cnt, max_kv, status);
    else
        k_index_topk<0><<<grid, warps * 32, 0, stream>>>(scores, rows, nKB, k_per_row, k_const, kv_idx,
                                                         kv_cnt, max_kv, status);
    return cudaGetLastError();
}

cudaError_t launch_reorder_rows(const int32_t* kv_cnt, const int32_t* order_in, int64_t heads,
                                int32_t nQB, int32_t wave, int32_t* row_perm, int32_t* status,
                                cudaStream_t stream) {
    if (heads == 0) return cudaSuccess;
    const int32_t w = wave < nQB ? wave : nQB;
    const dim3 grid((unsigned)((nQB + w - 1) / w), (unsigned)heads);
    const size_t smem = (size_t)2 * w * sizeof(int32_t);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(k_reorder_rows,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    k_reorder_rows<<<grid, 256, smem, stream>>>(kv_cnt, order_in, nQB, w, row_perm, status);
    return cudaGetLastError();
}

cudaError_t launch_sample_blocks(const float* scores, int64_t rows, int32_t nKB,
                                 const int32_t* exact_idx, const int32_t* exact_cnt,
                                 int32_t exact_stride, int32_t m, const double* u,
                                 int32_t* kv_idx, int32_t* kv_cnt, float* log_w, int32_t max_kv,
                                 int32_t* status, cudaStream_t stream) {
    if (rows == 0) return cudaSuccess;
    const dim3 grid((unsigned)((rows + kSampleThreads - 1) / kSampleThreads));
    k_sample_blocks<<<grid, kSampleThreads, 0, stream>>>(scores, rows, nKB, exact_idx, exact_cnt, exact_stride,
                                              m, u, kv_idx, kv_cnt, log_w, max_kv, status);
    return cudaGetLastError();
}

}  // namespace bsa
