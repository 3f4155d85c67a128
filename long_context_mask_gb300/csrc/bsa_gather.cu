// Token rows permuted into gathered order in HBM (bsa_gather_rows).
//
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

}  // namespace

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
