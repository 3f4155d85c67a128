// Self-test entry points (see include/bsa_selftest.h): the FMA-pipe exp2 next
// to CUDA's exp2f, and the bounded mbarrier wait giving up on a barrier that
// nothing will ever complete.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "bsa_internal.h"
#include "bsa_math.cuh"
#include "bsa_ptx.cuh"
#include "bsa_selftest.h"

namespace bsa {
namespace {

__global__ void k_selftest_exp2(const float* x, float* y_fma, float* y_mufu, float* y_ref, int64_t n) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    y_fma[i] = exp2_fma(x[i]);
    y_mufu[i] = ex2(x[i]);
    y_ref[i] = exp2f(x[i]);
}

// One thread waits (bounded) on an mbarrier that expects one arrival that
// never comes; on expiry it records BSA_ERR_TIMEOUT, exactly as the forward
// kernel's waits do.
__global__ void k_selftest_wait(uint64_t limit_ns, int32_t* status) {
    __shared__ uint64_t bar;
    const uint32_t b = ptx::smem_u32(&bar);
    if (threadIdx.x == 0) {
        ptx::mbar_init(b, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !ptx::mbar_wait(b, 0, limit_ns, status, BSA_ERR_TIMEOUT))
        atomicCAS(status, 0, BSA_ERR_TIMEOUT);
}

}  // namespace
}  // namespace bsa

extern "C" {

bsa_status bsa_selftest_exp2(const float* x, float* y_fma, float* y_mufu, float* y_ref, int64_t n,
                             void* stream) {
    if (n < 0 || (n > 0 && (!x || !y_fma || !y_mufu || !y_ref))) return BSA_ERR_INVALID_ARG;
    if (n == 0) return BSA_OK;
    const unsigned grid = (unsigned)((n + 255) / 256);
    bsa::k_selftest_exp2<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(x, y_fma, y_mufu,
                                                                              y_ref, n);
    return cudaGetLastError() == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}

bsa_status bsa_selftest_wait_timeout(int64_t limit_ns, void* stream) {
    if (limit_ns < 1000 || limit_ns > 1000000000) return BSA_ERR_INVALID_ARG;
    int32_t* status = bsa::status_word_ptr();
    if (!status) return BSA_ERR_CUDA;
    bsa::k_selftest_wait<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>((uint64_t)limit_ns, status);
    return cudaGetLastError() == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}

}  // extern "C"
