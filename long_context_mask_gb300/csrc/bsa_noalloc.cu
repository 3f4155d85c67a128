// bsa_spectral_order_noalloc: the spectral row order without any allocation.
//
// Some callers cannot allocate device memory at the point where they order
// rows.  Examples: a serving loop or host framework that owns the whole
// device memory pool and forbids allocations once it is running, where an
// allocation could fail or stall in the middle of a step; or an interface
// with no way to thread an extra workspace buffer through to this call.
// This entry point takes its scratch from a fixed array that lives in the
// library itself, so the caller passes only inputs and outputs, and nothing
// here calls cudaMalloc, cudaFree or any allocating library routine.
//
// The array is a file-scope __device__ variable of a fixed maximum size: every
// GPU that loads the library holds it until the process exits.  All calls
// share it and it keeps the previous call's contents; the launch sequence
// clears what must start at zero before using it.  Two calls whose work
// overlaps on the GPU (different streams, or different host threads) race
// on the array and may corrupt each other's result: serialise them.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "bsa.h"
#include "bsa_internal.h"

namespace {

// Scratch of the allocation-free spectral order (one copy per device).
static __device__ __align__(256) float g_noalloc_scratch[BSA_SPECTRAL_NOALLOC_SCRATCH_BYTES / sizeof(float)];

constexpr int kMaxDevices = 64;
float* g_scratch_ptr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device.  In host code
// `g_noalloc_scratch` is only a stand-in symbol; the real address is looked
// up once per device.  The same first call on a device looks up the status
// word and loads the spectral-order kernels: with lazy module loading (the
// default) those steps load modules, which is when the array and the kernels
// take their device memory.  Later calls allocate nothing.
float* scratch_on_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        float* p = nullptr;
        if (cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_noalloc_scratch) != cudaSuccess)
            return nullptr;
        if (bsa::status_word_ptr() == nullptr || bsa::load_spectral_kernels() != cudaSuccess) return nullptr;
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" bsa_status bsa_spectral_order_noalloc(const int32_t* kv_idx, const int32_t* kv_cnt,
                                                 int32_t max_kv, int64_t heads, int32_t nQB,
                                                 int32_t nKB, int32_t iters, const float* x0,
                                                 float* x_out, float* angle, int32_t* order,
                                                 void* stream) {
    // the same argument checks as bsa_spectral_order, first
    if (!bsa::spectral_args_ok(heads, nQB, nKB, max_kv, iters)) return BSA_ERR_INVALID_ARG;
    if (bsa_spectral_order_workspace_size(heads, nQB, nKB) > BSA_SPECTRAL_NOALLOC_SCRATCH_BYTES)
        return BSA_ERR_UNSUPPORTED;  // does not fit the fixed scratch
    if (heads > 0) {
        if (!kv_idx || !kv_cnt || !x0 || !order) return BSA_ERR_INVALID_ARG;
        if (!aligned(kv_idx, 4) || !aligned(kv_cnt, 4) || !aligned(x0, 8) || !aligned(order, 4) ||
            (x_out && !aligned(x_out, 8)) || (angle && !aligned(angle, 4)))
            return BSA_ERR_INVALID_ARG;
    }
    // The per-device set-up (see scratch_on_current_device) runs on every
    // device's first call, before the zero-size early return, so that a
    // heads = 0 call can serve as the warm-up after which no call on that
    // device allocates.
    float* scratch = scratch_on_current_device();
    if (!scratch) return BSA_ERR_CUDA;
    if (heads == 0) return BSA_OK;
    int32_t* status = bsa::status_word_ptr();
    if (!status) return BSA_ERR_CUDA;
    const cudaError_t e =
        bsa::launch_spectral_order(kv_idx, kv_cnt, max_kv, heads, nQB, nKB, iters, x0, scratch,
                                   x_out, angle, order, status, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}
