// C-ABI entry points of libbsa.so: argument validation, the per-device
// status word, and dispatch to the kernels.  Every check here runs on the
// host before anything is launched, so a rejected call touches no device.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "bsa.h"
#include "bsa_internal.h"

namespace bsa {
namespace {

// First device-side error since the last bsa_device_status(); one per device.
__device__ int32_t g_status_word = 0;

constexpr int kMaxDevices = 64;
int32_t* g_status_ptr[kMaxDevices] = {nullptr};
std::mutex g_status_mu;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// A logit scale must be finite (<= 0 selects 1/sqrt(D)).
bool scale_ok(float s) { return s == s && s - s == 0.0f; }

}  // namespace

int32_t* status_word_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_status_mu);
    if (g_status_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<int32_t*>(p);
    }
    return g_status_ptr[dev];
}

}  // namespace bsa

using bsa::aligned;
using bsa::scale_ok;

extern "C" {

const char* bsa_status_string(int32_t s) {
    switch (s) {
        case BSA_OK: return "BSA_OK";
        case BSA_ERR_INVALID_ARG: return "BSA_ERR_INVALID_ARG";
        case BSA_ERR_UNSUPPORTED: return "BSA_ERR_UNSUPPORTED";
        case BSA_ERR_OVERFLOW: return "BSA_ERR_OVERFLOW";
        case BSA_ERR_CUDA: return "BSA_ERR_CUDA";
        case BSA_ERR_TIMEOUT: return "BSA_ERR_TIMEOUT";
        case BSA_ERR_BOUNDS: return "BSA_ERR_BOUNDS";
        default: return "BSA_ERR_UNKNOWN";
    }
}

bsa_status bsa_build_index(bsa_idx_mode mode, const void* src, int64_t rows, int32_t nKB, float p,
                           const int32_t* k_per_row, int32_t k_const, int32_t* kv_idx,
                           int32_t* kv_cnt, int32_t max_kv, void* stream) {
    if (mode != BSA_IDX_MASK_U8 && mode != BSA_IDX_THRESHOLD_F32 && mode != BSA_IDX_TOPK_F32)
        return BSA_ERR_INVALID_ARG;
    if (rows < 0 || nKB < 1 || nKB > 65536 || max_kv < 1 || max_kv > nKB) return BSA_ERR_INVALID_ARG;
    if (rows > bsa::kListRowsPerBlock * bsa::kMaxGridX) return BSA_ERR_INVALID_ARG;
    if (rows == 0) return BSA_OK;
    if (!src || !kv_idx || !kv_cnt) return BSA_ERR_INVALID_ARG;
    if (!aligned(kv_idx, 4) || !aligned(kv_cnt, 4)) return BSA_ERR_INVALID_ARG;
    if (mode != BSA_IDX_MASK_U8 && !aligned(src, 4)) return BSA_ERR_INVALID_ARG;
    if (mode == BSA_IDX_TOPK_F32) {
        if (k_per_row && !aligned(k_per_row, 4)) return BSA_ERR_INVALID_ARG;
        if (!k_per_row && k_const < 0) return BSA_ERR_INVALID_ARG;
    }
    int32_t* status = bsa::status_word_ptr();
    if (!status) return BSA_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (mode == BSA_IDX_TOPK_F32)
        e = bsa::launch_index_topk(static_cast<const float*>(src), rows, nKB, k_per_row, k_const,
                                   kv_idx, kv_cnt, max_kv, status, st);
    else
        e = bsa::launch_index_predicate(mode, src, rows, nKB, p, kv_idx, kv_cnt, max_kv, status, st);
    return e == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}

bsa_status bsa_reorder_rows(const int32_t* kv_cnt, const int32_t* order_in, int64_t heads,
                            int32_t nQB, int32_t wave, int32_t* row_perm, void* stream) {
    if (heads < 0 || heads > 65535 || nQB < 1 || nQB > 65536 || wave < 1 || wave > 8192)
        return BSA_ERR_INVALID_ARG;
    if (heads == 0) return BSA_OK;
    if (!kv_cnt || !row_perm) return BSA_ERR_INVALID_ARG;
    if (!aligned(kv_cnt, 4) || !aligned(row_perm, 4) || (order_in && !aligned(order_in, 4)))
        return BSA_ERR_INVALID_ARG;
    int32_t* status = bsa::status_word_ptr();
    if (!status) return BSA_ERR_CUDA;
    cudaError_t e = bsa::launch_reorder_rows(kv_cnt, order_in, heads, nQB, wave, row_perm, status,
                                             static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}

bsa_status bsa_reorder_guard(const bsa_guard_args* a, bsa_guard_result* r) {
    if (!a || !r) return BSA_ERR_INVALID_ARG;
    if (a->heads < 1 || a->kv_heads < 1 || a->kv_heads > a->heads || a->nQB < 1 || a->nKB < 1 || a->D < 1 ||
        a->listed_blocks < 0 || !(a->l2_bytes >= 0.0) || !(a->tensor_tflops >= 0.0) || !(a->hbm_gbs >= 0.0))
        return BSA_ERR_INVALID_ARG;
    double l2 = a->l2_bytes;
    if (l2 == 0.0) {
        int dev = 0, bytes = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&bytes, cudaDevAttrL2CacheSize, dev) != cudaSuccess || bytes <= 0)
            return BSA_ERR_CUDA;
        l2 = (double)bytes;
    }
    const double flops_rate = (a->tensor_tflops > 0.0 ? a->tensor_tflops : 1500.0) * 1e12;  // FLOP/s
    const double bw = (a->hbm_gbs > 0.0 ? a->hbm_gbs : 6800.0) * 1e9;                       // B/s
    const double D = a->D, listed = (double)a->listed_blocks;
    const double rows_q = (double)a->heads * a->nQB * 128.0;  // query tokens
    const double F = (double)a->nKB * 128.0 * D * 4.0;       // one head's K and V
    const double C = 0.5 * l2;
    const double mu = F > C ? 1.0 - C / F : 0.0;
    const double tile = 512.0 * D;                           // K and V tile of one pair
    const double compulsory = rows_q * D * 2.0 * 2.0 + rows_q * 4.0 + (double)a->kv_heads * F;
    const double t_compute = listed * 4.0 * 128.0 * 128.0 * D / flops_rate;
    auto t_ms = [&](double miss) {
        const double t_mem = (compulsory + listed * tile * miss) / bw;
        return 1e3 * (t_compute > t_mem ? t_compute : t_mem);
    };
    const double rows = (double)a->heads * a->nQB;
    // the wave sort reads the counts and writes the order; the spectral stage
    // reads the lists twice per iteration (10 iterations), then sorts per head
    const double wave_cost = a->wave_ms >= 0.0 ? a->wave_ms : 1e3 * (rows * 8.0 / bw) + 0.01;
    const double spec_cost =
        a->spectral_ms >= 0.0 ? a->spectral_ms : 1e3 * (10.0 * 2.0 * 4.0 * listed / bw) + 0.01 * 32.0;
    r->kv_head_bytes = F;
    r->kv_cache_bytes = C;
    r->miss_fraction = mu;
    r->t_input_ms = t_ms(mu);
    r->t_wave_ms = t_ms(mu * (1.0 - 0.6889));
    r->t_spectral_ms = t_ms(mu * (1.0 - 0.8071));
    r->wave_cost_ms = wave_cost;
    r->spectral_cost_ms = spec_cost;
    const double net_wave = r->t_input_ms - r->t_wave_ms - wave_cost;
    const double net_spec = r->t_input_ms - r->t_spectral_ms - wave_cost - spec_cost;
    r->order = BSA_ORDER_INPUT;
    if (net_wave > 0.0 || net_spec > 0.0)
        r->order = net_spec > net_wave ? BSA_ORDER_SPECTRAL : BSA_ORDER_WAVE;
    return BSA_OK;
}

static bool score_sizes_ok(int32_t B, int32_t H, int32_t N, int32_t D) {
    return B >= 1 && H >= 1 && (int64_t)B * H <= 65535 && N >= 128 && (N % 128) == 0 &&
           N <= (1 << 24) && (int64_t)B * H * N < ((int64_t)1 << 31) && D >= 8 && D <= 256 &&
           (D % 8) == 0;
}

size_t bsa_block_scores_workspace_size(int32_t B, int32_t H, int32_t N, int32_t D) {
    if (!score_sizes_ok(B, H, N, D)) return 0;
    return bsa::block_scores_workspace_bytes((int64_t)B * H, N, D);
}

bsa_status bsa_block_scores(const void* q, const void* k, int32_t B, int32_t H, int32_t N,
                            int32_t D, const int32_t* q_map, const int32_t* kv_map, float scale,
                            bsa_score_mode mode, void* workspace, size_t workspace_bytes,
                            float* scores, void* stream) {
    if (!score_sizes_ok(B, H, N, D) || !scale_ok(scale)) return BSA_ERR_INVALID_ARG;
    if (mode != BSA_SCORE_MEAN_DOT && mode != BSA_SCORE_CENTROID_EXP) return BSA_ERR_INVALID_ARG;
    if (!q || !k || !scores || !workspace) return BSA_ERR_INVALID_ARG;
    if (workspace_bytes < bsa::block_scores_workspace_bytes((int64_t)B * H, N, D))
        return BSA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(scores, 4) || !aligned(workspace, 16) ||
        (q_map && !aligned(q_map, 4)) || (kv_map && !aligned(kv_map, 4)))
        return BSA_ERR_INVALID_ARG;
    int32_t* status = bsa::status_word_ptr();
    if (!status) return BSA_ERR_CUDA;
    cudaError_t e = bsa::launch_block_scores(q, k, B, H, N, D, q_map, kv_map, scale, (int32_t)mode,
                                             static_cast<float*>(workspace), scores, status,
                                             static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}

static bool spectral_sizes_ok(int64_t heads, int32_t nQB, int32_t nKB) {
    return heads >= 0 && heads <= 65535 && nQB >= 2 && nQB <= 8192 && nKB >= 1 && nKB <= 65536;
}

extern "C++" {
namespace bsa {
bool spectral_args_ok(int64_t heads, int32_t nQB, int32_t nKB, int32_t max_kv, int32_t iters) {
    return spectral_sizes_ok(heads, nQB, nKB) && max_kv >= 1 && max_kv <= nKB && iters >= 0 && iters <= 1000;
}
}  // namespace bsa
}

size_t bsa_spectral_order_workspace_size(int64_t heads, int32_t nQB, int32_t nKB) {
    if (!spectral_sizes_ok(heads, nQB, nKB)) return 0;
    return bsa::spectral_order_workspace_bytes(heads, nQB, nKB);
}

bsa_status bsa_spectral_order(const int32_t* kv_idx, const int32_t* kv_cnt, int32_t max_kv,
                              int64_t heads, int32_t nQB, int32_t nKB, int32_t iters,
                              const float* x0, void* workspace, size_t workspace_bytes,
                              float* x_out, float* angle, int32_t* order, void* stream) {
    if (!bsa::spectral_args_ok(heads, nQB, nKB, max_kv, iters)) return BSA_ERR_INVALID_ARG;
    if (heads == 0) return BSA_OK;
    if (!kv_idx || !kv_cnt || !x0 || !order || !workspace) return BSA_ERR_INVALID_ARG;
    if (workspace_bytes < bsa::spectral_order_workspace_bytes(heads, nQB, nKB))
        return BSA_ERR_INVALID_ARG;
    if (!aligned(kv_idx, 4) || !aligned(kv_cnt, 4) || !aligned(x0, 8) || !aligned(order, 4) ||
        !aligned(workspace, 8) || (x_out && !aligned(x_out, 8)) || (angle && !aligned(angle, 4)))
        return BSA_ERR_INVALID_ARG;
    int32_t* status = bsa::status_word_ptr();
    if (!status) return BSA_ERR_CUDA;
    cudaError_t e = bsa::launch_spectral_order(kv_idx, kv_cnt, max_kv, heads, nQB, nKB, iters, x0,
                                               static_cast<float*>(workspace), x_out, angle, order,
                                               status, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}

bsa_status bsa_sample_blocks(const float* scores, int64_t rows, int32_t nKB,
                             const int32_t* exact_idx, const int32_t* exact_cnt,
                             int32_t exact_stride, int32_t m, const double* u, int32_t* kv_idx,
                             int32_t* kv_cnt, float* log_w, int32_t max_kv, void* stream) {
    if (rows < 0 || rows > bsa::kSampleRowsPerBlock * bsa::kMaxGridX || nKB < 1 || nKB > 4096 ||
        exact_stride < 1 || m < 0 || max_kv < 1)
        return BSA_ERR_INVALID_ARG;
    if (rows == 0) return BSA_OK;
    if (!exact_idx || !exact_cnt || !u || !kv_idx || !kv_cnt || !log_w)
        return BSA_ERR_INVALID_ARG;  // scores may be NULL: the uniform sampler
    if ((scores && !aligned(scores, 4)) || !aligned(exact_idx, 4) || !aligned(exact_cnt, 4) || !aligned(u, 8) ||
        !aligned(kv_idx, 4) || !aligned(kv_cnt, 4) || !aligned(log_w, 4))
        return BSA_ERR_INVALID_ARG;
    int32_t* status = bsa::status_word_ptr();
    if (!status) return BSA_ERR_CUDA;
    cudaError_t e = bsa::launch_sample_blocks(scores, rows, nKB, exact_idx, exact_cnt, exact_stride,
                                              m, u, kv_idx, kv_cnt, log_w, max_kv, status,
                                              static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}

namespace {

// Host validation shared by bsa_forward, bsa_forward_masked and
// bsa_forward_packed.  nKB: key/value tiles a list entry may name (0: N/128).
bsa_status check_forward(const void* q, const void* k, const void* v, int32_t B, int32_t H,
                         int32_t H_kv, int32_t N, int32_t D, const int32_t* kv_idx,
                         const int32_t* kv_cnt, int32_t max_kv, const float* log_w,
                         const int32_t* q_map, const int32_t* kv_map, const int32_t* row_perm,
                         const void* o, const float* lse, float scale, int32_t nKB = 0) {
    if (D != 64 && D != 128) return BSA_ERR_UNSUPPORTED;
    if (!scale_ok(scale)) return BSA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || N < 128 || (N % 128) != 0 || N > (1 << 24)) return BSA_ERR_INVALID_ARG;
    if (H_kv < 1 || H_kv > H || H % H_kv != 0) return BSA_ERR_INVALID_ARG;
    const int64_t total_rows = (int64_t)B * H * N;
    if (total_rows >= ((int64_t)1 << 31) || (int64_t)B * H > 65535) return BSA_ERR_INVALID_ARG;
    if (nKB <= 0) nKB = N / 128;
    if (max_kv < 1 || max_kv > nKB) return BSA_ERR_INVALID_ARG;
    if (!q || !k || !v || !kv_idx || !kv_cnt || !o || !lse) return BSA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16))
        return BSA_ERR_INVALID_ARG;
    if (!aligned(kv_idx, 4) || !aligned(kv_cnt, 4) || !aligned(lse, 4)) return BSA_ERR_INVALID_ARG;
    if ((log_w && !aligned(log_w, 4)) || (row_perm && !aligned(row_perm, 4)))
        return BSA_ERR_INVALID_ARG;
    if ((q_map && !aligned(q_map, 16)) || (kv_map && !aligned(kv_map, 16)))
        return BSA_ERR_INVALID_ARG;
    return BSA_OK;
}

}  // namespace

bsa_status bsa_forward(const void* q, const void* k, const void* v, int32_t B, int32_t H, int32_t N,
                       int32_t D, const int32_t* kv_idx, const int32_t* kv_cnt, int32_t max_kv,
                       const float* log_w, const int32_t* q_map, const int32_t* kv_map,
                       const int32_t* row_perm, float scale, void* o, float* lse, void* stream) {
    const bsa_status c = check_forward(q, k, v, B, H, H, N, D, kv_idx, kv_cnt, max_kv, log_w, q_map,
                                       kv_map, row_perm, o, lse, scale);
    if (c != BSA_OK) return c;
    int32_t* status = bsa::status_word_ptr();
    if (!status) return BSA_ERR_CUDA;
    bsa::ForwardArgs a{q,      k,      v,     B,     H,      N,        D,     kv_idx, kv_cnt,
                       max_kv, log_w, q_map, kv_map, row_perm, scale, o,     lse,    nullptr, 0};
    return bsa::launch_forward(a, status, static_cast<cudaStream_t>(stream));
}

bsa_status bsa_forward_masked(const void* q, const void* k, const void* v, int32_t B, int32_t H,
                              int32_t H_kv, int32_t N, int32_t D, const int32_t* kv_idx,
                              const int32_t* kv_cnt, int32_t max_kv, const float* log_w,
                              const int32_t* q_map, const int32_t* kv_map,
                              const int32_t* row_perm, int32_t causal, int32_t n_valid,
                              int32_t window, int32_t sinks, float scale, void* o, float* lse,
                              void* stream) {
    const bsa_status c = check_forward(q, k, v, B, H, H_kv, N, D, kv_idx, kv_cnt, max_kv, log_w,
                                       q_map, kv_map, row_perm, o, lse, scale);
    if (c != BSA_OK) return c;
    if ((causal != 0 && causal != 1) || n_valid < 0 || n_valid > N || window < 0 || sinks < 0)
        return BSA_ERR_INVALID_ARG;
    int32_t* status = bsa::status_word_ptr();
    if (!status) return BSA_ERR_CUDA;
    bsa::ForwardArgs a{q,      k,      v,     B,     H,      N,        D,     kv_idx, kv_cnt,
                       max_kv, log_w, q_map, kv_map, row_perm, scale, o,     lse,    nullptr, 0};
    a.H_kv = H_kv;
    a.masked = causal != 0 || window > 0 || (n_valid > 0 && n_valid < N);
    a.causal = causal;
    a.n_valid = n_valid;
    a.window = window;
    a.sinks = sinks;
    return bsa::launch_forward(a, status, static_cast<cudaStream_t>(stream));
}

bsa_status bsa_forward_packed(const void* q, const void* k, const void* v, int32_t B, int32_t H,
                              int32_t H_kv, int32_t N, int32_t D, const int32_t* kv_idx,
                              const int32_t* kv_cnt, int32_t max_kv, const float* log_w,
                              const int32_t* q_map, const int32_t* kv_map, int32_t N_kv,
                              const uint8_t* quad_mask, const int32_t* row_perm, int32_t causal,
                              int32_t n_valid, int32_t window, int32_t sinks, float scale, void* o,
                              float* lse, void* stream) {
    if (kv_map == nullptr || N_kv < 128 || (N_kv % 128) != 0 || N_kv > (1 << 26))
        return BSA_ERR_INVALID_ARG;
    if (B >= 1 && H_kv >= 1 && (int64_t)B * H_kv * N_kv >= ((int64_t)1 << 40)) return BSA_ERR_INVALID_ARG;
    const bsa_status c = check_forward(q, k, v, B, H, H_kv, N, D, kv_idx, kv_cnt, max_kv, log_w,
                                       q_map, kv_map, row_perm, o, lse, scale, N_kv / 128);
    if (c != BSA_OK) return c;
    if ((causal != 0 && causal != 1) || n_valid < 0 || n_valid > N || window < 0 || sinks < 0)
        return BSA_ERR_INVALID_ARG;
    int32_t* status = bsa::status_word_ptr();
    if (!status) return BSA_ERR_CUDA;
    bsa::ForwardArgs a{q,      k,      v,     B,     H,      N,        D,     kv_idx, kv_cnt,
                       max_kv, log_w, q_map, kv_map, row_perm, scale, o,     lse,    nullptr, 0};
    a.H_kv = H_kv;
    a.masked = quad_mask != nullptr || causal != 0 || window > 0 || (n_valid > 0 && n_valid < N);
    a.causal = causal;
    a.n_valid = n_valid;
    a.window = window;
    a.sinks = sinks;
    a.n_kv = N_kv;
    a.quad_mask = quad_mask;
    return bsa::launch_forward(a, status, static_cast<cudaStream_t>(stream));
}

bsa_status bsa_gather0_sizes(int32_t img_h, int32_t img_w, int32_t n_text, int32_t groups,
                             int32_t* N, int32_t* N_kv, int32_t* max_kv) {
    bsa::Gather0Geom g;
    if (!bsa::gather0_geometry(img_h, img_w, n_text, groups, &g)) return BSA_ERR_INVALID_ARG;
    if (N) *N = g.N;
    if (N_kv) *N_kv = g.N_kv;
    if (max_kv) *max_kv = g.max_kv;
    return BSA_OK;
}

bsa_status bsa_gather0_layout(int32_t img_h, int32_t img_w, int32_t n_text, int32_t groups,
                              int64_t heads, int32_t* q_map, int32_t* kv_map, int32_t* kv_idx,
                              int32_t* kv_cnt, uint8_t* quad_mask, int32_t max_kv, void* stream) {
    bsa::Gather0Geom g;
    if (!bsa::gather0_geometry(img_h, img_w, n_text, groups, &g)) return BSA_ERR_INVALID_ARG;
    if (heads < 0 || heads > 65535 || max_kv < g.max_kv || max_kv > (1 << 20)) return BSA_ERR_INVALID_ARG;
    if (heads == 0) return BSA_OK;
    if (!q_map || !kv_map || !kv_idx || !kv_cnt || !quad_mask) return BSA_ERR_INVALID_ARG;
    if (!aligned(q_map, 16) || !aligned(kv_map, 16) || !aligned(kv_idx, 16) || !aligned(kv_cnt, 16))
        return BSA_ERR_INVALID_ARG;
    cudaError_t e = bsa::launch_gather0_layout(g, heads, q_map, kv_map, kv_idx, kv_cnt, quad_mask, max_kv,
                                               static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}

bsa_status bsa_forward_gather0(const void* q, const void* k, const void* v, int32_t B, int32_t H,
                               int32_t H_kv, int32_t D, int32_t img_h, int32_t img_w, int32_t n_text,
                               int32_t groups, const int32_t* kv_idx, const int32_t* kv_cnt,
                               const uint8_t* quad_mask, int32_t max_kv, const int32_t* row_perm,
                               float scale, void* o, float* lse, void* stream) {
    bsa::Gather0Geom g;
    if (!bsa::gather0_geometry(img_h, img_w, n_text, groups, &g)) return BSA_ERR_INVALID_ARG;
    if (B >= 1 && H_kv >= 1 && (int64_t)B * H_kv * g.N_kv >= ((int64_t)1 << 40)) return BSA_ERR_INVALID_ARG;
    const bsa_status c = check_forward(q, k, v, B, H, H_kv, g.N, D, kv_idx, kv_cnt, max_kv, nullptr,
                                       nullptr, nullptr, row_perm, o, lse, scale, g.N_kv / 128);
    if (c != BSA_OK) return c;
    int32_t* status = bsa::status_word_ptr();
    if (!status) return BSA_ERR_CUDA;
    bsa::ForwardArgs a{q,      k,       v,       B,        H,     g.N, D,   kv_idx, kv_cnt,
                       max_kv, nullptr, nullptr, nullptr, row_perm, scale, o, lse, nullptr, 0};
    a.H_kv = H_kv;
    a.masked = true;
    a.n_kv = g.N_kv;
    a.quad_mask = quad_mask;
    a.gather0 = &g;
    return bsa::launch_forward(a, status, static_cast<cudaStream_t>(stream));
}

bsa_status bsa_forward_scatter(const void* q, const void* k, const void* v, int32_t B, int32_t H,
                               int32_t H_kv, int32_t N, int32_t D, int32_t R, const int32_t* kv_idx,
                               const int32_t* kv_cnt, int32_t max_kv, const float* log_w,
                               const int32_t* row_perm, float scale, void* o, float* lse, void* stream) {
    if (R < 1 || N < 128 || (N % R) != 0 || ((N / R) % 128) != 0) return BSA_ERR_INVALID_ARG;
    const bsa_status c = check_forward(q, k, v, B, H, H_kv, N, D, kv_idx, kv_cnt, max_kv, log_w,
                                       nullptr, nullptr, row_perm, o, lse, scale);
    if (c != BSA_OK) return c;
    int32_t* status = bsa::status_word_ptr();
    if (!status) return BSA_ERR_CUDA;
    bsa::ForwardArgs a{q,      k,     v,       B,       H,        N,     D, kv_idx, kv_cnt,
                       max_kv, log_w, nullptr, nullptr, row_perm, scale, o, lse,    nullptr, 0};
    a.H_kv = H_kv;
    a.scatter_R = R;
    return bsa::launch_forward(a, status, static_cast<cudaStream_t>(stream));
}

bsa_status bsa_forward_crm(const void* q, const void* k, const void* v, int32_t B, int32_t H,
                           int32_t N, int32_t D, const uint32_t* crm, int32_t crm_words,
                           const int32_t* q_map, const int32_t* kv_map, const int32_t* row_perm,
                           float scale, void* o, float* lse, void* stream) {
    if (D != 64 && D != 128) return BSA_ERR_UNSUPPORTED;
    if (!scale_ok(scale)) return BSA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || N < 128 || (N % 128) != 0 || N > (1 << 24)) return BSA_ERR_INVALID_ARG;
    const int64_t total_rows = (int64_t)B * H * N;
    if (total_rows >= ((int64_t)1 << 31) || (int64_t)B * H > 65535) return BSA_ERR_INVALID_ARG;
    const int32_t nKB = N / 128;
    if (crm_words < (nKB + 31) / 32 || crm_words > (1 << 20)) return BSA_ERR_INVALID_ARG;
    if (!q || !k || !v || !crm || !o || !lse) return BSA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
        !aligned(crm, 4) || !aligned(lse, 4) || (row_perm && !aligned(row_perm, 4)) ||
        (q_map && !aligned(q_map, 16)) || (kv_map && !aligned(kv_map, 16)))
        return BSA_ERR_INVALID_ARG;
    int32_t* status = bsa::status_word_ptr();
    if (!status) return BSA_ERR_CUDA;
    bsa::ForwardArgs a{q,   k,      v,     B,     H,      N,        D,     nullptr, nullptr,
                       nKB, nullptr, q_map, kv_map, row_perm, scale, o,     lse,     crm, crm_words};
    return bsa::launch_forward(a, status, static_cast<cudaStream_t>(stream));
}

bsa_status bsa_build_crm(bsa_idx_mode mode, const void* src, int64_t rows, int32_t nKB, float p,
                         uint32_t* words, int32_t crm_words, void* stream) {
    if (mode != BSA_IDX_MASK_U8 && mode != BSA_IDX_THRESHOLD_F32) return BSA_ERR_INVALID_ARG;
    if (rows < 0 || rows > bsa::kListRowsPerBlock * bsa::kMaxGridX || nKB < 1 || nKB > 65536 ||
        crm_words < (nKB + 31) / 32 || crm_words > (1 << 20))
        return BSA_ERR_INVALID_ARG;
    if (rows == 0) return BSA_OK;
    if (!src || !words || !aligned(words, 4) || (mode != BSA_IDX_MASK_U8 && !aligned(src, 4)))
        return BSA_ERR_INVALID_ARG;
    cudaError_t e = bsa::launch_crm_rows(mode, src, rows, nKB, p, words, crm_words,
                                         static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}

bsa_status bsa_upscale_threshold(const float* T_base, int64_t heads, int32_t Ub, int32_t Vb,
                                 int32_t Ut, int32_t Vt, float* T_target, void* stream) {
    if (heads < 0 || heads > bsa::kMaxGridYZ || Ub < 1 || Vb < 1 || Ut < 1 || Vt < 1 || Ub > 65536 ||
        Vb > 65536 || Ut > bsa::kMaxGridYZ || Vt > 65536)
        return BSA_ERR_INVALID_ARG;
    if (heads == 0) return BSA_OK;
    if (!T_base || !T_target || !aligned(T_base, 4) || !aligned(T_target, 4)) return BSA_ERR_INVALID_ARG;
    cudaError_t e = bsa::launch_upscale_threshold(T_base, heads, Ub, Vb, Ut, Vt, T_target,
                                                  static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}

bsa_status bsa_gather_rows(const void* src, const int32_t* map, int64_t heads, int32_t N,
                           int32_t D, void* dst, void* stream) {
    if (D != 64 && D != 128) return BSA_ERR_UNSUPPORTED;
    if (heads < 0 || heads > 65535 || N < 1 || N > (1 << 24)) return BSA_ERR_INVALID_ARG;
    if (heads * (int64_t)N >= ((int64_t)1 << 31)) return BSA_ERR_INVALID_ARG;
    if (heads == 0) return BSA_OK;
    if (!src || !map || !dst || !aligned(src, 16) || !aligned(dst, 16) || !aligned(map, 4))
        return BSA_ERR_INVALID_ARG;
    const uintptr_t s0 = reinterpret_cast<uintptr_t>(src), d0 = reinterpret_cast<uintptr_t>(dst);
    const uintptr_t bytes = (uintptr_t)(heads * (int64_t)N) * (uintptr_t)D * 2u;
    if (s0 < d0 + bytes && d0 < s0 + bytes) return BSA_ERR_INVALID_ARG;  // overlapping buffers
    int32_t* status = bsa::status_word_ptr();
    if (!status) return BSA_ERR_CUDA;
    cudaError_t e = bsa::launch_gather_rows(src, map, heads, N, D, dst, status,
                                            static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}

bsa_status bsa_set_forward_options(const bsa_forward_options* o) {
    if (o == nullptr) {
        bsa::forward_options() = bsa_forward_options{BSA_SCHEDULE_AUTO, 0};
        return BSA_OK;
    }
    if ((o->schedule != BSA_SCHEDULE_AUTO && o->schedule != BSA_SCHEDULE_PER_ROW &&
         o->schedule != BSA_SCHEDULE_PER_ITEM) ||
        (o->exp2_fma != 0 && o->exp2_fma != 2))
        return BSA_ERR_INVALID_ARG;
    bsa::forward_options() = *o;
    return BSA_OK;
}

bsa_status bsa_device_status(void* stream, int32_t* first_error) {
    if (!first_error) return BSA_ERR_INVALID_ARG;
    int32_t* status = bsa::status_word_ptr();
    if (!status) return BSA_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    if (cudaStreamSynchronize(st) != cudaSuccess) return BSA_ERR_CUDA;
    if (cudaMemcpyAsync(&v, status, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return BSA_ERR_CUDA;
    if (cudaMemsetAsync(status, 0, sizeof(v), st) != cudaSuccess) return BSA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return BSA_ERR_CUDA;
    *first_error = v;
    return BSA_OK;
}

int32_t bsa_resident_ctas(int32_t D) { return bsa::forward_resident_ctas(D); }

}  // extern "C"
