// Internal declarations shared by the translation units of libbsa.so.
// Host-side launchers; each takes the device address of the status word.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "bsa.h"

namespace bsa {

constexpr int kBlock = 128;  // query / key block edge

// Launch shapes of the list kernels, which bound the rows one call may pass:
// the index, top-k and CRM launches give each warp of an 8-warp block one
// row, the sampler one thread of a 64-thread block, and grid.x is at most
// 2^31 - 1 (grid.y and grid.z at most 65535).
constexpr int kListRowsPerBlock = 8;
constexpr int kSampleRowsPerBlock = 64;
constexpr int64_t kMaxGridX = 2147483647;
constexpr int64_t kMaxGridYZ = 65535;

// Status word helpers (defined in bsa_api.cu).
int32_t* status_word_ptr();  // device address of the current device's status word

// bsa_index.cu
cudaError_t launch_index_predicate(bsa_idx_mode mode, const void* src, int64_t rows, int32_t nKB,
                                   float p, int32_t* kv_idx, int32_t* kv_cnt, int32_t max_kv,
                                   int32_t* status, cudaStream_t stream);
cudaError_t launch_index_topk(const float* scores, int64_t rows, int32_t nKB,
                              const int32_t* k_per_row, int32_t k_const, int32_t* kv_idx,
                              int32_t* kv_cnt, int32_t max_kv, int32_t* status,
                              cudaStream_t stream);
cudaError_t launch_crm_rows(bsa_idx_mode mode, const void* src, int64_t rows, int32_t nKB, float p,
                            uint32_t* words, int32_t n_words, cudaStream_t stream);
// dst[bh][p] = src[bh][map[bh][p]] for bf16 rows of D elements (bsa_gather.cu).
cudaError_t launch_gather_rows(const void* src, const int32_t* map, int64_t heads, int32_t N,
                               int32_t D, void* dst, int32_t* status, cudaStream_t stream);
// The INTRA Gather 0 layer's sizes (host; false: arguments out of range) and
// its maps, lists and quadrant masks (bsa_gather.cu).
struct Gather0Geom {
    int32_t img_h, img_w, n_text, groups;
    int32_t N, N_kv, max_kv;
};
bool gather0_geometry(int32_t img_h, int32_t img_w, int32_t n_text, int32_t groups, Gather0Geom* out);
cudaError_t launch_gather0_layout(const Gather0Geom& geo, int64_t heads, int32_t* q_map, int32_t* kv_map,
                                  int32_t* kv_idx, int32_t* kv_cnt, uint8_t* quad_mask, int32_t max_kv,
                                  cudaStream_t stream);
cudaError_t launch_upscale_threshold(const float* T, int64_t heads, int32_t Ub, int32_t Vb,
                                     int32_t Ut, int32_t Vt, float* out, cudaStream_t stream);
cudaError_t launch_reorder_rows(const int32_t* kv_cnt, const int32_t* order_in, int64_t heads,
                                int32_t nQB, int32_t wave, int32_t* row_perm, int32_t* status,
                                cudaStream_t stream);
cudaError_t launch_sample_blocks(const float* scores, int64_t rows, int32_t nKB,
                                 const int32_t* exact_idx, const int32_t* exact_cnt,
                                 int32_t exact_stride, int32_t m, const double* u,
                                 int32_t* kv_idx, int32_t* kv_cnt, float* log_w, int32_t max_kv,
                                 int32_t* status, cudaStream_t stream);

// bsa_scores.cu
size_t block_scores_workspace_bytes(int64_t BH, int32_t N, int32_t D);
cudaError_t launch_block_scores(const void* q, const void* k, int32_t B, int32_t H, int32_t N,
                                int32_t D, const int32_t* q_map, const int32_t* kv_map, float scale,
                                int32_t mode, float* workspace, float* scores, int32_t* status,
                                cudaStream_t stream);

// bsa_order.cu
size_t spectral_order_workspace_bytes(int64_t heads, int32_t nQB, int32_t nKB);
// Loads the spectral-order kernels on the current device (no launch).
cudaError_t load_spectral_kernels();
// Sizes and counts every spectral-order entry point accepts (bsa_api.cu).
bool spectral_args_ok(int64_t heads, int32_t nQB, int32_t nKB, int32_t max_kv, int32_t iters);
cudaError_t launch_spectral_order(const int32_t* kv_idx, const int32_t* kv_cnt, int32_t max_kv,
                                  int64_t heads, int32_t nQB, int32_t nKB, int32_t iters,
                                  const float* x0, float* workspace, float* x_out, float* angle,
                                  int32_t* order, int32_t* status, cudaStream_t stream);

// bsa_attn.cu
struct ForwardArgs {
    const void* q;
    const void* k;
    const void* v;
    int32_t B, H, N, D;
    const int32_t* kv_idx;
    const int32_t* kv_cnt;
    int32_t max_kv;
    const float* log_w;
    const int32_t* q_map;
    const int32_t* kv_map;
    const int32_t* row_perm;
    float scale;
    void* o;
    float* lse;
    const uint32_t* crm;  // non-NULL: CRM rows instead of kv_idx / kv_cnt
    int32_t crm_words;
    int32_t H_kv = 0;     // key/value heads per batch entry (0: H)
    bool masked = false;  // token mask below applies
    int32_t causal = 0, n_valid = 0, window = 0, sinks = 0;
    int32_t n_kv = 0;                     // kv_map entries per key/value head (0: N)
    const uint8_t* quad_mask = nullptr;   // [rows, max_kv] 32-row quadrant visibility
    const Gather0Geom* gather0 = nullptr;  // non-NULL: Gather 0 tiles by geometry
    int32_t scatter_R = 0;                 // > 0: Scatter layer tiles by geometry (R groups)
};
// Returns BSA_OK, BSA_ERR_CUDA (launch / descriptor failure) or BSA_ERR_UNSUPPORTED.
bsa_status launch_forward(const ForwardArgs& a, int32_t* status, cudaStream_t stream);
// The calling host thread's forward options (bsa_set_forward_options).
bsa_forward_options& forward_options();
int32_t forward_resident_ctas(int32_t D);

}  // namespace bsa
