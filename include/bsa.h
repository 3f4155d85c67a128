/*
 * bsa.h - C ABI of libbsa.so, GB300-native (sm_103a) forward block-sparse
 * attention over 128 x 128 blocks.
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 *  - The caller owns every buffer.  Array arguments are DEVICE pointers
 *    unless stated otherwise; the library allocates no device memory.
 *  - All launches are asynchronous on `stream` (a cudaStream_t passed as
 *    void*; NULL is the legacy default stream).  Results are ready when the
 *    stream is synchronised.
 *  - Errors the host can see (null or misaligned pointers, bad sizes, an
 *    unsupported head dimension) are returned immediately and nothing is
 *    launched.  Conditions only the device can see (an index list longer
 *    than max_kv, an index or map entry out of range, a wait that timed out)
 *    are recorded in a per-device status word: the first such code wins and
 *    bsa_device_status() reads and clears it.  No kernel traps.
 *  - Tensors are row-major and contiguous.  "rows" of an index list are the
 *    (batch, head, query block) triples in that nesting order:
 *    row = (b * H + h) * nQB + qb.
 *  - Block edge is 128 tokens for queries and keys (nQB = nKB = N / 128).
 *  - A pointer carries no length: every array must hold at least the
 *    entries its layout below gives (the library reads and writes exactly
 *    those), on the device that is current when the call is made.  The
 *    Python binding checks both before it calls.
 */
#ifndef BSA_H
#define BSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    BSA_OK = 0,
    BSA_ERR_INVALID_ARG = 1, /* host-detected: bad pointer, size or alignment   */
    BSA_ERR_UNSUPPORTED = 2, /* host-detected: e.g. D not in {64, 128}         */
    BSA_ERR_OVERFLOW = 3,    /* device: a list longer than max_kv (truncated)  */
    BSA_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed               */
    BSA_ERR_TIMEOUT = 5,     /* device: a bounded wait gave up                  */
    BSA_ERR_BOUNDS = 6       /* device: an index/map/perm entry out of range    */
} bsa_status;

typedef enum {
    BSA_SCORE_MEAN_DOT = 0,     /* mean(Q_u) . mean(K_v) * scale                     */
    BSA_SCORE_CENTROID_EXP = 1  /* exp(mean(Q_u) . mean(K_v) * scale): centroid score */
} bsa_score_mode;

typedef enum {
    BSA_IDX_MASK_U8 = 0,       /* src: uint8 [rows, nKB], keep entries != 0             */
    BSA_IDX_THRESHOLD_F32 = 1, /* src: fp32 threshold map [rows, nKB], keep T <= p     */
    BSA_IDX_TOPK_F32 = 2       /* src: fp32 block scores [rows, nKB], keep the k largest */
} bsa_idx_mode;

/*
 * bsa_build_index - compact a mask / threshold map / score matrix into
 * per-row KV-block index lists.
 *
 * Defined by: ScalingAttention, section 5.2 eq. (2) (the mask M_p = I(T <= p)
 * instantiated from a threshold map) and section 7.2 (index-based row
 * format); WaveAlign, "B. Sparse Attention for Long-Video Generation" (one
 * mask row per query block, one kept entry per executed block product);
 * MC-Sparse, "The MC-Sparse Architecture" and InstaGen section 3.2.1 (keep
 * the top-k blocks by score).
 *
 *  mode      which predicate selects a block (see bsa_idx_mode).
 *  src       device, [rows, nKB] uint8 (MASK) or fp32 (THRESHOLD, TOPK).
 *  rows      number of (b, h, qb) rows, 0 .. 8 * (2^31 - 1).
 *  nKB       KV blocks per row, 1 .. 65536.
 *  p         THRESHOLD: keep src <= p, compared in fp32 (inclusive).
 *  k_per_row TOPK: device int32 [rows] or NULL to use k_const for every row.
 *  k_const   TOPK: k when k_per_row is NULL.  k is clamped to [0, nKB].
 *            Ties in score go to the lower block index; -0.0 equals +0.0.
 *            Scores must not be NaN.
 *  kv_idx    device int32 [rows, max_kv] out: the kept blocks of each row in
 *            ascending block order, unused tail entries set to -1.
 *  kv_cnt    device int32 [rows] out: number of valid entries.
 *  max_kv    list capacity, 1 .. nKB.  A row with more kept blocks keeps its
 *            first max_kv (ascending) and raises BSA_ERR_OVERFLOW on the
 *            device status word.
 *  Pointers must be 4-byte aligned (src of MASK: any alignment).
 */
bsa_status bsa_build_index(bsa_idx_mode mode, const void* src, int64_t rows, int32_t nKB,
                           float p, const int32_t* k_per_row, int32_t k_const,
                           int32_t* kv_idx, int32_t* kv_cnt, int32_t max_kv, void* stream);

/*
 * bsa_block_scores - per-head score of every (query block, KV block) pair
 * from the blocks' mean vectors, the input of top-k selection and of
 * importance sampling.
 *
 * Defined by: MC-Sparse, "The MC-Sparse Architecture" (block-sparse attention
 * scores blocks by mean-pooled similarity); InstaGen, section 3.3 and
 * Algorithm 1 step 2 (centroid score s_gc = exp(q_g . k_c / sqrt d) of a
 * query group and a key cluster).  A group / cluster is a 128-token block of
 * the gathered order (q_map / kv_map, identity when NULL).
 *
 *  q, k      device bf16 [B, H, N, D], 16-byte aligned; N a multiple of 128,
 *            D 8 .. 256 (x8).
 *  q_map, kv_map  device int32 [B*H, N] or NULL (as in bsa_forward).
 *  scale     <= 0 selects 1/sqrt(D); a NaN or infinite scale is rejected
 *            (BSA_ERR_INVALID_ARG).
 *  mode      BSA_SCORE_MEAN_DOT or BSA_SCORE_CENTROID_EXP.
 *  workspace device scratch of at least bsa_block_scores_workspace_size()
 *            bytes (the fp32 block means), 16-byte aligned.
 *  scores    device fp32 [B*H*nQB, nKB] out.
 *  fp32 means and dot products; a map entry outside [0, N) is read as row 0
 *  and raises BSA_ERR_BOUNDS.
 */
bsa_status bsa_block_scores(const void* q, const void* k, int32_t B, int32_t H, int32_t N,
                            int32_t D, const int32_t* q_map, const int32_t* kv_map, float scale,
                            bsa_score_mode mode, void* workspace, size_t workspace_bytes,
                            float* scores, void* stream);

/* Bytes of workspace bsa_block_scores needs (0 for sizes it rejects). */
size_t bsa_block_scores_workspace_size(int32_t B, int32_t H, int32_t N, int32_t D);

/*
 * bsa_reorder_rows - query-row execution order, NNZ-guided within waves.
 *
 * Defined by: WaveAlign, section IV-B (waves of at most W rows per head) and
 * section IV-D "NNZ-Guided Intra-Wave Temporal Alignment" (consecutive
 * buckets of at most W rows, each sorted by descending KV-block count).
 * Ties keep their input order.  Buckets restart at every head.
 *
 *  kv_cnt    device int32 [heads, nQB]: KV-block count of each query block.
 *  order_in  device int32 [heads, nQB] input order (each row a permutation
 *            of 0..nQB-1, e.g. a spatial ordering), or NULL for identity.
 *  heads     B * H, >= 0.
 *  nQB       query blocks per head, 1 .. 65536.
 *  wave      W, 1 .. 8192: typically bsa_resident_ctas(D).
 *  row_perm  device int32 [heads, nQB] out: row_perm[h][slot] = query block
 *            executed in that slot; pass it to bsa_forward.
 *  An order_in entry outside [0, nQB) raises BSA_ERR_BOUNDS on the device.
 */
bsa_status bsa_reorder_rows(const int32_t* kv_cnt, const int32_t* order_in, int64_t heads,
                            int32_t nQB, int32_t wave, int32_t* row_perm, void* stream);

/*
 * bsa_reorder_guard - whether reordering query rows pays for one forward
 * call, and with which stages (host-side arithmetic; launches nothing).
 *
 * Defined by: WaveAlign, "A. Design Rationale" and "E. Runtime
 * Coordination" of its design section (an adaptive guard skips reordering
 * when its estimated latency reduction does not exceed its overhead); "C.
 * Why Access Is Irregular: Two Root Causes" (reuse is lost when a wave's K/V
 * working set overflows L2); "D. L2 Cache Locality and HBM Traffic" of its
 * evaluation (HBM reads fall by 68.89 %-83.67 % with the intra-wave NNZ sort
 * alone and by 80.71 %-92.11 % with both stages); "F. Other Factors"
 * (reordering skipped at short sequences and low densities).
 *
 * The pages give no formula; this guard estimates the forward's latency as
 * max(compute, DRAM traffic) for three orders and picks the one whose
 * saving beats its cost by the most:
 *   F   = nKB * 128 * D * 4 bytes, one head's K and V;
 *   C   = l2_bytes / 2, the L2 share K/V keep (the rest streams Q, O and
 *         the next head's first blocks; heads run one after another);
 *   mu  = max(0, 1 - C / F), the fraction of K/V tile reads that miss L2 in
 *         the input order (a head's blocks compete for C at random);
 *   DRAM(order) = Q + O + LSE + kv_heads * F + listed_blocks * 512 * D * mu_order
 *         with mu_input = mu, mu_wave = mu * (1 - 0.6889),
 *         mu_spectral = mu * (1 - 0.8071) (the smallest cuts the page reports);
 *   t(order) = max(listed_blocks * 4 * 128^2 * D / tensor rate, DRAM / HBM rate).
 * The wave sort is chosen when t(input) - t(wave) > its cost, the spectral
 * stage (plus wave sort) when its saving over the wave sort also beats its
 * extra cost.  When one head's K/V fits its L2 share (mu = 0) nothing can be
 * saved and the input order is kept.
 *
 *  a->heads        B*H query heads, >= 1.   a->kv_heads  B*H_kv, 1 .. heads.
 *  a->nQB, a->nKB  query / key blocks per head, >= 1.   a->D  head dimension, >= 1.
 *  a->listed_blocks  listed (query block, key block) pairs of the call, >= 0.
 *  a->l2_bytes     L2 capacity in bytes; 0: the current device's.
 *  a->tensor_tflops  effective block-pair rate of the forward (TFLOP/s);
 *                  0: 1500.   a->hbm_gbs  DRAM bandwidth (GB/s); 0: 6800.
 *  a->wave_ms, a->spectral_ms  measured cost of bsa_reorder_rows and of
 *                  bsa_spectral_order for this call; a negative value asks
 *                  for the guard's estimate (bytes moved at the HBM rate plus
 *                  10 us per launch; the spectral stage 10 iterations).
 *  r               host out: the decision and the estimates behind it.
 * Returns BSA_ERR_INVALID_ARG for null pointers or sizes out of range,
 * BSA_ERR_CUDA if l2_bytes is 0 and no device answers.
 */
typedef struct {
    int64_t heads;
    int64_t kv_heads;
    int32_t nQB;
    int32_t nKB;
    int32_t D;
    int64_t listed_blocks;
    double l2_bytes;
    double tensor_tflops;
    double hbm_gbs;
    double wave_ms;
    double spectral_ms;
} bsa_guard_args;

typedef enum {
    BSA_ORDER_INPUT = 0,    /* keep the input order (reordering skipped)          */
    BSA_ORDER_WAVE = 1,     /* NNZ-guided intra-wave sort (bsa_reorder_rows)      */
    BSA_ORDER_SPECTRAL = 2  /* spectral order, then the wave sort                 */
} bsa_row_order;

typedef struct {
    bsa_row_order order;
    double kv_head_bytes;   /* F */
    double kv_cache_bytes;  /* C */
    double miss_fraction;   /* mu */
    double t_input_ms, t_wave_ms, t_spectral_ms;  /* estimated forward times */
    double wave_cost_ms, spectral_cost_ms;        /* costs used */
} bsa_guard_result;

bsa_status bsa_reorder_guard(const bsa_guard_args* a, bsa_guard_result* r);

/*
 * bsa_spectral_order - spatial row order from the rank-2 embedding of each
 * head's centered block mask (the first stage of row reordering).
 *
 * Defined by: WaveAlign, section IV-C "SVD-Based Global Spatial Ordering"
 * (polar spectral ordering; matrix-free centered subspace iteration with
 * the rank-1 centering correction, 5-15 iterations suffice because the
 * angular sort ignores in-plane rotations and sign flips).
 *
 * Per head the mask A (row = query block, column = KV block listed in that
 * row) is centered by its mean row mu.  Starting from x0 (orthonormalised),
 * `iters` times: Z = A^T X - mu (1^T X); X = Gram-Schmidt(A Z - 1 (mu^T Z)).
 * Rows are then sorted by atan2(X[r][1], X[r][0]) ascending, ties to the lower
 * query block.  fp32, one warp per query block across the whole GPU; the
 * sums are fp32 atomics, so the last bits of the embedding (and the order of
 * rows whose angles nearly coincide) may differ between runs.  Pass the
 * result as order_in to bsa_reorder_rows.
 *
 *  kv_idx, kv_cnt, max_kv  the index lists of B*H*nQB rows (as bsa_forward).
 *  heads     B * H.        nQB  query blocks per head, 2 .. 8192.
 *  nKB       KV blocks per head, 1 .. 65536.   iters  0 .. 1000.
 *  x0        device fp32 [heads, nQB, 2]: starting vectors (e.g. random).
 *  workspace device scratch of at least
 *            bsa_spectral_order_workspace_size(heads, nQB, nKB) bytes,
 *            8-byte aligned; its contents on entry do not matter.  Calls
 *            that share a workspace must not overlap on the GPU.
 *  x_out     device fp32 [heads, nQB, 2] or NULL: the final embedding.
 *  angle     device fp32 [heads, nQB] or NULL: the polar angles.
 *  order     device int32 [heads, nQB] out: order[h][s] = query block.
 *  A list entry outside [0, nKB) is ignored and raises BSA_ERR_BOUNDS.
 */
bsa_status bsa_spectral_order(const int32_t* kv_idx, const int32_t* kv_cnt, int32_t max_kv,
                              int64_t heads, int32_t nQB, int32_t nKB, int32_t iters,
                              const float* x0, void* workspace, size_t workspace_bytes,
                              float* x_out, float* angle, int32_t* order, void* stream);

/* Bytes of workspace bsa_spectral_order needs (0 for sizes it rejects). */
size_t bsa_spectral_order_workspace_size(int64_t heads, int32_t nQB, int32_t nKB);

/* Size of the fixed scratch array behind bsa_spectral_order_noalloc. */
#define BSA_SPECTRAL_NOALLOC_SCRATCH_BYTES (4u << 20)

/*
 * bsa_spectral_order_noalloc - bsa_spectral_order for callers that cannot
 * allocate device memory.  The pages have no counterpart; it exists for
 * programs that must not allocate while they run (for example a serving
 * loop or host framework that owns the whole device memory pool, where an
 * allocation could fail or stall in the middle of a step) or that cannot
 * pass a workspace buffer down to this call.
 *
 * Same arguments and results as bsa_spectral_order, without the workspace:
 * its scratch is a fixed array of BSA_SPECTRAL_NOALLOC_SCRATCH_BYTES inside
 * the library, present on every device that loads it until the process
 * exits.  Nothing in this call allocates memory.
 *  - Sizes whose workspace (bsa_spectral_order_workspace_size) exceeds
 *    BSA_SPECTRAL_NOALLOC_SCRATCH_BYTES are rejected with
 *    BSA_ERR_UNSUPPORTED before anything is launched.
 *  - The first call on each device sets that device up: it looks up the
 *    array's device address (cudaGetSymbolAddress) and the status word, and
 *    loads the spectral-order kernels.  With CUDA's lazy module loading (the
 *    default) that set-up is when the array and the kernels take their
 *    device memory.  Make one call per device, before any stream capture and
 *    before the phase in which nothing may allocate; a call with heads = 0
 *    (every pointer may then be NULL) does the set-up and nothing else.
 *  - Arguments are checked as bsa_spectral_order checks them, first.
 *  - All calls share the array.  Calls whose work overlaps on the GPU (other
 *    streams, other host threads) race on it: serialise them.  Each call
 *    clears what must start at zero, so leftovers of an earlier call do not
 *    matter.
 */
bsa_status bsa_spectral_order_noalloc(const int32_t* kv_idx, const int32_t* kv_cnt,
                                      int32_t max_kv, int64_t heads, int32_t nQB, int32_t nKB,
                                      int32_t iters, const float* x0, float* x_out, float* angle,
                                      int32_t* order, void* stream);

/*
 * bsa_sample_blocks - exact set plus an importance-weighted PPSWOR sample of
 * the remaining KV blocks, with Horvitz-Thompson log-weights.
 *
 * Defined by: InstaGen, section 3.2.1 eq. (4) (pi_j = min(1, lambda s_j),
 * sum over the residual = m, by capping at 1 and renormalising), eq. (5)
 * (Horvitz-Thompson), the promotion of blocks whose pi reaches 1, systematic
 * PPS sampling, and Algorithm 1 step 13 (w = 1 / pi).
 *
 * Per row, the residual is every block not in the exact list.  Blocks with
 * pi = 1 are promoted (kept, weight 1).  The other m - |promoted| blocks are
 * drawn by systematic PPS in ascending block order with the row's uniform
 * u: block j is drawn when a point u + i falls in [C_{j-1}, C_j), C the
 * running sum of pi.  lambda, pi and C are fp32 (u is rounded to fp32),
 * summed in ascending block order with IEEE round-to-nearest and no fused
 * multiply-adds, so the drawn set is reproducible.
 *
 *  scores       device fp32 [rows, nKB], every entry > 0; or NULL for the
 *               uniform sampler (InstaGen Algorithm 1 steps 6-8): every
 *               residual block gets pi = m / |residual|.
 *  exact_idx    device int32 [rows, exact_stride]: exact blocks, ascending.
 *  exact_cnt    device int32 [rows].
 *  exact_stride row stride of exact_idx, >= 1.
 *  m            blocks to draw per row (sampling budget), >= 0.
 *  u            device fp64 [rows], each in [0, 1).
 *  kv_idx       device int32 [rows, max_kv] out: exact, promoted and drawn
 *               blocks merged in ascending order (tail -1).
 *  kv_cnt       device int32 [rows] out.
 *  log_w        device fp32 [rows, max_kv] out: 0 for exact and promoted
 *               entries, -log(pi_j) (fp32 log) for drawn ones (tail 0).
 *  max_kv       capacity; a longer merged list is truncated and raises
 *               BSA_ERR_OVERFLOW.
 *  Outputs must not alias inputs.  nKB <= 4096; rows 0 .. 64 * (2^31 - 1).
 */
bsa_status bsa_sample_blocks(const float* scores, int64_t rows, int32_t nKB,
                             const int32_t* exact_idx, const int32_t* exact_cnt,
                             int32_t exact_stride, int32_t m, const double* u,
                             int32_t* kv_idx, int32_t* kv_cnt, float* log_w, int32_t max_kv,
                             void* stream);

/*
 * bsa_forward - block-sparse attention forward, O and LSE.
 *
 * Defined by: InstaGen, section 3.1 eqs. (1)-(3) (scaled dot-product
 * attention) and Algorithm 1 step 14 (softmax over the kept keys of
 * l_ij + log w_j, w the block's Horvitz-Thompson weight); INTRA,
 * "CQS-Aware Token-Sparse FlashAttention Kernel" (query and key tokens
 * reached through index maps, packed into dense tiles, outputs scattered
 * back through the query map); WaveAlign, section V (rows run in a
 * permuted order, outputs land in their original rows).
 *
 * For head bh = b*H + h, gathered position p holds query token q_map[bh][p]
 * and key/value token kv_map[bh][p] (p itself when the map is NULL).  Query
 * block qb = p / 128 attends to the keys at gathered positions
 * 128*kb .. 128*kb+127 for every kb in its list, each block with log-weight
 * lw = log_w[row][e] (0 when log_w is NULL):
 *     s_ij  = (q_i . k_j) * scale + lw
 *     LSE_i = ln sum_j exp(s_ij)           (natural log, of the weighted sum)
 *     O_i   = sum_j exp(s_ij - LSE_i) v_j
 * written to O[bh][i] and LSE[bh][i] with i = q_map[bh][p].  An empty list
 * gives O_i = 0 and LSE_i = -inf.  Execution slot s of head bh computes
 * query block row_perm[bh][s] (s when NULL); the order changes only the
 * schedule, never the result.
 *
 *  q, k, v   device bf16 [B, H, N, D] contiguous, 16-byte aligned.
 *  B, H, N   N a multiple of 128, 128 .. 2^24; B*H*N < 2^31.
 *  D         head dimension, 64 or 128.
 *  kv_idx    device int32 [B*H*nQB, max_kv]; kv_cnt device int32 [B*H*nQB].
 *            Entries must be distinct within a row.  An entry outside
 *            [0, nKB) is skipped and raises BSA_ERR_BOUNDS; a count above
 *            max_kv is clamped and raises BSA_ERR_OVERFLOW.
 *  max_kv    list capacity, 1 .. nKB.
 *  log_w     device fp32 [B*H*nQB, max_kv] or NULL.
 *  q_map, kv_map  device int32 [B*H, N] or NULL; each row must be a
 *            permutation of 0..N-1 (a q_map entry outside [0, N) skips that
 *            output row and raises BSA_ERR_BOUNDS).
 *  row_perm  device int32 [B*H, nQB] or NULL (see bsa_reorder_rows).
 *  scale     logit scale; <= 0 selects 1/sqrt(D); a NaN or infinite scale
 *            is rejected (BSA_ERR_INVALID_ARG).
 *  o         device bf16 [B, H, N, D] out, 16-byte aligned.
 *  lse       device fp32 [B, H, N] out.
 */
bsa_status bsa_forward(const void* q, const void* k, const void* v, int32_t B, int32_t H,
                       int32_t N, int32_t D, const int32_t* kv_idx, const int32_t* kv_cnt,
                       int32_t max_kv, const float* log_w, const int32_t* q_map,
                       const int32_t* kv_map, const int32_t* row_perm, float scale, void* o,
                       float* lse, void* stream);

/*
 * bsa_forward_masked - bsa_forward with grouped key/value heads and a token
 * mask inside the listed blocks.
 *
 * Defined by: INTRA, "Mapping Back to INTRA" (block-level sparse layers
 * subject to causal masking; sliding windows with sink tokens), "CQS-Aware
 * Token-Sparse FlashAttention Kernel" (masking within the packed tiles) and
 * "Attention Timing Comparison" (32 query heads over 8 key/value heads).
 *
 * As bsa_forward, except:
 *  - k and v hold H_kv heads per batch entry, [B, H_kv, N, D]; query head h
 *    of batch entry b reads key/value head b*H_kv + h/(H/H_kv).  kv_map, if
 *    given, is [B*H_kv, N].  H must be a multiple of H_kv.
 *  - With i the original query token and j the original key token (after
 *    the maps), key j is dropped from row i's softmax unless
 *        j < n_valid                        (n_valid = 0: N)
 *        and (causal == 0 or j <= i)
 *        and (window == 0 or j > i - window or j < sinks).
 *    A row whose listed keys are all dropped gets O = 0 and LSE = -inf.
 *    Dropped keys still cost their block's work: list only blocks that hold
 *    some visible key.
 *  - Without a mask (causal = 0, window = 0, n_valid = 0 or N) the result is
 *    bit-identical to bsa_forward on K/V heads repeated H/H_kv times.
 *  - Scheduling: when window > 0 bounds every row to 16 listed blocks or
 *    fewer ((window + 254) / 128 + ceil(sinks / 128) <= 16) and no map is
 *    given, one thread block per SM walks the rows in order (short rows
 *    otherwise leave the tensor cores idle between blocks); else one thread
 *    block per row.  Results are bit-identical either way.
 *
 *  H_kv      1 .. H, dividing H.
 *  causal    0 or 1.   n_valid 0 .. N.   window >= 0.   sinks >= 0.
 */
bsa_status bsa_forward_masked(const void* q, const void* k, const void* v, int32_t B, int32_t H,
                              int32_t H_kv, int32_t N, int32_t D, const int32_t* kv_idx,
                              const int32_t* kv_cnt, int32_t max_kv, const float* log_w,
                              const int32_t* q_map, const int32_t* kv_map,
                              const int32_t* row_perm, int32_t causal, int32_t n_valid,
                              int32_t window, int32_t sinks, float scale, void* o, float* lse,
                              void* stream);

/*
 * bsa_forward_packed - bsa_forward_masked over key/value tiles packed
 * through a map that may repeat tokens, with per-quadrant visibility.
 *
 * Defined by: INTRA, "CQS-Aware Token-Sparse FlashAttention Kernel" (the
 * kernel loads the selected key/value tokens through an index mapping and
 * packs them into dense tiles; masking within the packed tiles) and
 * appendix "Sparse Pattern Index Function", Gather 0 (overlapping 16 x 16
 * key windows packed as key tiles).
 *
 * As bsa_forward_masked, except:
 *  - kv_map is [B*H_kv, N_kv] (N_kv a multiple of 128, not tied to N): key
 *    tile t of a key/value head holds tokens kv_map[.., 128 t .. 128 t + 127].
 *    Tiles may overlap (a token may appear in several tiles).  List entries
 *    name tiles 0 .. N_kv/128 - 1.  kv_map entries must lie in [0, N).
 *  - quad_mask (optional, NULL = all set) is uint8 [B*H*nQB, max_kv]: bit g
 *    of entry (row, j) set means query rows 32 g .. 32 g + 31 of the row's
 *    query tile see listed tile j; with the bit clear every key of that tile
 *    is dropped for those 32 rows (they skip its exponentials; the tile's
 *    matrix products still run for the whole query tile).  Bits 4..7 are
 *    ignored.  The token mask (causal, n_valid, window, sinks) applies on
 *    top, to the original key tokens.
 *  - Without quad_mask or token mask and with N_kv = N the result is
 *    bit-identical to bsa_forward_masked.
 *
 *  kv_map    required, 16-byte aligned.
 *  N_kv      128 .. 2^26, a multiple of 128; B*H_kv*N_kv < 2^40.
 *  max_kv    1 .. N_kv/128.
 */
bsa_status bsa_forward_packed(const void* q, const void* k, const void* v, int32_t B, int32_t H,
                              int32_t H_kv, int32_t N, int32_t D, const int32_t* kv_idx,
                              const int32_t* kv_cnt, int32_t max_kv, const float* log_w,
                              const int32_t* q_map, const int32_t* kv_map, int32_t N_kv,
                              const uint8_t* quad_mask, const int32_t* row_perm, int32_t causal,
                              int32_t n_valid, int32_t window, int32_t sinks, float scale, void* o,
                              float* lse, void* stream);

/*
 * bsa_gather0_sizes / bsa_gather0_layout - the INTRA Gather 0 image layer as
 * maps, lists and quadrant masks for bsa_forward_packed.
 *
 * Defined by: INTRA, appendix "Sparse Pattern Index Function", Gather 0,
 * and "Mapping Back to INTRA" (FLUX.1-dev: 512 text tokens ahead of the
 * image, Scatter with 8 groups).  The sequence is n_text text tokens
 * followed by an img_h x img_w image in row-major order (token n_text +
 * y*img_w + x).  Each 8 x 8 patch of image queries (patch row r, column c)
 * attends to the 16 x 16 window of image keys with top-left corner
 *     (clamp(8r - 4, 0, img_h - 16), clamp(8c - 4, 0, img_w - 16))
 * (the window centred on the patch, shifted inward at the image edges) and
 * to every text key.  Text query i belongs to Scatter group
 * g = i / (n_text / groups) and attends to every text key and to the image
 * tokens n_text + t*groups + g (t = 0 .. img_h*img_w/groups - 1).
 *
 * Layout (per head; heads identical copies):
 *  - query tiles 0 .. n_text/128 - 1 are the text tokens in order; query
 *    tile n_text/128 + s*(img_w/8) + c holds patch (2s, c) in rows 0..63 and
 *    patch (2s+1, c) in rows 64..127, each patch row-major;
 *  - key tiles 0 .. n_text/128 - 1 are the text tokens; then four tile
 *    slots per query tile pair for its windows' 8-row x 16-column bands
 *    (two per window; shared bands of the two windows stored once, so 2-4
 *    slots used); then, when n_text > 0, the Scatter groups, 128 tokens per
 *    tile in group order;
 *  - each list holds the text tiles (seen by all rows) and then the row's
 *    window bands or Scatter-group tiles in increasing tile order, with
 *    quad_mask giving the 32-row quadrants that see each;
 *  - unused list entries are 0 with quad_mask 0.
 *
 * bsa_gather0_sizes (host only) writes N = n_text + img_h*img_w, N_kv
 * (= n_text + 4*img_h*img_w, plus img_h*img_w when n_text > 0) and the
 * list capacity max_kv the layout needs.  bsa_gather0_layout writes the
 * device arrays q_map [heads, N], kv_map [heads, N_kv], kv_idx
 * [heads*N/128, max_kv], kv_cnt [heads*N/128], quad_mask [heads*N/128,
 * max_kv] (int32 arrays 16-byte aligned).  For grouped heads pass the first
 * B*H_kv copies of kv_map.
 *
 *  img_h     16 .. 4096, a multiple of 16 (two patch rows per query tile).
 *  img_w     16 .. 4096, a multiple of 8.
 *  n_text    0 .. 2^20, a multiple of 128.
 *  groups    with n_text > 0: n_text/groups a multiple of 32 and
 *            img_h*img_w/groups a multiple of 128; ignored when n_text = 0.
 *  heads     0 .. 65535 (0: nothing to do); max_kv >= the size returned.
 */
bsa_status bsa_gather0_sizes(int32_t img_h, int32_t img_w, int32_t n_text, int32_t groups,
                             int32_t* N, int32_t* N_kv, int32_t* max_kv);
bsa_status bsa_gather0_layout(int32_t img_h, int32_t img_w, int32_t n_text, int32_t groups,
                              int64_t heads, int32_t* q_map, int32_t* kv_map, int32_t* kv_idx,
                              int32_t* kv_cnt, uint8_t* quad_mask, int32_t max_kv, void* stream);

/*
 * bsa_forward_gather0 - the INTRA Gather 0 image layer, with every tile
 * fetched as one tensor-memory-access box computed from the layer's index
 * functions instead of through maps.
 *
 * Defined by: INTRA, appendix "Sparse Pattern Index Function", Gather 0
 * (query patches, 16 x 16 windows shifted inward at the edges, text keys)
 * and "CQS-Aware Token-Sparse FlashAttention Kernel" (index mappings
 * computed at run time, outputs scattered back).
 *
 * One thread block per SM walks the query tiles (rows of 7-8 tiles).  Same
 * result as bsa_forward_packed with the same quad_mask (bit for bit, also
 * with quad_mask = NULL) on the maps of bsa_gather0_layout, without reading
 * them: a query tile of two patches is
 * a 16-row x 8-column box of the image, a window band an 8-row x 16-column
 * box, a Scatter-group tile 128 tokens at stride groups, a text tile 128
 * consecutive tokens.  O and LSE rows go to the original tokens.
 *
 *  q, o      device bf16 [B, H, N, D], N = n_text + img_h*img_w.
 *  k, v      device bf16 [B, H_kv, N, D].
 *  kv_idx, kv_cnt, quad_mask   from bsa_gather0_layout with the same
 *            img_h, img_w, n_text, groups (quad_mask may be NULL: every
 *            quadrant sees every listed tile); max_kv their row stride.
 *  Geometry arguments as bsa_gather0_layout; other arguments as bsa_forward.
 */
bsa_status bsa_forward_gather0(const void* q, const void* k, const void* v, int32_t B, int32_t H,
                               int32_t H_kv, int32_t D, int32_t img_h, int32_t img_w, int32_t n_text,
                               int32_t groups, const int32_t* kv_idx, const int32_t* kv_cnt,
                               const uint8_t* quad_mask, int32_t max_kv, const int32_t* row_perm,
                               float scale, void* o, float* lse, void* stream);

/*
 * bsa_forward_scatter - block-sparse attention over the Scatter layer's
 * gathered order, with every tile fetched as one tensor-memory-access box.
 *
 * Defined by: INTRA, "Why Scatter Is Uniform and Non-Contiguous" (N = R*T
 * tokens as (t, r) = t*R + r in T neighbourhoods of R; group S_r = {(t, r)})
 * and "CQS-Aware Token-Sparse FlashAttention Kernel" (mappings computed at
 * run time, outputs scattered back).
 *
 * One thread block per SM walks the rows (each row is short: the launch,
 * prologue and epilogue of a block per row would dominate).
 *
 * The result is bsa_forward_masked without a token mask on the maps
 *     q_map[bh][p] = kv_map[bh][p] = (p mod T)*R + p / T,   T = N / R,
 * for every head (gathered position p = r*T + t holds token t*R + r), bit
 * for bit, without reading maps: a 128-position tile is 128 tokens of one
 * group at stride R.  List entries name gathered blocks 0 .. N/128 - 1 (block
 * b covers group b / (T/128)); O and LSE rows go to the original tokens.
 *
 *  R         1 .. N, dividing N, with N / R a multiple of 128.
 *  k, v      device bf16 [B, H_kv, N, D] (H_kv dividing H).
 *  Other arguments as bsa_forward.
 */
bsa_status bsa_forward_scatter(const void* q, const void* k, const void* v, int32_t B, int32_t H,
                               int32_t H_kv, int32_t N, int32_t D, int32_t R, const int32_t* kv_idx,
                               const int32_t* kv_cnt, int32_t max_kv, const float* log_w,
                               const int32_t* row_perm, float scale, void* o, float* lse, void* stream);

/*
 * bsa_gather_rows - token rows permuted into gathered order in HBM:
 *     dst[bh][p][:] = src[bh][map[bh][p]][:]    for p in 0..N-1.
 *
 * Defined by: InstaGen, section 3.3 and Introduction (permuted block-sparse
 * attention: tokens permuted so that every cluster is a contiguous block)
 * and INTRA, "CQS-Aware Token-Sparse FlashAttention Kernel" (the index
 * maps).  bsa_forward with kv_map reads the same rows through the map
 * inside the kernel; calling bsa_forward on the outputs of this call with
 * kv_map = NULL gives the same O and LSE (bit for bit) and loads every
 * listed block as one contiguous tile.  That pays when a head's key/value
 * blocks are listed by several query blocks each; a row-granular gather
 * inside the kernel costs the same for every listing.
 *
 *  src     device bf16 [heads, N, D] contiguous, 16-byte aligned.
 *  map     device int32 [heads, N], 4-byte aligned; entries in [0, N).  An
 *          entry outside [0, N) writes a zero row and raises
 *          BSA_ERR_BOUNDS.  Duplicate entries are allowed (rows repeat).
 *  heads   0 .. 65535 (0: nothing to do); N 1 .. 2^24; heads * N < 2^31.
 *  D       64 or 128.
 *  dst     device bf16 [heads, N, D] out, 16-byte aligned; must not overlap
 *          src.
 */
bsa_status bsa_gather_rows(const void* src, const int32_t* map, int64_t heads, int32_t N,
                           int32_t D, void* dst, void* stream);

/*
 * bsa_build_crm - the CRM (compressed row mask) form of a mask or threshold
 * map: per row, uint32 words in which bit i of word w is set when KV block
 * 32w + i is kept (ScalingAttention, section 7.2: one 32-bit load decodes 32
 * block states).  Same selection as bsa_build_index (MASK / THRESHOLD);
 * bits at or beyond nKB are 0.
 *
 *  rows       0 .. 8 * (2^31 - 1), as for bsa_build_index.
 *  words      device uint32 [rows, crm_words] out; crm_words >= ceil(nKB/32)
 *             (words beyond ceil(nKB/32) are written as 0).
 */
bsa_status bsa_build_crm(bsa_idx_mode mode, const void* src, int64_t rows, int32_t nKB, float p,
                         uint32_t* words, int32_t crm_words, void* stream);

/*
 * bsa_forward_crm - bsa_forward with the KV-block sets given as CRM rows.
 *
 * Defined by: ScalingAttention, sections 7.2-7.3 (CRM rows walked with bit
 * scan and bit clear in place of the dense block iterator; Algorithm 2).
 * The forward pass visits the set bits of each row in ascending block order
 * (count trailing zeros, then clear the lowest bit); results equal
 * bsa_forward on the equivalent index lists.  No per-block log-weights.
 *
 *  crm        device uint32 [B*H*nQB, crm_words], crm_words >= ceil(nKB/32);
 *             bits at or beyond nKB must be 0 (else BSA_ERR_BOUNDS, row
 *             unspecified).  Other arguments as bsa_forward.
 */
bsa_status bsa_forward_crm(const void* q, const void* k, const void* v, int32_t B, int32_t H,
                           int32_t N, int32_t D, const uint32_t* crm, int32_t crm_words,
                           const int32_t* q_map, const int32_t* kv_map, const int32_t* row_perm,
                           float scale, void* o, float* lse, void* stream);

/*
 * bsa_upscale_threshold - carry a threshold map built at a base resolution
 * to a target resolution (ScalingAttention, section 7.1 eq. (7),
 * R_target(u, v) = ceil(Phi(R_base, u / s_h, v / s_w)), Phi bilinear).
 *
 * Target block u samples base coordinate u * Ub / Ut (likewise v); on every
 * mask M_p = I(T <= p) the ceiling keeps a target block when any base block
 * with a nonzero bilinear weight is active, so the target threshold is the
 * minimum of T over those (one or two per axis, the upper index clamped).
 *
 *  T_base    device fp32 [heads, Ub, Vb];  T_target device fp32 [heads, Ut, Vt] out.
 *  heads <= 65535, Ut <= 65535; Ub, Vb, Vt <= 65536 (all >= 1).
 */
bsa_status bsa_upscale_threshold(const float* T_base, int64_t heads, int32_t Ub, int32_t Vb,
                                 int32_t Ut, int32_t Vt, float* T_target, void* stream);

/*
 * bsa_set_forward_options - how this host thread's later forward calls
 * launch (every bsa_forward* entry point).  The result does not depend on
 * the schedule: every choice computes the same per-row arithmetic, bit for
 * bit.  The exponential option changes the last bits of O and LSE.
 *
 *  schedule   BSA_SCHEDULE_AUTO (default): per-item thread blocks for the
 *             Scatter and Gather 0 layers and for windowed token masks that
 *             bound every row to 16 listed blocks, one thread block per row
 *             otherwise;  BSA_SCHEDULE_PER_ROW: one thread block per query
 *             block always;  BSA_SCHEDULE_PER_ITEM: one thread block per SM
 *             walking the rows wherever the per-item kernel applies (the
 *             Scatter and Gather 0 layers, and the tile path without maps).
 *  exp2_fma   0 (default) or 2: exponentials out of every 8 that the plain
 *             tile path (bsa_forward without maps, masks or CRM rows)
 *             computes on the FMA pipe (Cody-Waite reduction and a degree-3
 *             minimax polynomial, 7.5e-5 relative error) instead of
 *             ex2.approx; other paths ignore it.
 * o = NULL restores the defaults.  The options are per host thread (thread
 * local storage in the library); other threads keep theirs.
 */
typedef enum {
    BSA_SCHEDULE_AUTO = 0,
    BSA_SCHEDULE_PER_ROW = 1,
    BSA_SCHEDULE_PER_ITEM = 2
} bsa_schedule;

typedef struct {
    bsa_schedule schedule;
    int32_t exp2_fma;
} bsa_forward_options;

bsa_status bsa_set_forward_options(const bsa_forward_options* o);

/*
 * bsa_device_status - read and clear the status word of the current device.
 * Synchronises `stream` first.  *first_error (host pointer) receives the
 * first device-side bsa_status code raised since the last read (BSA_OK if
 * none).  Returns BSA_ERR_CUDA if the synchronisation or copy failed.
 */
bsa_status bsa_device_status(void* stream, int32_t* first_error);

/*
 * bsa_resident_ctas - how many bsa_forward thread blocks the current device
 * runs at once for head dimension D (SM count x resident blocks per SM):
 * the wave size W that WaveAlign's scheduling model uses.  Returns a value
 * <= 0 on error (no device, bad D).
 */
int32_t bsa_resident_ctas(int32_t D);

/* Human-readable name of a status code (static string). */
const char* bsa_status_string(int32_t status);

#ifdef __cplusplus
}
#endif

#endif /* BSA_H */
