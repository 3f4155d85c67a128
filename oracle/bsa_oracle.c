/*
 * Block-sparse attention oracle: plain, slow, obviously-correct CPU code.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or helper with the
 * CUDA library.  Floating point is IEEE binary64 throughout; the inputs that
 * arrive as bf16 or fp32 are widened exactly.  Build with
 * -ffp-contract=off so that no multiply-add is fused: the sampler below
 * takes integer decisions from fp64 sums and must round exactly as written.
 *
 * What each function follows (page title, then the passage):
 *   oracle_index_mask_u8   WaveAlign, "B. Sparse Attention for Long-Video
 *                          Generation": a mask row per query block, a kept
 *                          entry per executed (query block, KV block) pair.
 *   oracle_index_threshold ScalingAttention, section 5.2 eq. (2):
 *                          M_p = I(T <= p), compared in fp32.
 *   oracle_index_topk      MC-Sparse, "The MC-Sparse Architecture" (keep the
 *                          highest-scoring KV blocks of a query block) and
 *                          InstaGen section 3.2.1 (top-k = the heavy set).
 *   oracle_reorder_rows    WaveAlign, section IV-D "NNZ-Guided Intra-Wave
 *                          Temporal Alignment": consecutive buckets of at
 *                          most W rows, each sorted by descending NNZ.
 *   oracle_sample_blocks   InstaGen, section 3.2.1 eq. (4) (inclusion
 *                          probabilities, cap at 1 and renormalise), the
 *                          promotion of pi = 1 keys, systematic PPS sampling,
 *                          and Algorithm 1 step 13 (w = 1/pi).
 *   oracle_crm_rows        ScalingAttention, section 7.2 (CRM bitmask rows).
 *   oracle_upscale_threshold ScalingAttention, section 7.1 eq. (7).
 *   oracle_block_scores    MC-Sparse, "The MC-Sparse Architecture" (mean-pooled
 *                          block similarity) and InstaGen Algorithm 1 step 2
 *                          (centroid scores exp(q_g . k_c / sqrt d)).
 *   oracle_spectral_order  WaveAlign, section IV-C (rank-2 embedding of the
 *                          centered mask by matrix-free subspace iteration,
 *                          rows ordered by polar angle).
 *   oracle_attention       InstaGen, section 3.1 eqs. (1)-(3) and Algorithm 1
 *                          step 14 (softmax of l_ij + log w_j over the kept
 *                          keys); INTRA, "CQS-Aware Token-Sparse
 *                          FlashAttention Kernel" (keys and queries reached
 *                          through index maps, outputs scattered back).
 *   oracle_gather0_set     INTRA, appendix "Sparse Pattern Index Function",
 *                          Gather 0 (8 x 8 query patch, 16 x 16 key window
 *                          shifted inward at the edges, text tokens first)
 *                          and "Mapping Back to INTRA" (text queries keep
 *                          their Scatter image-key groups; Scatter groups
 *                          same-position tokens, "Why Scatter Is Uniform").
 *   oracle_attention_set   the softmax attention of one query set over one
 *                          key set (InstaGen section 3.1 eqs. (1)-(3)).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_BLOCK 128 /* query and key block edge (ScalingAttention 5.1, B = 128) */

/* bf16 bit pattern -> exact double (bf16 is the top half of an fp32). */
static double bf16_to_double(uint16_t h) {
    uint32_t bits = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------------- */
/* Index lists from a mask or a threshold map.                               */
/* A row keeps the KV blocks whose predicate holds, in ascending block       */
/* order.  A row with more than max_kv kept blocks is truncated to its first */
/* max_kv entries and counted as an overflow; the return value is the number */
/* of overflowing rows.                                                      */
/* ------------------------------------------------------------------------- */
static int32_t emit_row(const uint8_t* keep, int32_t nKB, int32_t* idx_row,
                        int32_t max_kv, int32_t* cnt_out) {
    int32_t n = 0, total = 0;
    for (int32_t kb = 0; kb < nKB; ++kb) {
        if (!keep[kb]) continue;
        if (n < max_kv) idx_row[n++] = kb;
        ++total;
    }
    for (int32_t e = n; e < max_kv; ++e) idx_row[e] = -1;
    *cnt_out = n;
    return total > max_kv;
}

int64_t oracle_index_mask_u8(const uint8_t* mask, int64_t rows, int32_t nKB,
                             int32_t* kv_idx, int32_t* kv_cnt, int32_t max_kv) {
    int64_t overflow = 0;
    uint8_t* keep = (uint8_t*)malloc((size_t)nKB);
    for (int64_t r = 0; r < rows; ++r) {
        for (int32_t kb = 0; kb < nKB; ++kb) keep[kb] = mask[r * nKB + kb] != 0;
        overflow += emit_row(keep, nKB, kv_idx + r * max_kv, max_kv, kv_cnt + r);
    }
    free(keep);
    return overflow;
}

int64_t oracle_index_threshold(const float* T, int64_t rows, int32_t nKB, float p,
                               int32_t* kv_idx, int32_t* kv_cnt, int32_t max_kv) {
    int64_t overflow = 0;
    uint8_t* keep = (uint8_t*)malloc((size_t)nKB);
    for (int64_t r = 0; r < rows; ++r) {
        /* M_p = I(T <= p): inclusive, both operands fp32. */
        for (int32_t kb = 0; kb < nKB; ++kb) keep[kb] = T[r * nKB + kb] <= p;
        overflow += emit_row(keep, nKB, kv_idx + r * max_kv, max_kv, kv_cnt + r);
    }
    free(keep);
    return overflow;
}

/* ------------------------------------------------------------------------- */
/* Top-k per row: a full sort by (score descending, block ascending), keep   */
/* the first k, then list the kept blocks in ascending block order.          */
/* ------------------------------------------------------------------------- */
typedef struct {
    float s;
    int32_t kb;
} scored_t;

static int by_score_desc_then_kb(const void* a, const void* b) {
    const scored_t* x = (const scored_t*)a;
    const scored_t* y = (const scored_t*)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->kb > y->kb) - (x->kb < y->kb);
}

int64_t oracle_index_topk(const float* scores, int64_t rows, int32_t nKB,
                          const int32_t* k_per_row, int32_t k_const,
                          int32_t* kv_idx, int32_t* kv_cnt, int32_t max_kv) {
    int64_t overflow = 0;
    scored_t* tmp = (scored_t*)malloc(sizeof(scored_t) * (size_t)nKB);
    uint8_t* keep = (uint8_t*)malloc((size_t)nKB);
    for (int64_t r = 0; r < rows; ++r) {
        int32_t k = k_per_row ? k_per_row[r] : k_const;
        if (k > nKB) k = nKB;
        if (k < 0) k = 0;
        for (int32_t kb = 0; kb < nKB; ++kb) {
            tmp[kb].s = scores[r * nKB + kb];
            tmp[kb].kb = kb;
        }
        qsort(tmp, (size_t)nKB, sizeof(scored_t), by_score_desc_then_kb);
        memset(keep, 0, (size_t)nKB);
        for (int32_t i = 0; i < k; ++i) keep[tmp[i].kb] = 1;
        overflow += emit_row(keep, nKB, kv_idx + r * max_kv, max_kv, kv_cnt + r);
    }
    free(keep);
    free(tmp);
    return overflow;
}

/* ------------------------------------------------------------------------- */
/* Query-row reordering, stage 2 of WaveAlign.  For each head the input     */
/* order (identity when order_in is NULL) is cut into consecutive buckets of */
/* `wave` slots; each bucket is stably sorted by descending KV-block count.  */
/* row_perm[h][slot] is the query block that runs in that execution slot.    */
/* ------------------------------------------------------------------------- */
void oracle_reorder_rows(const int32_t* kv_cnt, const int32_t* order_in, int64_t heads,
                         int32_t nQB, int32_t wave, int32_t* row_perm) {
    int32_t* ord = (int32_t*)malloc(sizeof(int32_t) * (size_t)nQB);
    for (int64_t h = 0; h < heads; ++h) {
        const int32_t* cnt = kv_cnt + h * nQB;
        for (int32_t i = 0; i < nQB; ++i) ord[i] = order_in ? order_in[h * nQB + i] : i;
        for (int32_t b0 = 0; b0 < nQB; b0 += wave) {
            int32_t b1 = b0 + wave < nQB ? b0 + wave : nQB;
            /* stable insertion sort on descending count */
            for (int32_t i = b0 + 1; i < b1; ++i) {
                int32_t q = ord[i];
                int32_t j = i - 1;
                while (j >= b0 && cnt[ord[j]] < cnt[q]) {
                    ord[j + 1] = ord[j];
                    --j;
                }
                ord[j + 1] = q;
            }
        }
        memcpy(row_perm + h * nQB, ord, sizeof(int32_t) * (size_t)nQB);
    }
    free(ord);
}

/* ------------------------------------------------------------------------- */
/* Exact set + PPSWOR sample of the residual, InstaGen section 3.2.1.        */
/*                                                                           */
/* Per row: the residual R is every KV block not in the exact list.  The     */
/* inclusion probabilities are pi_j = min(1, lambda s_j) with                */
/* sum_R pi_j = m (eq. 4), found by capping at 1 and renormalising until the */
/* capped set stops growing.  Capped blocks (pi = 1) are promoted: always    */
/* kept, weight 1.  The other m' = m - |capped| blocks are drawn by          */
/* systematic PPS: with one uniform u in [0,1) the points u, u+1, ...,       */
/* u+m'-1 are laid on the running sum C_j of pi over the uncapped residual   */
/* in ascending block order, and block j is drawn when a point falls in      */
/* [C_{j-1}, C_j), i.e. when ceil(C_j - u) > ceil(C_{j-1} - u).  Every drawn */
/* block gets log-weight -log(pi_j) (Algorithm 1 step 13, w = 1/pi).        */
/*                                                                           */
/* Output list: exact, promoted and sampled blocks merged in ascending block */
/* order, with log_w 0 for exact and promoted entries.  Returns the number   */
/* of rows whose merged list did not fit in max_kv (truncated).              */
/* Arithmetic: these floating-point values decide integers (which blocks    */
/* are capped and drawn), so they are computed in the GPU sampler's          */
/* precision, fp32 (the pages fix none): sums in ascending block order,      */
/* IEEE round-to-nearest, no fused multiply-adds (the file is built with     */
/* -ffp-contract=off).  u is rounded to fp32 first.  The log-weights are     */
/* -log(pi) evaluated in double from the fp32 pi and rounded to fp32.        */
/* ------------------------------------------------------------------------- */
int64_t oracle_sample_blocks(const float* scores, int64_t rows, int32_t nKB,
                             const int32_t* exact_idx, const int32_t* exact_cnt,
                             int32_t exact_stride, int32_t m, const double* u,
                             int32_t* kv_idx, int32_t* kv_cnt, float* log_w,
                             int32_t max_kv) {
    int64_t overflow = 0;
    uint8_t* state = (uint8_t*)malloc((size_t)nKB); /* 0 residual, 1 exact, 2 promoted, 3 sampled */
    float* pi = (float*)malloc(sizeof(float) * (size_t)nKB);
    /* NULL scores: the uniform sampler (InstaGen Algorithm 1 steps 6-8), i.e.
       every residual block with the same score and pi_j = m / |R|. */
    float* ones = NULL;
    if (!scores) {
        ones = (float*)malloc(sizeof(float) * (size_t)nKB);
        for (int32_t kb = 0; kb < nKB; ++kb) ones[kb] = 1.0f;
    }
    for (int64_t r = 0; r < rows; ++r) {
        const float* s = scores ? scores + r * nKB : ones;
        memset(state, 0, (size_t)nKB);
        for (int32_t e = 0; e < exact_cnt[r]; ++e) state[exact_idx[r * exact_stride + e]] = 1;
        int32_t n_res = 0;
        for (int32_t kb = 0; kb < nKB; ++kb) n_res += state[kb] == 0;

        if (n_res <= m) {
            /* the budget covers the whole residual: every block has pi = 1 */
            for (int32_t kb = 0; kb < nKB; ++kb)
                if (state[kb] == 0) state[kb] = 2;
        } else {
            /* eq. (4): cap at 1 and renormalise until the capped set is stable */
            int32_t n_cap = 0;
            float lambda = 0.0f;
            for (;;) {
                float sum = 0.0f;
                for (int32_t kb = 0; kb < nKB; ++kb)
                    if (state[kb] == 0) sum += s[kb];
                lambda = (float)(m - n_cap) / sum;
                int32_t grew = 0;
                for (int32_t kb = 0; kb < nKB; ++kb) {
                    if (state[kb] == 0 && lambda * s[kb] >= 1.0f) {
                        state[kb] = 2;
                        ++n_cap;
                        grew = 1;
                    }
                }
                if (!grew) break;
            }
            /* systematic PPS over the uncapped residual */
            const int32_t m_rest = m - n_cap;
            const float ur = (float)u[r];
            float C = 0.0f;
            int32_t drawn = 0;
            for (int32_t kb = 0; kb < nKB; ++kb) {
                if (state[kb] != 0) continue;
                const float p = lambda * s[kb];
                const float C_prev = C;
                C = C + p;
                if (drawn < m_rest && ceilf(C - ur) > ceilf(C_prev - ur)) {
                    state[kb] = 3;
                    pi[kb] = p;
                    ++drawn;
                }
            }
        }
        /* merge in ascending block order */
        int32_t n = 0, total = 0;
        for (int32_t kb = 0; kb < nKB; ++kb) {
            if (state[kb] == 0) continue;
            if (n < max_kv) {
                kv_idx[r * max_kv + n] = kb;
                log_w[r * max_kv + n] = state[kb] == 3 ? (float)(-log((double)pi[kb])) : 0.0f;
                ++n;
            }
            ++total;
        }
        for (int32_t e = n; e < max_kv; ++e) {
            kv_idx[r * max_kv + e] = -1;
            log_w[r * max_kv + e] = 0.0f;
        }
        kv_cnt[r] = n;
        overflow += total > max_kv;
    }
    free(ones);
    free(pi);
    free(state);
    return overflow;
}

/* ------------------------------------------------------------------------- */
/* Masked, log-weighted softmax attention from its definition.               */
/*                                                                           */
/* Tensor q is a bf16 bit pattern laid out [B*H, N, D].  Gathered           */
/* position p of head bh holds query token q_map[bh][p] (p itself when       */
/* q_map is NULL) and key/value token kv_map[bh][p] (likewise).  The query   */
/* block of p is p / 128; its KV list is kv_idx[row][0..kv_cnt[row]) with   */
/* row = bh * nQB + qb, and list entry e covers gathered key positions       */
/* 128*kb .. 128*kb+127, all with log-weight log_w[row][e] (0 when NULL).    */
/*                                                                           */
/* For each selected query block (sel[i] = bh * nQB + qb) and each of its    */
/* 128 positions p, with i = q_map(p):                                       */
/*     s_j   = (q_i . k_j) * scale + lw          over every listed key j     */
/*     LSE_i = ln sum_j exp(s_j)                 (max-shifted)               */
/*     O_i   = sum_j exp(s_j - LSE_i) v_j                                    */
/* Grouped keys/values (INTRA, "Attention Timing Comparison": 32 query      */
/* heads over 8 key/value heads): k, v and kv_map hold H_kv heads per batch  */
/* entry, and query head h of batch b reads key/value head                   */
/* b * H_kv + h / (H / H_kv).                                                */
/*                                                                           */
/* Token mask (INTRA, "Mapping Back to INTRA" and "CQS-Aware Token-Sparse    */
/* FlashAttention Kernel": causal masking inside packed tiles, sliding       */
/* windows with sink tokens): key token j is dropped from query token i's   */
/* sum unless                                                                */
/*     j < n_valid                      (tail padding; n_valid <= 0: N)      */
/*     and (!causal or j <= i)                                               */
/*     and (window <= 0 or j > i - window or j < sinks).                     */
/* An empty list, or a row whose listed keys are all dropped, gives          */
/* O_i = 0 and LSE_i = -inf.  Results go to                                  */
/* O[(i_sel*128 + r) * D + d], LSE[i_sel*128 + r], and tok[...] = i, the     */
/* original token the row belongs to (the scatter-back target).             */
/* scale <= 0 selects 1/sqrt(D).                                             */
/* ------------------------------------------------------------------------- */
void oracle_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                      int32_t B, int32_t H, int32_t H_kv, int32_t N, int32_t D,
                      const int32_t* kv_idx, const int32_t* kv_cnt, int32_t max_kv,
                      const float* log_w, const int32_t* q_map, const int32_t* kv_map,
                      int32_t causal, int32_t n_valid, int32_t window, int32_t sinks,
                      double scale, const int64_t* sel, int64_t nsel,
                      double* O, double* LSE, int32_t* tok) {
    const int32_t nQB = N / ORACLE_BLOCK;
    if (scale <= 0.0) scale = 1.0 / sqrt((double)D);
    if (n_valid <= 0) n_valid = N;
    const int32_t group = H / H_kv;
    (void)B;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t w = 0; w < nsel * ORACLE_BLOCK; ++w) {
        const int64_t i_sel = w / ORACLE_BLOCK;
        const int32_t r = (int32_t)(w % ORACLE_BLOCK);
        const int64_t row = sel[i_sel];
        const int64_t bh = row / nQB;
        const int32_t qb = (int32_t)(row % nQB);
        const int32_t p = qb * ORACLE_BLOCK + r;
        const int32_t i = q_map ? q_map[bh * N + p] : p;
        const int64_t kvh = (bh / H) * H_kv + (bh % H) / group; /* key/value head */
        const int32_t cnt = kv_cnt[row];
        double* o = O + w * D;
        tok[w] = i;
        for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
        if (cnt <= 0) {
            LSE[w] = -INFINITY;
            continue;
        }
        const int64_t nkeys = (int64_t)cnt * ORACLE_BLOCK;
        double* s = (double*)malloc(sizeof(double) * (size_t)nkeys);
        int32_t* key = (int32_t*)malloc(sizeof(int32_t) * (size_t)nkeys);
        double* qi = (double*)malloc(sizeof(double) * (size_t)D);
        for (int32_t d = 0; d < D; ++d) qi[d] = bf16_to_double(q[(bh * N + i) * D + d]);
        for (int32_t e = 0; e < cnt; ++e) {
            const int32_t kb = kv_idx[row * max_kv + e];
            const double lw = log_w ? (double)log_w[row * max_kv + e] : 0.0;
            for (int32_t t = 0; t < ORACLE_BLOCK; ++t) {
                const int32_t pos = kb * ORACLE_BLOCK + t;
                const int32_t j = kv_map ? kv_map[kvh * N + pos] : pos;
                const int visible = j < n_valid && (!causal || j <= i) &&
                                    (window <= 0 || j > i - window || j < sinks);
                double dot = 0.0;
                for (int32_t d = 0; d < D; ++d) dot += qi[d] * bf16_to_double(k[(kvh * N + j) * D + d]);
                s[e * ORACLE_BLOCK + t] = visible ? dot * scale + lw : -INFINITY;
                key[e * ORACLE_BLOCK + t] = j;
            }
        }
        double mx = -INFINITY;
        for (int64_t x = 0; x < nkeys; ++x) mx = s[x] > mx ? s[x] : mx;
        if (mx == -INFINITY) { /* every listed key dropped */
            LSE[w] = -INFINITY;
            free(qi);
            free(key);
            free(s);
            continue;
        }
        double z = 0.0;
        for (int64_t x = 0; x < nkeys; ++x) z += exp(s[x] - mx);
        const double lse = mx + log(z);
        for (int64_t x = 0; x < nkeys; ++x) {
            const double a = exp(s[x] - lse);
            if (s[x] == -INFINITY) continue;
            const uint16_t* vj = v + (kvh * N + key[x]) * D;
            for (int32_t d = 0; d < D; ++d) o[d] += a * bf16_to_double(vj[d]);
        }
        LSE[w] = lse;
        free(qi);
        free(key);
        free(s);
    }
}

/* ------------------------------------------------------------------------- */
/* INTRA Gather 0: the query set and key set of one CQS.                     */
/*                                                                           */
/* The sequence is n_text text tokens followed by an img_h x img_w image in  */
/* zero-based row-major order: pixel (y, x) is token n_text + y*img_w + x.   */
/* Sets 0 .. img_h*img_w/64 - 1 are the image CQS in the page's order: for   */
/* CQS index i, r = i / (img_w/8) and c = i mod (img_w/8); its 64 queries   */
/* are the 8 x 8 patch                                                       */
/*     i_l^q -> pixel (8r + i_l^q / 8, 8c + i_l^q mod 8),   0 <= i_l^q < 64  */
/* and its 256 image keys the 16 x 16 window with top-left corner            */
/*     (r0, c0) = (clamp(8r - 4, 0, img_h - 16), clamp(8c - 4, 0, img_w - 16))*/
/*     i_l^k -> pixel (r0 + i_l^k / 16, c0 + i_l^k mod 16), 0 <= i_l^k < 256 */
/* (the page's four 64-key tiles i_l^k = 64t + j cover rows r0 + 4t ..      */
/* r0 + 4t + 3, i.e. the same order), preceded by every text key.  The page  */
/* prints neither equation; the window centred on the patch and clamped      */
/* inside the image is the plain reading of "shifted inward at image         */
/* boundaries" with every index in [0, HW).                                  */
/* Sets img_h*img_w/64 + g (0 <= g < groups, only when n_text > 0) are the   */
/* text queries of Scatter group g, i = g*(n_text/groups) .. +n_text/groups  */
/* - 1, with every text key and the image tokens of Scatter group g: with   */
/* image token index u = t*groups + g (neighbourhood t, local index g), the  */
/* tokens n_text + t*groups + g for t = 0 .. img_h*img_w/groups - 1.        */
/* Writes *nq query tokens to q_tok and returns the number of key tokens     */
/* written to k_tok (-1 for a set index out of range).                       */
/* ------------------------------------------------------------------------- */
static int64_t clamp64(int64_t x, int64_t lo, int64_t hi) { return x < lo ? lo : (x > hi ? hi : x); }

int64_t oracle_gather0_set(int32_t img_h, int32_t img_w, int32_t n_text, int32_t groups,
                           int64_t set, int32_t* q_tok, int64_t* nq, int32_t* k_tok) {
    const int64_t hw = (int64_t)img_h * img_w, n_img = hw / 64;
    int64_t nk = 0;
    if (set >= 0 && set < n_img) {
        const int64_t r = set / (img_w / 8), c = set % (img_w / 8);
        for (int64_t il = 0; il < 64; ++il)
            q_tok[il] = (int32_t)(n_text + (8 * r + il / 8) * img_w + 8 * c + il % 8);
        *nq = 64;
        for (int64_t j = 0; j < n_text; ++j) k_tok[nk++] = (int32_t)j;
        const int64_t r0 = clamp64(8 * r - 4, 0, img_h - 16), c0 = clamp64(8 * c - 4, 0, img_w - 16);
        for (int64_t lk = 0; lk < 256; ++lk)
            k_tok[nk++] = (int32_t)(n_text + (r0 + lk / 16) * img_w + c0 + lk % 16);
        return nk;
    }
    const int64_t g = set - n_img;
    if (n_text <= 0 || groups <= 0 || g < 0 || g >= groups) return -1;
    const int64_t per = n_text / groups;
    for (int64_t i = 0; i < per; ++i) q_tok[i] = (int32_t)(g * per + i);
    *nq = per;
    for (int64_t j = 0; j < n_text; ++j) k_tok[nk++] = (int32_t)j;
    for (int64_t t = 0; t < hw / groups; ++t) k_tok[nk++] = (int32_t)(n_text + t * groups + g);
    return nk;
}

/* ------------------------------------------------------------------------- */
/* Softmax attention of the query tokens q_tok[0..nq) of query head bh over  */
/* the key tokens k_tok[0..nk) of key/value head kvh (tensors [heads, N, D]  */
/* as bf16 bit patterns):                                                    */
/*     s_j = (q_i . k_j) * scale,  LSE_i = ln sum_j exp(s_j),                */
/*     O_i = sum_j exp(s_j - LSE_i) v_j.                                     */
/* Row x of O [nq, D] and LSE [nq] belongs to query token q_tok[x].  nk = 0  */
/* gives O = 0, LSE = -inf.  scale <= 0 selects 1/sqrt(D).                   */
/* ------------------------------------------------------------------------- */
void oracle_attention_set(const uint16_t* q, const uint16_t* k, const uint16_t* v, int32_t N,
                          int32_t D, int64_t bh, int64_t kvh, int64_t nq, const int32_t* q_tok,
                          int64_t nk, const int32_t* k_tok, double scale, double* O, double* LSE) {
    if (scale <= 0.0) scale = 1.0 / sqrt((double)D);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t x = 0; x < nq; ++x) {
        const int64_t i = q_tok[x];
        double* o = O + x * D;
        for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
        if (nk <= 0) {
            LSE[x] = -INFINITY;
            continue;
        }
        double* s = (double*)malloc(sizeof(double) * (size_t)nk);
        double mx = -INFINITY;
        for (int64_t e = 0; e < nk; ++e) {
            const int64_t j = k_tok[e];
            double dot = 0.0;
            for (int32_t d = 0; d < D; ++d)
                dot += bf16_to_double(q[(bh * N + i) * D + d]) * bf16_to_double(k[(kvh * N + j) * D + d]);
            s[e] = dot * scale;
            mx = s[e] > mx ? s[e] : mx;
        }
        double z = 0.0;
        for (int64_t e = 0; e < nk; ++e) z += exp(s[e] - mx);
        const double lse = mx + log(z);
        for (int64_t e = 0; e < nk; ++e) {
            const double a = exp(s[e] - lse);
            const uint16_t* vj = v + (kvh * N + k_tok[e]) * D;
            for (int32_t d = 0; d < D; ++d) o[d] += a * bf16_to_double(vj[d]);
        }
        LSE[x] = lse;
        free(s);
    }
}

/* Number of threads the OpenMP runtime will use (reported by the timer). */
int32_t oracle_num_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------- */
/* Spectral row order, WaveAlign section IV-C ("SVD-Based Global Spatial    */
/* Ordering": polar spectral ordering and matrix-free centered subspace      */
/* iteration).                                                               */
/*                                                                           */
/* Per head the mask A (rows = query blocks, columns = KV blocks, A[r][c] = */
/* 1 when c is in row r's list) is centered by its mean row mu, so that     */
/* pairwise row distances are kept and the all-ones direction gets a zero   */
/* singular value.  The top-2 left singular subspace of the centered mask   */
/* is found by subspace iteration that never forms it:                      */
/*     Z = A^T X - mu (1^T X)          (the rank-1 centering correction)     */
/*     Y = A Z   - 1 (mu^T Z)                                                */
/*     X = Gram-Schmidt(Y)                                                   */
/* starting from the given X0 (orthonormalised first).  Each row's polar    */
/* angle atan2(X[r][1], X[r][0]) then orders the rows (ascending, ties to   */
/* the lower query block).  Outputs: X [heads, nQB, 2], the angle           */
/* [heads, nQB] and the order [heads, nQB] (order[h][s] = query block).     */
/* ------------------------------------------------------------------------- */
typedef struct {
    double a;
    int32_t r;
} angled_t;

static int by_angle_then_row(const void* x, const void* y) {
    const angled_t* p = (const angled_t*)x;
    const angled_t* q = (const angled_t*)y;
    if (p->a < q->a) return -1;
    if (p->a > q->a) return 1;
    return (p->r > q->r) - (p->r < q->r);
}

static void gram_schmidt2(double* X, int32_t n) {
    double n0 = 0.0;
    for (int32_t r = 0; r < n; ++r) n0 += X[2 * r] * X[2 * r];
    n0 = sqrt(n0);
    for (int32_t r = 0; r < n; ++r) X[2 * r] /= n0;
    double d = 0.0;
    for (int32_t r = 0; r < n; ++r) d += X[2 * r] * X[2 * r + 1];
    for (int32_t r = 0; r < n; ++r) X[2 * r + 1] -= d * X[2 * r];
    double n1 = 0.0;
    for (int32_t r = 0; r < n; ++r) n1 += X[2 * r + 1] * X[2 * r + 1];
    n1 = sqrt(n1);
    for (int32_t r = 0; r < n; ++r) X[2 * r + 1] /= n1;
}

void oracle_spectral_order(const int32_t* kv_idx, const int32_t* kv_cnt, int32_t max_kv,
                           int64_t heads, int32_t nQB, int32_t nKB, int32_t iters,
                           const double* x0, double* x_out, double* angle, int32_t* order) {
    double* mu = (double*)malloc(sizeof(double) * (size_t)nKB);
    double* Z = (double*)malloc(sizeof(double) * 2 * (size_t)nKB);
    double* X = (double*)malloc(sizeof(double) * 2 * (size_t)nQB);
    angled_t* srt = (angled_t*)malloc(sizeof(angled_t) * (size_t)nQB);
    for (int64_t h = 0; h < heads; ++h) {
        const int32_t* idx = kv_idx + h * nQB * (int64_t)max_kv;
        const int32_t* cnt = kv_cnt + h * nQB;
        for (int32_t c = 0; c < nKB; ++c) mu[c] = 0.0;
        for (int32_t r = 0; r < nQB; ++r)
            for (int32_t e = 0; e < cnt[r]; ++e) mu[idx[r * (int64_t)max_kv + e]] += 1.0;
        for (int32_t c = 0; c < nKB; ++c) mu[c] /= (double)nQB;
        memcpy(X, x0 + h * 2 * (int64_t)nQB, sizeof(double) * 2 * (size_t)nQB);
        gram_schmidt2(X, nQB);
        for (int32_t it = 0; it < iters; ++it) {
            double s0 = 0.0, s1 = 0.0; /* 1^T X */
            for (int32_t r = 0; r < nQB; ++r) {
                s0 += X[2 * r];
                s1 += X[2 * r + 1];
            }
            for (int32_t c = 0; c < 2 * nKB; ++c) Z[c] = 0.0;
            for (int32_t r = 0; r < nQB; ++r)
                for (int32_t e = 0; e < cnt[r]; ++e) {
                    const int32_t c = idx[r * (int64_t)max_kv + e];
                    Z[2 * c] += X[2 * r];
                    Z[2 * c + 1] += X[2 * r + 1];
                }
            double m0 = 0.0, m1 = 0.0; /* mu^T Z (after centering) */
            for (int32_t c = 0; c < nKB; ++c) {
                Z[2 * c] -= mu[c] * s0;
                Z[2 * c + 1] -= mu[c] * s1;
                m0 += mu[c] * Z[2 * c];
                m1 += mu[c] * Z[2 * c + 1];
            }
            for (int32_t r = 0; r < nQB; ++r) {
                double y0 = 0.0, y1 = 0.0;
                for (int32_t e = 0; e < cnt[r]; ++e) {
                    const int32_t c = idx[r * (int64_t)max_kv + e];
                    y0 += Z[2 * c];
                    y1 += Z[2 * c + 1];
                }
                X[2 * r] = y0 - m0;
                X[2 * r + 1] = y1 - m1;
            }
            gram_schmidt2(X, nQB);
        }
        for (int32_t r = 0; r < nQB; ++r) {
            srt[r].a = atan2(X[2 * r + 1], X[2 * r]);
            srt[r].r = r;
            angle[h * nQB + r] = srt[r].a;
        }
        memcpy(x_out + h * 2 * (int64_t)nQB, X, sizeof(double) * 2 * (size_t)nQB);
        qsort(srt, (size_t)nQB, sizeof(angled_t), by_angle_then_row);
        for (int32_t s = 0; s < nQB; ++s) order[h * nQB + s] = srt[s].r;
    }
    free(srt);
    free(X);
    free(Z);
    free(mu);
}

/* ------------------------------------------------------------------------- */
/* Block scores from block means.                                            */
/* MC-Sparse, "The MC-Sparse Architecture" (block-sparse attention keeps the */
/* KV blocks with the highest mean-pooled similarity) and InstaGen section   */
/* 3.3 / Algorithm 1 step 2 (centroid score s_gc = exp(q_g . k_c / sqrt d)   */
/* with q_g, k_c the means of a query group and a key cluster).  A group /   */
/* cluster is a 128-token block of the gathered order (q_map / kv_map, or    */
/* the identity).  mode 0: mean(Q_u) . mean(K_v) * scale;  mode 1:           */
/* exp(mean(Q_u) . mean(K_v) * scale).  scale <= 0 selects 1/sqrt(D).        */
/* Output scores [B*H*nQB, nKB] in fp64.                                      */
/* ------------------------------------------------------------------------- */
void oracle_block_scores(const uint16_t* q, const uint16_t* k, int32_t B, int32_t H, int32_t N,
                         int32_t D, const int32_t* q_map, const int32_t* kv_map, double scale,
                         int32_t mode, double* scores) {
    const int32_t nb = N / ORACLE_BLOCK;
    if (scale <= 0.0) scale = 1.0 / sqrt((double)D);
    const int64_t BH = (int64_t)B * H;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < BH; ++bh) {
        double* qm = (double*)malloc(sizeof(double) * (size_t)nb * D);
        double* km = (double*)malloc(sizeof(double) * (size_t)nb * D);
        for (int32_t b = 0; b < nb; ++b) {
            for (int32_t d = 0; d < D; ++d) {
                double sq = 0.0, sk = 0.0;
                for (int32_t t = 0; t < ORACLE_BLOCK; ++t) {
                    const int32_t p = b * ORACLE_BLOCK + t;
                    const int32_t i = q_map ? q_map[bh * N + p] : p;
                    const int32_t j = kv_map ? kv_map[bh * N + p] : p;
                    sq += bf16_to_double(q[(bh * N + i) * D + d]);
                    sk += bf16_to_double(k[(bh * N + j) * D + d]);
                }
                qm[(int64_t)b * D + d] = sq / ORACLE_BLOCK;
                km[(int64_t)b * D + d] = sk / ORACLE_BLOCK;
            }
        }
        for (int32_t u = 0; u < nb; ++u)
            for (int32_t v = 0; v < nb; ++v) {
                double dot = 0.0;
                for (int32_t d = 0; d < D; ++d) dot += qm[(int64_t)u * D + d] * km[(int64_t)v * D + d];
                const double s = dot * scale;
                scores[(bh * nb + u) * (int64_t)nb + v] = mode == 1 ? exp(s) : s;
            }
        free(km);
        free(qm);
    }
}

/* ------------------------------------------------------------------------- */
/* CRM rows, ScalingAttention section 7.2: each row is an array of uint32     */
/* words, bit i of word w set when KV block 32w + i is kept.  mode 0: mask    */
/* (nonzero keeps), mode 1: threshold map (T <= p in fp32 keeps).             */
/* ------------------------------------------------------------------------- */
void oracle_crm_rows(int32_t mode, const void* src, int64_t rows, int32_t nKB, float p,
                     uint32_t* words, int32_t n_words) {
    for (int64_t r = 0; r < rows; ++r) {
        for (int32_t w = 0; w < n_words; ++w) words[r * n_words + w] = 0u;
        for (int32_t kb = 0; kb < nKB; ++kb) {
            int keep;
            if (mode == 0) keep = ((const uint8_t*)src)[r * nKB + kb] != 0;
            else keep = ((const float*)src)[r * nKB + kb] <= p;
            if (keep) words[r * n_words + kb / 32] |= 1u << (kb % 32);
        }
    }
}

/* ------------------------------------------------------------------------- */
/* Resolution upscaling of a threshold map, ScalingAttention section 7.1     */
/* eq. (7): R_target(u, v) = ceil(Phi(R_base, u / s_h, v / s_w)) with Phi    */
/* bilinear interpolation and s = target / base size.  On a 0/1 mask the     */
/* ceiling keeps a target block when any base block with a nonzero bilinear  */
/* weight is active; applied to every mask M_p = I(T <= p) at once, that is  */
/* the minimum of T over those base blocks.  Base coordinate of target index */
/* u is x = u * Ub / Ut; its neighbours are floor(x) and floor(x) + 1        */
/* (clamped to the last index), the second with weight x - floor(x), which   */
/* is nonzero exactly when u * Ub is not a multiple of Ut (integer test).    */
/* ------------------------------------------------------------------------- */
void oracle_upscale_threshold(const float* T, int64_t heads, int32_t Ub, int32_t Vb,
                              int32_t Ut, int32_t Vt, float* out) {
    for (int64_t h = 0; h < heads; ++h)
        for (int32_t u = 0; u < Ut; ++u) {
            const int64_t xu = (int64_t)u * Ub;
            const int32_t i0 = (int32_t)(xu / Ut);
            const int32_t i1 = (xu % Ut != 0 && i0 + 1 < Ub) ? i0 + 1 : i0;
            for (int32_t v = 0; v < Vt; ++v) {
                const int64_t yv = (int64_t)v * Vb;
                const int32_t j0 = (int32_t)(yv / Vt);
                const int32_t j1 = (yv % Vt != 0 && j0 + 1 < Vb) ? j0 + 1 : j0;
                const float* b = T + h * (int64_t)Ub * Vb;
                float m = b[(int64_t)i0 * Vb + j0];
                if (b[(int64_t)i0 * Vb + j1] < m) m = b[(int64_t)i0 * Vb + j1];
                if (b[(int64_t)i1 * Vb + j0] < m) m = b[(int64_t)i1 * Vb + j0];
                if (b[(int64_t)i1 * Vb + j1] < m) m = b[(int64_t)i1 * Vb + j1];
                out[(h * Ut + u) * (int64_t)Vt + v] = m;
            }
        }
}
