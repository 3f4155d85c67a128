// Block-sparse attention forward for sm_103a (tcgen05 + TMEM + TMA).
//
// What it computes (InstaGen, section 3.1 eqs. (1)-(3) and Algorithm 1
// step 14; INTRA, "CQS-Aware Token-Sparse FlashAttention Kernel"): for every
// (head, 128-row query block) the online softmax over the 128-key blocks in
// its list, each block's scores shifted by the block's log-weight, and
// O = P V / l, LSE = ln l + max, written back through the query map.
//
// Work mapping.  One thread block owns one (head, query block) work item;
// blockIdx.x is the execution slot within the head (query block
// row_perm[head][slot]) and blockIdx.y the head, so blocks are issued
// head-major in slot order: the sequential-head, wave-ordered schedule of
// WaveAlign section V.  Short rows (the Scatter and Gather 0 layers, sliding
// windows) run in k_bsa_forward_items instead: one block per SM walks the
// items in the same order (see the comment above that kernel).
//
// Warp roles (8 warps):
//   warp 0      producer: Q once (one TMA tile copy; with q_map the softmax
//               warps gather it), then K_j and V_j of every listed block
//               into a ring of kStages shared-memory slots, one TMA tile
//               copy each.  The list is read 32 entries at a time by the
//               whole warp; every lane waits for a free slot and one lane
//               elected with elect.sync issues the copy, so the warp's
//               control flow stays uniform.
//   warps 6, 7  with kv_map given, warp 0 and these two gather the K/V
//               tiles in turn: each copies the 128 token rows of its tiles
//               with 16-byte cp.async into the swizzled layout, one warp
//               alone being too slow for row-granular copies (INTRA's
//               gather, on the load/store path instead of the tensor-copy
//               unit).
//   warp 1      allocates tensor memory and issues tcgen05.mma in the order
//               QK(0), QK(1), QK(2), then for i = 0..n-1: PV(i), QK(i+3):
//               S_j = Q K_j^T into TMEM score buffer j % 3 (QK runs up to
//               three blocks ahead of the softmax), O += P_i V_i with P read
//               from TMEM.  The whole warp walks this schedule (the waits,
//               the descriptor and TMEM address arithmetic) and one elected
//               lane issues each group of MMAs and its commit: with lane 0
//               alone inside a divergent branch the same schedule ran about
//               5 % slower.  The warp touches no global memory; it waits
//               only for P_i and for data.
//   warps 2..5  softmax: one thread per query row (TMEM lane); with q_map
//               each warp first copies its 32 query rows into the Q tile
//               (cp.async, 16 bytes per lane); reads S_j,
//               updates the running max (log2 domain) and sum, rescales O in
//               TMEM when the max grows by more than 2^8, writes P_j (bf16)
//               over S_j, and runs the epilogue (O / l -> bf16 through the
//               query map, LSE).
//
// The producer loads K/V tiles in exactly the MMA's consumption order
// (K_0, K_1, K_2, then V_i, K_{i+3}), so the ring is a plain FIFO.  Each MMA
// group ends with a single commit, on the empty barrier of the ring slot it
// read; the softmax waits on that same barrier for S_j (slot of K_j) and,
// before touching O, for PV_{j-1} (slot of V_{j-1}).  The next completion of
// such a barrier needs a later P from this softmax, so parity waits on it
// are unambiguous.
//
// Tensor memory (512 columns): S_0, S_1, S_2 = [0,384) in 128-column
// buffers, O = [384, 384+D).
// Shared memory: Q tile + kStages K/V tiles, each tile stored as D/64 boxes
// of 128 rows x 128 bytes with the 128-byte swizzle (canonical K-major
// layout for Q and K, MN-major for V).
//
// Every mbarrier wait is bounded (1 s of wall time); on expiry the status
// word gets BSA_ERR_TIMEOUT, the roles stop, in-flight copies and MMAs are
// drained (again bounded) and tensor memory is freed before exit.  Blocks
// that start, or are waiting, while the status word holds BSA_ERR_TIMEOUT
// give up at once, so a broken launch ends within about a second per wave
// instead of a second per block.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>

#include "bsa_gather0.cuh"
#include "bsa_internal.h"
#include "bsa_math.cuh"
#include "bsa_ptx.cuh"

namespace bsa {
namespace {

using namespace ptx;

constexpr uint64_t kWaitNs = 1000000000ull;  // 1 s per wait
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kDefaultPoly = 0;  // exponentials per 8 on the FMA pipe (see bsa_set_forward_options)
constexpr float kRescaleThreshold = 8.0f;  // blocks that compute their maximum rescale O when it grows by > 2^8
// A block's exponentials are taken against the running maximum without
// computing the block's own maximum; only a block whose exponentials sum
// above 2^64 (or to inf / NaN) is redone with its maximum.  That bound keeps
// P (bf16), the row sum and O (fp32) far from overflow.
constexpr float kSumBound = 18446744073709551616.0f;  // 2^64
constexpr int kProducerWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kFirstSoftmaxWarp = 2;
constexpr int kGatherWarps = 3;  // warp 0 and the two extra producer warps
// Softmax warps: with a token mask (kMask) one per TMEM lane quadrant, each
// thread a whole 128-column row; without, two per quadrant, each warp 16
// rows with four threads per row (the row split, see softmax_block_rows).
constexpr int softmax_warps(bool mask) { return mask ? 4 : 8; }
// Extra producer warps (gathered K/V rows) follow the softmax warps.
constexpr int extra_producer_warp(bool mask) { return kFirstSoftmaxWarp + softmax_warps(mask); }
constexpr int threads_for(bool gather, bool mask) {
    return 32 * (extra_producer_warp(mask) + (gather ? kGatherWarps - 1 : 0));
}
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 384;
constexpr int kSBuf = 3;  // TMEM score buffers

template <int D>
struct Cfg {
    static constexpr int kBoxBytes = 128 * 128;  // 128 rows x 64 bf16
    static constexpr int kBoxes = D / 64;
    static constexpr int kTile = kBoxBytes * kBoxes;
    static constexpr int kStages = D == 128 ? 6 : 12;
    static constexpr int kData = kTile * (1 + kStages);
    static constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, 0, 0);
    static constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, 0, 1);
};

struct Barriers {
    uint64_t full[16];
    uint64_t empty[16];
    uint64_t q_full;
    uint64_t p_full[kSBuf];
    uint64_t mma_done;
    uint32_t tmem_base;
    int32_t abort;
};

struct Params {
    // Tile maps view a [rows, D] bf16 tensor as 3D (64 columns, rows, D/64
    // column halves) so that one copy brings a whole 128-row tile, reading
    // each 2D-byte row in full, and lands it as D/64 swizzled 16 KB boxes.
    CUtensorMap map_q, map_k, map_v;     // 3D box 64 x 128 rows x D/64
    const __nv_bfloat16* q;              // gathered rows are copied with cp.async
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    const int32_t* kv_idx;
    const int32_t* kv_cnt;
    const float* log_w;
    const int32_t* q_map;
    const int32_t* kv_map;
    const int32_t* row_perm;
    const uint32_t* crm;  // CRM rows [rows, crm_words] (the CRM variant only)
    int32_t crm_words;
    __nv_bfloat16* o;
    float* lse;
    int32_t* status;
    int32_t N, nQB, max_kv;
    int32_t H, group;  // query heads per batch entry; query heads per key/value head
    int32_t causal, n_valid, window, sinks;  // token mask (the kMask variant only)
    float scale_log2;
    // packed key tiles and quadrant masks (the kQuad variants)
    int32_t n_kv;      // kv_map entries per key/value head (a multiple of 128)
    const uint8_t* quad_mask;  // [rows, max_kv] quadrant visibility
    // Gather 0 geometry mode: the image as (64, x, y, D/64, head) with boxes
    // of 8 x 16 (queries) and 16 x 8 (key/value bands) pixels, and the
    // Scatter groups as (64, group, t, D/64, head) with boxes of 1 x 128
    g0::Geom geo;
    CUtensorMap map_qi, map_ki, map_vi, map_kg, map_vg;
    CUtensorMap map_qg;  // Scatter layer: queries as (64, group, t, D/64, head), box 1 x 128
};

__device__ __forceinline__ void raise_status(int32_t* status, int32_t code) {
    atomicCAS(status, 0, code);
}

// Bits lo .. hi-1 of a 32-bit word, the bounds clamped to [0, 32].
__device__ __forceinline__ uint32_t run_bits(int32_t lo, int32_t hi) {
    const uint32_t l = (uint32_t)min(max(lo, 0), 32), h = (uint32_t)min(max(hi, 0), 32);
    return h > l ? (uint32_t)(((1ull << h) - 1ull) ^ ((1ull << l) - 1ull)) : 0u;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Two fp32 values in one 64-bit register pair, and the packed f32x2
// arithmetic of sm_100+ (each lane rounds exactly as fmaf / +).
__device__ __forceinline__ uint64_t f2pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2unpack(uint64_t r, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Largest of a row's 128 raw scores.
__device__ __forceinline__ float max128(const uint32_t (&s)[128]) {
    float a = -INFINITY, b = -INFINITY, c = -INFINITY, d = -INFINITY;
#pragma unroll
    for (int i = 0; i < 128; i += 8) {
        a = fmax3(a, __uint_as_float(s[i + 0]), __uint_as_float(s[i + 1]));
        b = fmax3(b, __uint_as_float(s[i + 2]), __uint_as_float(s[i + 3]));
        c = fmax3(c, __uint_as_float(s[i + 4]), __uint_as_float(s[i + 5]));
        d = fmax3(d, __uint_as_float(s[i + 6]), __uint_as_float(s[i + 7]));
    }
    return fmaxf(fmaxf(a, b), fmaxf(c, d));
}

// P = 2^(s * sl2 + bias) for a row's 128 scores, packed as bf16 pairs into
// s[0..63]; returns their fp32 sum.  The affine step and the sum run two
// columns per instruction; columns c with c % 8 < kPoly take the FMA-pipe
// exponential instead of ex2.approx.
template <int kPoly>
__device__ __forceinline__ float exp128(uint32_t (&s)[128], float sl2, float bias) {
    const uint64_t a2 = f2pack(sl2, sl2), b2 = f2pack(bias, bias);
    uint64_t acc0 = f2pack(0.f, 0.f), acc1 = acc0, acc2 = acc0, acc3 = acc0;
#pragma unroll
    for (int c = 0; c < 128; c += 8) {
        float x[8];
#pragma unroll
        for (int i = 0; i < 8; i += 2)
            f2unpack(fma2(f2pack(__uint_as_float(s[c + i]), __uint_as_float(s[c + i + 1])), a2, b2), x[i], x[i + 1]);
        float p[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) p[i] = (i < kPoly) ? exp2_fma(x[i]) : ex2(x[i]);
        acc0 = add2(acc0, f2pack(p[0], p[1]));
        acc1 = add2(acc1, f2pack(p[2], p[3]));
        acc2 = add2(acc2, f2pack(p[4], p[5]));
        acc3 = add2(acc3, f2pack(p[6], p[7]));
#pragma unroll
        for (int i = 0; i < 8; i += 2) s[c / 2 + i / 2] = pack_bf16(p[i], p[i + 1]);
    }
    float lo, hi;
    f2unpack(add2(add2(acc0, acc1), add2(acc2, acc3)), lo, hi);
    return lo + hi;
}

// ---------------------------------------------------------------- row split
// Two softmax warps per TMEM lane quadrant, each over 16 lanes (query rows):
// thread t holds rows t/4 and t/4 + 8 of its warp's 16 ("a" and "b") and,
// of each, the 32 columns 2 (t % 4) + 8 k and 2 (t % 4) + 8 k + 1 (the
// tcgen05 16x256b layout: s[4k], s[4k+1] row a, s[4k+2], s[4k+3] row b).
// The four threads of a row are lanes 4 (t/4) .. 4 (t/4) + 3 of the warp.

// Row maxima of rows a and b over all 128 columns (shuffles within the row's
// four threads).
__device__ __forceinline__ void max_rows(const uint32_t (&s)[64], float& ma, float& mb) {
    float a0 = -INFINITY, a1 = -INFINITY, b0 = -INFINITY, b1 = -INFINITY;
#pragma unroll
    for (int k = 0; k < 16; k += 2) {
        a0 = fmax3(a0, __uint_as_float(s[4 * k + 0]), __uint_as_float(s[4 * k + 1]));
        b0 = fmax3(b0, __uint_as_float(s[4 * k + 2]), __uint_as_float(s[4 * k + 3]));
        a1 = fmax3(a1, __uint_as_float(s[4 * k + 4]), __uint_as_float(s[4 * k + 5]));
        b1 = fmax3(b1, __uint_as_float(s[4 * k + 6]), __uint_as_float(s[4 * k + 7]));
    }
    ma = fmaxf(a0, a1);
    mb = fmaxf(b0, b1);
    ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 1));
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
    ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 2));
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
}

// P = 2^(s * sl2 + bias) for this thread's 64 scores, packed as bf16 pairs
// in the 16x128b layout (s[2k] row a, s[2k+1] row b, column (t % 4) + 4 k);
// la, lb receive this thread's share of the two row sums.
template <int kPoly>
__device__ __forceinline__ void exp_rows(uint32_t (&s)[64], float sl2, float bias_a, float bias_b, float& la,
                                         float& lb) {
    const uint64_t a2 = f2pack(sl2, sl2), ba = f2pack(bias_a, bias_a), bb = f2pack(bias_b, bias_b);
    uint64_t acc_a0 = f2pack(0.f, 0.f), acc_a1 = acc_a0, acc_b0 = acc_a0, acc_b1 = acc_a0;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        float x[4];
        f2unpack(fma2(f2pack(__uint_as_float(s[4 * k]), __uint_as_float(s[4 * k + 1])), a2, ba), x[0], x[1]);
        f2unpack(fma2(f2pack(__uint_as_float(s[4 * k + 2]), __uint_as_float(s[4 * k + 3])), a2, bb), x[2], x[3]);
        float p[4];
        // column of x[i]: 2 (t % 4) + 8 k + (i & 1); its residue mod 8 decides the unit
#pragma unroll
        for (int i = 0; i < 4; ++i) p[i] = kPoly > 0 && (((threadIdx.x & 3) * 2 + (i & 1)) < kPoly) ? exp2_fma(x[i]) : ex2(x[i]);
        if (k & 1) {
            acc_a1 = add2(acc_a1, f2pack(p[0], p[1]));
            acc_b1 = add2(acc_b1, f2pack(p[2], p[3]));
        } else {
            acc_a0 = add2(acc_a0, f2pack(p[0], p[1]));
            acc_b0 = add2(acc_b0, f2pack(p[2], p[3]));
        }
        s[2 * k] = pack_bf16(p[0], p[1]);
        s[2 * k + 1] = pack_bf16(p[2], p[3]);
    }
    float x0, x1;
    f2unpack(add2(acc_a0, acc_a1), x0, x1);
    la = x0 + x1;
    f2unpack(add2(acc_b0, acc_b1), x0, x1);
    lb = x0 + x1;
}

// One block of the online softmax for rows a and b (no token mask, so the
// running maxima are finite after the first block): as softmax_block, the
// block maximum only for the first block or when some row's exponentials
// outgrow 2^64 (summed over this thread's 32 columns; a row's sum is then
// below 2^66).  Returns true (warp-uniform) when O must be rescaled.
template <int kPoly, typename Reload>
__device__ __forceinline__ bool softmax_block_rows(uint32_t (&s)[64], int32_t j, float sl2, float lw2, float (&m)[2],
                                                   float (&l)[2], float (&alpha)[2], Reload&& reload) {
    alpha[0] = alpha[1] = 1.0f;
    float la, lb;
    if (j > 0) {
        exp_rows<kPoly>(s, sl2, lw2 - m[0], lw2 - m[1], la, lb);
        if (!__any_sync(0xffffffffu, !(la <= kSumBound) || !(lb <= kSumBound))) {
            l[0] += la;
            l[1] += lb;
            return false;
        }
        reload();
    }
    float ma, mb;
    max_rows(s, ma, mb);
    const float mt[2] = {ma * sl2 + lw2, mb * sl2 + lw2};
    bool rescale = false;
    if (j == 0) {
        m[0] = mt[0];
        m[1] = mt[1];
    } else {
        rescale = __any_sync(0xffffffffu, mt[0] > m[0] + kRescaleThreshold || mt[1] > m[1] + kRescaleThreshold);
        if (rescale) {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const float m_new = fmaxf(m[i], mt[i]);
                alpha[i] = ex2(m[i] - m_new);
                l[i] *= alpha[i];
                m[i] = m_new;
            }
        }
    }
    exp_rows<kPoly>(s, sl2, lw2 - m[0], lw2 - m[1], la, lb);
    l[0] += la;
    l[1] += lb;
    return rescale;
}

// P = 0 for this warp's 16 rows of a score buffer (the 16x128b layout the
// softmax writes P in), for a block that no row of its quadrant sees.
__device__ __forceinline__ void store_p_zero(uint32_t taddr) {
    uint32_t z[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) z[c] = 0u;
    tmem_st16x128_x16(taddr, z);
    tmem_wait_st();
}

// A row's sum over its four threads (the same value in each).
__device__ __forceinline__ float row_sum4(float x) {
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    return x + __shfl_xor_sync(0xffffffffu, x, 2);
}

// Transpose of a 4 x 4 block of words held by the four threads of a row
// (thread c of the row holds x[0..3]; afterwards x[j] is thread j's former
// x[c]), by two butterfly exchanges.
__device__ __forceinline__ void transpose4(uint32_t x[4], int c) {
#pragma unroll
    for (int m = 2; m >= 1; m >>= 1) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (j & m) continue;
            const bool hi = (c & m) != 0;
            const uint32_t recv = __shfl_xor_sync(0xffffffffu, hi ? x[j] : x[j | m], m);
            if (hi) x[j] = recv;
            else x[j | m] = recv;
        }
    }
}

// O rows a and b (16x256b layout: o[4k..4k+3] = row a's columns 8k + 2c,
// 8k + 2c + 1, then row b's, c = thread % 4) divided by their sums, as bf16
// pairs: pk[k] row a's, pk[D/8 + k] row b's.
template <int D>
__device__ __forceinline__ void pack_o_pairs(const uint32_t* o, float inv_a, float inv_b, uint32_t* pk) {
#pragma unroll
    for (int k = 0; k < D / 8; ++k) {
        pk[k] = pack_bf16(__uint_as_float(o[4 * k]) * inv_a, __uint_as_float(o[4 * k + 1]) * inv_a);
        pk[D / 8 + k] = pack_bf16(__uint_as_float(o[4 * k + 2]) * inv_b, __uint_as_float(o[4 * k + 3]) * inv_b);
    }
}

// Stores packed O rows.  Within each group of four words the row's four
// threads exchange words, so that thread c then holds 8 consecutive columns,
// 8 (4g + c) .., and writes them with one 16-byte store: the four threads of
// a row write 64 bytes of it per store instead of 16.  Every lane takes part
// in the exchanges; a null row pointer skips that row's stores.
template <int D>
__device__ __forceinline__ void store_packed_pairs(const uint32_t* pk, __nv_bfloat16* row_a, __nv_bfloat16* row_b) {
    const int c = threadIdx.x & 3;
#pragma unroll
    for (int g = 0; g < D / 32; ++g) {
        uint32_t xa[4], xb[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            xa[j] = pk[4 * g + j];
            xb[j] = pk[D / 8 + 4 * g + j];
        }
        transpose4(xa, c);
        transpose4(xb, c);
        if (row_a) *reinterpret_cast<uint4*>(row_a + 8 * (4 * g + c)) = make_uint4(xa[0], xa[1], xa[2], xa[3]);
        if (row_b) *reinterpret_cast<uint4*>(row_b + 8 * (4 * g + c)) = make_uint4(xb[0], xb[1], xb[2], xb[3]);
    }
}

template <int D>
__device__ __forceinline__ void store_o_pairs(const uint32_t* o, float inv_a, float inv_b, __nv_bfloat16* row_a,
                                              __nv_bfloat16* row_b) {
    uint32_t pk[D / 4];
    pack_o_pairs<D>(o, inv_a, inv_b, pk);
    store_packed_pairs<D>(pk, row_a, row_b);
}

// O columns of rows a and b out of tensor memory (16x256b layout, D / 4 per
// row per thread), multiplied by per-row factors, back in.
template <int D>
__device__ __forceinline__ void scale_o_rows(uint32_t taddr, float fa, float fb) {
    uint32_t o[D / 2];
    if constexpr (D == 128) tmem_ld16x256_x16(taddr, o);
    else tmem_ld16x256_x8(taddr, o);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < D / 2; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * (((i >> 1) & 1) ? fb : fa));
    if constexpr (D == 128) tmem_st16x256_x16(taddr, o);
    else tmem_st16x256_x8(taddr, o);
}

// Normalised O of rows a and b (bf16) to their output rows: this thread's
// column pairs 2 (t % 4) + 8 k.
template <int D>
__device__ __forceinline__ void store_o_rows(uint32_t taddr, float inv_a, float inv_b, __nv_bfloat16* row_a,
                                             __nv_bfloat16* row_b) {
    uint32_t o[D / 2];
    if constexpr (D == 128) tmem_ld16x256_x16(taddr, o);
    else tmem_ld16x256_x8(taddr, o);
    tmem_wait_ld();
    store_o_pairs<D>(o, inv_a, inv_b, row_a, row_b);
}

// One block of the online softmax for this thread's row.  On entry s holds
// the row's 128 raw scores of block j (dropped keys -inf); on exit s[0..63]
// holds P_j as bf16 pairs.  m is the running maximum (log2 domain, scale and
// log-weight applied), l the running sum.  The first block of a row, and a
// block while the row has seen no key (m = -inf, masked rows), compute the
// block maximum and rescale when it grows by more than 2^8; other blocks take
// their exponentials against m directly and fall back to the maximum only if
// their sum leaves (0, 2^64] as a whole (reload() then refills s with the raw
// scores).  Returns true when O must be multiplied by alpha before P_j V_j is
// added; the decision is warp-uniform (the rescale's tensor-memory accesses
// are warp-wide).
template <int kPoly, bool kMask, typename Reload>
__device__ __forceinline__ bool softmax_block(uint32_t (&s)[128], int32_t j, float sl2, float lw2, float& m,
                                              float& l, float& alpha, Reload&& reload) {
    alpha = 1.0f;
    if (j > 0 && !__any_sync(0xffffffffu, m == -INFINITY)) {
        const float l_blk = exp128<kPoly>(s, sl2, lw2 - m);
        if (!__any_sync(0xffffffffu, !(l_blk <= kSumBound))) {
            l += l_blk;
            return false;
        }
        reload();  // rare: some row's block outgrew the running maximum by ~2^57
    }
    const float mt = max128(s) * sl2 + lw2;
    bool rescale = false;
    if (j == 0) {
        m = mt;
    } else {
        rescale = __any_sync(0xffffffffu, mt > m + kRescaleThreshold);
        if (rescale) {
            const float m_new = fmaxf(m, mt);
            // a row with every key so far dropped has l = 0 and O = 0
            alpha = (kMask && m == -INFINITY) ? 0.0f : ex2(m - m_new);
            l *= alpha;
            m = m_new;
        }
    }
    // a row with every key so far dropped keeps m = -inf: its exponentials
    // are all 0 (avoid -inf - -inf)
    const float bias = lw2 - ((kMask && m == -INFINITY) ? 0.0f : m);
    l += exp128<kPoly>(s, sl2, bias);
    return rescale;
}

__device__ __forceinline__ bool aborted(const Barriers* b) {
    return *reinterpret_cast<const volatile int32_t*>(&b->abort) != 0;
}
__device__ __forceinline__ void set_abort(Barriers* b, int32_t* status) {
    *reinterpret_cast<volatile int32_t*>(&b->abort) = 1;
    raise_status(status, BSA_ERR_TIMEOUT);
}

// One K/V tile gathered through a map, copied 16 bytes per lane into the
// 128-byte-swizzled box layout that a TMA tile copy would write (chunk c of
// row r lands at chunk c ^ (r mod 8) of its 128-byte line).  Lane l holds
// the tokens of rows l, l + 32, l + 64, l + 96 in tok[0..3].  Lanes covering
// one row copy consecutive 16-byte chunks of it, so every warp-wide copy
// reads whole 128-byte lines.
template <int D>
__device__ __forceinline__ void copy_tile(uint32_t dst, const __nv_bfloat16* base, int64_t bh,
                                          int32_t N, int lane, const int32_t (&tok)[4]) {
    using C = Cfg<D>;
    constexpr int kLanesPerRow = D / 8;              // 16-byte chunks per token row
    constexpr int kRowsPerCopy = 32 / kLanesPerRow;  // rows covered by one warp-wide copy
    const int sub = lane / kLanesPerRow, chunk = lane % kLanesPerRow;
    const int box = chunk >> 3, c = chunk & 7;
    const uint32_t d0 = dst + box * C::kBoxBytes + ((uint32_t)c << 4);
    const __nv_bfloat16* s0 = base + bh * N * D + box * 64 + c * 8;
    // rows 32 j .. 32 j + 31 take their tokens from tok[j]; the inner loop is
    // kept rolled so that the producer's code stays small next to the softmax
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll 2
        for (int k = 0; k < 32 / kRowsPerCopy; ++k) {
            const int rl = k * kRowsPerCopy + sub;  // row within this group of 32
            const int r = 32 * j + rl;
            const int32_t t = __shfl_sync(0xffffffffu, tok[j], rl);
            cp_async16((d0 + r * 128) ^ ((uint32_t)(r & 7) << 4), s0 + (int64_t)t * D);
        }
    }
}

// Rows 32 g .. 32 g + 31 of a tile gathered through a map (lane l holds the
// token of row 32 g + l), copied like copy_tile.  The softmax warps load the
// query tile this way, each warp the 32 rows it owns.
template <int D>
__device__ __forceinline__ void copy_rows32(uint32_t dst, const __nv_bfloat16* base, int64_t bh,
                                            int32_t N, int g, int lane, int32_t tok) {
    using C = Cfg<D>;
    constexpr int kLanesPerRow = D / 8;
    constexpr int kRowsPerCopy = 32 / kLanesPerRow;
    const int sub = lane / kLanesPerRow, chunk = lane % kLanesPerRow;
    const int box = chunk >> 3, c = chunk & 7;
    const uint32_t d0 = dst + box * C::kBoxBytes + ((uint32_t)c << 4);
    const __nv_bfloat16* s0 = base + bh * N * D + box * 64 + c * 8;
#pragma unroll
    for (int k = 0; k < 32 / kRowsPerCopy; ++k) {
        const int rl = k * kRowsPerCopy + sub;
        const int r = 32 * g + rl;
        const int32_t t = __shfl_sync(0xffffffffu, tok, rl);
        cp_async16((d0 + r * 128) ^ ((uint32_t)(r & 7) << 4), s0 + (int64_t)t * D);
    }
}

// Positions in the K/V load order K_0, K_1, K_2, then V_i, K_{i+3} (i < n):
// K_j sits at j for j < 3 and at 2j - 2 after that (right behind V_{j-3});
// V_i sits behind the min(n, 3) leading K tiles, the i earlier V tiles and
// the min(i, n - 3) K tiles that follow them.
__device__ __forceinline__ int32_t ring_pos_k(int32_t j) { return j < kSBuf ? j : 2 * j - 2; }
__device__ __forceinline__ int32_t ring_pos_v(int32_t i, int32_t n) {
    const int32_t lead = n < kSBuf ? n : kSBuf;
    const int32_t mid = n - kSBuf > 0 ? (i < n - kSBuf ? i : n - kSBuf) : 0;
    return lead + i + mid;
}

// Next set bit of a CRM row (ScalingAttention section 7.3, Algorithm 2:
// ADVANCE to the next nonzero word, INDEX by count-trailing-zeros, NEXT by
// clearing the lowest set bit).  Warp-uniform.
struct CrmIter {
    const uint32_t* words;
    int32_t n_words, w;
    uint32_t val;
    __device__ __forceinline__ int32_t next() {
        while (val == 0u && w + 1 < n_words) val = words[++w];
        if (val == 0u) return -1;  // exhausted (cannot happen for a consistent count)
        const int32_t bit = __ffs(val) - 1;
        val &= val - 1u;
        return 32 * w + bit;
    }
};

// Geometry mode: the query tile qb of head bh, and key/value tile kb of
// key/value head bh_kv, each as one TMA box (Scatter group tile, pair of
// image patches, window band, or 128 consecutive text tokens).
__device__ __forceinline__ void geo_load_q(const Params& P, uint32_t dst, uint32_t bar, int64_t bh, int32_t qb) {
    if (P.geo.scatter) {
        // 128 queries of one Scatter group at stride R
        tma_load_5d(dst, &P.map_qg, 0, qb / P.geo.G, 128 * (qb % P.geo.G), 0, (int32_t)bh, bar);
    } else if (qb >= P.geo.nT) {
        // two vertically adjacent 8 x 8 patches: 16 image rows x 8 columns
        const int32_t pq = qb - P.geo.nT;
        tma_load_5d(dst, &P.map_qi, 0, 8 * (pq % P.geo.pw), 16 * (pq / P.geo.pw), 0, (int32_t)bh, bar);
    } else {
        tma_load_3d(dst, &P.map_q, 0, (int32_t)(bh * P.N) + qb * 128, 0, bar);
    }
}
__device__ __forceinline__ void geo_load_kv(const Params& P, uint32_t dst, uint32_t bar, bool is_v, int64_t bh_kv,
                                            int32_t kb) {
    if (kb >= P.geo.nT) {
        const int32_t pk = kb - P.geo.nT;
        if (pk < 4 * P.geo.P) {
            // a window band: 8 image rows x 16 columns
            int32_t c0;
            const int32_t y0 = g0::band_top(P.geo, pk / 4, pk % 4, c0);
            tma_load_5d(dst, is_v ? &P.map_vi : &P.map_ki, 0, c0, y0, 0, (int32_t)bh_kv, bar);
        } else {
            // 128 tokens of one Scatter group
            const int32_t v = pk - 4 * P.geo.P;
            tma_load_5d(dst, is_v ? &P.map_vg : &P.map_kg, 0, v / P.geo.G, 128 * (v % P.geo.G), 0, (int32_t)bh_kv,
                        bar);
        }
    } else {
        tma_load_3d(dst, is_v ? &P.map_v : &P.map_k, 0, (int32_t)(bh_kv * P.N) + kb * 128, 0, bar);
    }
}

template <int D, int kPoly, bool kCrm, bool kGather, bool kMask, bool kGeom, bool kQuad>
__global__ void __launch_bounds__(threads_for(kGather, kMask), 1) k_bsa_forward(const __grid_constant__ Params P) {
    static_assert(!(kCrm && kMask), "the token mask reads block indices from the lists");
    static_assert(!kGeom || (!kGather && !kCrm), "the geometry mode loads tiles by TMA boxes");
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s_q = smem_u32(smem);
    const uint32_t s_ring = s_q + C::kTile;
    Barriers* bars = reinterpret_cast<Barriers*>(smem + C::kData);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t bh = blockIdx.y;
    // key/value head of this query head: b * H_kv + h / group (grouped heads)
    const int64_t bh_kv = (bh / P.H) * (P.H / P.group) + (bh % P.H) / P.group;
    const int32_t N = P.N, nQB = P.nQB, max_kv = P.max_kv;
    // key/value tiles: blocks of the sequence, or 128-entry groups of kv_map
    const int32_t nKB = (kGeom || kGather) ? P.n_kv / 128 : nQB;

    // A block of this launch (or an unread earlier one) timed out: abandon.
    if (*reinterpret_cast<const volatile int32_t*>(P.status) == BSA_ERR_TIMEOUT) return;

    int32_t qb = blockIdx.x;
    if (P.row_perm != nullptr) {
        qb = P.row_perm[bh * nQB + blockIdx.x];
        if (qb < 0 || qb >= nQB) {
            if (threadIdx.x == 0) raise_status(P.status, BSA_ERR_BOUNDS);
            return;
        }
    }
    const int64_t row = bh * nQB + qb;
    int32_t n;
    const int32_t* list = nullptr;
    const uint32_t* crm_row = nullptr;
    if constexpr (kCrm) {
        // count = popcount of the row's words (every warp computes it)
        crm_row = P.crm + row * P.crm_words;
        int32_t c = 0;
        for (int32_t w = lane; w < P.crm_words; w += 32) c += __popc(crm_row[w]);
        n = __reduce_add_sync(0xffffffffu, c);
    } else {
        n = P.kv_cnt[row];
        if (n > max_kv) {
            if (threadIdx.x == 0) raise_status(P.status, BSA_ERR_OVERFLOW);
            n = max_kv;
        }
        if (n < 0) {
            if (threadIdx.x == 0) raise_status(P.status, BSA_ERR_BOUNDS);
            n = 0;
        }
        list = P.kv_idx + row * max_kv;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            // tile loads: one arrive.expect_tx; gathered rows: one cp.async
            // arrival per lane of the warp that copied the tile
            mbar_init(smem_u32(&bars->full[s]), kGather ? 32 : 1);
            mbar_init(smem_u32(&bars->empty[s]), 1);
        }
        // Q by one TMA tile copy, or gathered by the 128 softmax threads
        mbar_init(smem_u32(&bars->q_full), P.q_map ? 128 : 1);
        for (int s = 0; s < kSBuf; ++s) mbar_init(smem_u32(&bars->p_full[s]), 32 * softmax_warps(kMask));
        mbar_init(smem_u32(&bars->mma_done), 1);
        bars->abort = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(&bars->tmem_base), kTmemCols);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        if constexpr (!kGather) {
            prefetch_tensormap(&P.map_k);
            prefetch_tensormap(&P.map_v);
        }
        if constexpr (kGeom) {
            prefetch_tensormap(&P.map_ki);
            prefetch_tensormap(&P.map_vi);
            if (P.geo.nt > 0 || P.geo.scatter) {
                prefetch_tensormap(&P.map_kg);
                prefetch_tensormap(&P.map_vg);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    constexpr int kExtraProducerWarp = extra_producer_warp(kMask);
    if (warp == kProducerWarp || warp >= kExtraProducerWarp) {
        // ------------------------------------------------------------ producers
        // Tile loads: warp 0 alone (one TMA copy per tile).  Gathered K/V
        // (kv_map given): warps 0, 6, 7 take the tiles in turn and copy each
        // with cp.async, because a single issuing warp cannot keep up with
        // row-granular copies.  Every producer warp walks the whole list, so
        // each knows every tile's ring slot and phase.
        const int g = warp == kProducerWarp ? 0 : warp - kExtraProducerWarp + 1;
        constexpr int n_prod = kGather ? kGatherWarps : 1;
        if (g < n_prod) {
            int32_t issued = 0;
            if (g == 0 && P.q_map == nullptr && lane == 0) {  // gathered Q: the softmax warps
                mbar_arrive_expect_tx(smem_u32(&bars->q_full), C::kTile);
                if constexpr (kGeom) geo_load_q(P, s_q, smem_u32(&bars->q_full), bh, qb);
                else tma_load_3d(s_q, &P.map_q, 0, (int32_t)(bh * N) + qb * 128, 0, smem_u32(&bars->q_full));
            }
            // Load order = MMA consumption order: K_0, K_1, K_2, then V_i, K_{i+3}.
            // The list is read 32 entries at a time with one coalesced load and
            // broadcast by shuffles.
            int32_t chunk_base = -64, kb_lane = 0;
            auto block_kb = [&](int32_t e) -> int32_t {
                if (e - chunk_base >= 32 || e < chunk_base) {
                    chunk_base = e & ~31;
                    kb_lane = chunk_base + lane < n ? list[chunk_base + lane] : 0;
                    if (kb_lane < 0 || kb_lane >= nKB) {
                        raise_status(P.status, BSA_ERR_BOUNDS);
                        kb_lane = 0;  // keeps the pipeline in step; this row's result is unspecified
                    }
                }
                return __shfl_sync(0xffffffffu, kb_lane, e - chunk_base);
            };
            CrmIter it_k{crm_row, P.crm_words, -1, 0u}, it_v{crm_row, P.crm_words, -1, 0u};
            // Tile t of the load sequence is K_t for t < min(n, 3); then V_i at
            // 3 + 2i and K_{i+3} at 3 + 2i + 1 while i + 3 < n; then the
            // remaining V tiles.  K blocks are fetched in increasing order
            // (lookahead 3) and V blocks trail; both read the list through the
            // same 32-entry window, refetched when a block falls outside it.
            const int32_t lead = n < kSBuf ? n : kSBuf;
            const int32_t inter = 2 * (n - lead);  // interleaved V/K positions
            auto tile_is_v = [&](int32_t t) -> bool {
                return t >= lead && (t - lead >= inter || ((t - lead) & 1) == 0);
            };
            // Block of tile t.  Called once per tile in increasing t: the CRM
            // iterators (one per stream) advance one set bit per call.
            auto tile_kb = [&](int32_t t) -> int32_t {
                int32_t e;
                const bool is_v = tile_is_v(t);
                if (t < lead) e = t;
                else if (t - lead < inter) e = ((t - lead) >> 1) + (is_v ? 0 : kSBuf);
                else e = (n - lead) + (t - lead - inter);
                int32_t kb;
                if constexpr (kCrm) {
                    kb = is_v ? it_v.next() : it_k.next();
                    if (kb < 0 || kb >= nKB) {
                        if (lane == 0) raise_status(P.status, BSA_ERR_BOUNDS);
                        kb = 0;
                    }
                } else {
                    kb = block_kb(e);
                }
                return kb;
            };
            // Blocks of tiles t .. t + n_prod - 1.  With gathered rows a warp
            // copies every n_prod-th tile and reads the tokens of its next
            // tile while copying the current one, so that the map read (which
            // queues behind the row copies on the load/store path) is off the
            // critical path.
            const int32_t n_tiles = 2 * n;
            int32_t kb_q[n_prod];
#pragma unroll
            for (int i = 0; i < n_prod; ++i) kb_q[i] = i < n_tiles ? tile_kb(i) : 0;
            int32_t tok[4] = {0, 0, 0, 0}, tok_next[4] = {0, 0, 0, 0};
            // lane l reads the tokens of rows l, l + 32, l + 64, l + 96
            const int32_t* map_head = P.kv_map + bh_kv * P.n_kv + lane;
            if constexpr (kGather) {
                if (g < n_tiles) {
                    int32_t kb_g = kb_q[0];  // kb_q[g] without a dynamic register index
#pragma unroll
                    for (int i = 1; i < n_prod; ++i) kb_g = i == g ? kb_q[i] : kb_g;
                    const int32_t* mrow = map_head + (int64_t)kb_g * 128;
#pragma unroll
                    for (int j = 0; j < 4; ++j) tok[j] = mrow[32 * j];
                }
            }
            for (int32_t t = 0; t < n_tiles; ++t) {
                const int32_t kb = kb_q[0];
                const bool is_v = tile_is_v(t);
#pragma unroll
                for (int i = 0; i + 1 < n_prod; ++i) kb_q[i] = kb_q[i + 1];
                kb_q[n_prod - 1] = t + n_prod < n_tiles ? tile_kb(t + n_prod) : 0;
                if (t % n_prod != g) {  // another warp's tile
                    issued = t + 1;
                    continue;
                }
                if constexpr (kGather) {
                    if (t + n_prod < n_tiles) {
                        const int32_t* mrow = map_head + (int64_t)kb_q[n_prod - 1] * 128;
#pragma unroll
                        for (int j = 0; j < 4; ++j) tok_next[j] = mrow[32 * j];
                    }
                }
                const int32_t slot = t % C::kStages;
                const uint32_t phase = (uint32_t)(t / C::kStages) & 1u;
                // every lane waits (warp-uniform control flow); one elected lane issues tile loads
                const bool w = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->empty[slot]), phase ^ 1u, kWaitNs,
                                                                 P.status, BSA_ERR_TIMEOUT));
                if (!w || aborted(bars)) {
                    if (lane == 0) set_abort(bars, P.status);
                    break;
                }
                const uint32_t fb = smem_u32(&bars->full[slot]);
                const uint32_t dst = s_ring + slot * C::kTile;
                if constexpr (kGather) {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (tok[j] < 0 || tok[j] >= N) {
                            raise_status(P.status, BSA_ERR_BOUNDS);
                            tok[j] = 0;
                        }
                    copy_tile<D>(dst, is_v ? P.v : P.k, bh_kv, N, lane, tok);
                    cp_async_arrive_noinc(fb);
#pragma unroll
                    for (int j = 0; j < 4; ++j) tok[j] = tok_next[j];
                } else {
                    // tile load by one elected lane
                    if (elect_one()) {
                        mbar_arrive_expect_tx(fb, C::kTile);
                        if constexpr (kGeom) geo_load_kv(P, dst, fb, is_v, bh_kv, kb);
                        else tma_load_3d(dst, is_v ? &P.map_v : &P.map_k, 0, (int32_t)(bh_kv * N) + kb * 128, 0, fb);
                    }
                    __syncwarp();
                }
                issued = t + 1;
            }
            // Drain: every issued copy must land before the block exits.
            if constexpr (kGather) cp_async_wait_all();
            if (g == 0 && lane == 0) {
                if (!mbar_wait(smem_u32(&bars->q_full), 0, kWaitNs, P.status, BSA_ERR_TIMEOUT)) raise_status(P.status, BSA_ERR_TIMEOUT);
                const int32_t first = issued > C::kStages ? issued - C::kStages : 0;
                for (int32_t i = first; i < issued; ++i)
                    if (!mbar_wait(smem_u32(&bars->full[i % C::kStages]), (uint32_t)(i / C::kStages) & 1u, kWaitNs, P.status, BSA_ERR_TIMEOUT))
                        raise_status(P.status, BSA_ERR_TIMEOUT);
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp walks the schedule, so that its control flow and the
        // descriptor / tensor-memory address arithmetic stay warp-uniform; one
        // elected lane issues each group of MMAs and its commit.
        // descriptors of the K-major Q tile and of ring slot 0; a slot / k-step
        // offset is added to the start-address field (bits 0..13, 16-byte units)
        const uint64_t dq = smem_desc_sw128(s_q, 16, 1024);
        const uint64_t dk = smem_desc_sw128(s_ring, 16, 1024);
        const uint64_t dv = smem_desc_sw128(s_ring, C::kBoxBytes, 1024);
        bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->q_full), 0, kWaitNs, P.status, BSA_ERR_TIMEOUT));
        if (P.q_map != nullptr) fence_proxy_async_smem();  // Q rows written by cp.async
        tc_fence_after();
        int32_t item = 0;  // ring position of the next tile (same order as the producer)
        auto issue_qk = [&](int32_t j) -> bool {
            const int32_t slot = item % C::kStages;
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->full[slot]), (uint32_t)(item / C::kStages) & 1u,
                                                   kWaitNs, P.status, BSA_ERR_TIMEOUT)))
                return false;
            if constexpr (kGather) fence_proxy_async_smem();  // rows written by cp.async
            tc_fence_after();
            const uint64_t ks = dk + (uint64_t)((slot * C::kTile) >> 4);
            const uint32_t d_col = (uint32_t)(j % kSBuf) * 128u;
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = ((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4;
                    mma_ss(tmem + d_col, dq + off, ks + off, C::kIdescQK, kk > 0 ? 1u : 0u);
                }
                mma_commit(smem_u32(&bars->empty[slot]));  // also signals S_j to the softmax
            }
            __syncwarp();
            ++item;
            return true;
        };
        for (int32_t j = 0; ok && j < n && j < kSBuf; ++j) ok = issue_qk(j);
        for (int32_t i = 0; ok && i < n; ++i) {
            // O += P_i V_i once the softmax has written P_i (and rescaled O)
            ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->p_full[i % kSBuf]), (uint32_t)(i / kSBuf) & 1u,
                                                   kWaitNs, P.status, BSA_ERR_TIMEOUT));
            if (!ok) break;
            const int32_t slot = item % C::kStages;
            ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->full[slot]), (uint32_t)(item / C::kStages) & 1u,
                                                   kWaitNs, P.status, BSA_ERR_TIMEOUT));
            if (!ok) break;
            if constexpr (kGather) fence_proxy_async_smem();
            tc_fence_after();
            const uint64_t vs = dv + (uint64_t)((slot * C::kTile) >> 4);
            const uint32_t p_col = (uint32_t)(i % kSBuf) * 128u;
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ts(tmem + kColO, tmem + p_col + kk * 8, vs + (uint64_t)(kk * 2048 >> 4),
                           C::kIdescPV, (i > 0 || kk > 0) ? 1u : 0u);
                mma_commit(smem_u32(&bars->empty[slot]));  // also signals PV_i to the softmax
            }
            __syncwarp();
            ++item;
            // S buffer i % 3 is free again once PV_i (issued above) has read P_i
            if (i + kSBuf < n) ok = issue_qk(i + kSBuf);
        }
        if (!ok && lane == 0) set_abort(bars, P.status);
        // Drain: nothing of ours may still be running when TMEM is freed.
        if (elect_one()) mma_commit(smem_u32(&bars->mma_done));
        __syncwarp();
        if (!mbar_wait(smem_u32(&bars->mma_done), 0, kWaitNs, P.status, BSA_ERR_TIMEOUT) && lane == 0)
            raise_status(P.status, BSA_ERR_TIMEOUT);
        __syncwarp();
    } else if constexpr (!kMask) {
        // ------------------------------------------------ softmax + epilogue (row split)
        // Warp `half` of quadrant qd owns rows 32 qd + 16 half .. + 15; thread
        // t rows ra = .. + t/4 and rb = ra + 8 (see softmax_block_rows).
        const int qd = warp & 3;  // a warp reaches TMEM lanes 32 (warp % 4) .. + 31
        const int half = (warp - kFirstSoftmaxWarp) >> 2;
        const int ra = qd * 32 + half * 16 + (lane >> 2), rb = ra + 8;
        const uint32_t t_base = tmem + ((uint32_t)(qd * 32 + half * 16) << 16);
        int32_t tok[2] = {qb * 128 + ra, qb * 128 + rb};
        bool tok_ok[2] = {true, true};
        if constexpr (kGeom) {
            tok[0] = g0::query_token(P.geo, qb * 128 + ra);
            tok[1] = g0::query_token(P.geo, qb * 128 + rb);
        }
        if (P.q_map != nullptr) {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                tok[i] = P.q_map[bh * N + qb * 128 + (i ? rb : ra)];
                if (tok[i] < 0 || tok[i] >= N) {
                    raise_status(P.status, BSA_ERR_BOUNDS);
                    tok_ok[i] = false;
                }
            }
            // the half-0 warps copy the quadrant's 32 query rows into the Q
            // tile, lane l row 32 qd + l (row 0 stands in for an invalid token;
            // that row's output is not written)
            if (half == 0) {
                int32_t tq = P.q_map[bh * N + qb * 128 + qd * 32 + lane];
                if (tq < 0 || tq >= N) tq = 0;
                copy_rows32<D>(s_q, P.q, bh, N, qd, lane, tq);
                cp_async_arrive_noinc(smem_u32(&bars->q_full));
            }
        }
        const float sl2 = P.scale_log2;
        const float* lw_row = P.log_w ? P.log_w + row * max_kv : nullptr;
        // quadrant visibility of the listed blocks (bit qd of entry j: this
        // warp's rows see block j), 32 entries at a time, lane e entry base + e
        const uint8_t* qm_row = (kQuad && P.quad_mask != nullptr) ? P.quad_mask + row * max_kv : nullptr;
        uint32_t qm_chunk = 0xFu;
        if constexpr (kQuad) qm_chunk = (qm_row != nullptr && lane < n) ? qm_row[lane] : 0xFu;
        float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.0f, 0.0f};  // l: this thread's share of each row
        bool ok = true;
        float lw_next = (lw_row && n > 0) ? lw_row[0] : 0.0f;
        for (int32_t j = 0; j < n; ++j) {
            const float lw2 = lw_next * kLog2e;
            lw_next = (lw_row && j + 1 < n) ? lw_row[j + 1] : 0.0f;
            if (kQuad && j > 0 && (j & 31) == 0)
                qm_chunk = (qm_row != nullptr && j + lane < n) ? qm_row[j + lane] : 0xFu;
            bool hidden = false;  // warp-uniform: no row of this quadrant sees block j
            if constexpr (kQuad) hidden = ((__shfl_sync(0xffffffffu, qm_chunk, j & 31) >> qd) & 1u) == 0u;
            const uint32_t sbuf = (uint32_t)(j % kSBuf) * 128u;
            const int32_t pk = ring_pos_k(j);
            const bool w = mbar_wait(smem_u32(&bars->empty[pk % C::kStages]), (uint32_t)(pk / C::kStages) & 1u, kWaitNs, P.status, BSA_ERR_TIMEOUT);
            if (__any_sync(0xffffffffu, !w || aborted(bars))) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (kQuad && hidden) {
                // P_j = 0 for these rows; m, l and O are unchanged
                store_p_zero(t_base + sbuf);
                tc_fence_before();
                mbar_arrive(smem_u32(&bars->p_full[j % kSBuf]));
                continue;
            }
            uint32_t s[64];
            auto load_s = [&]() {
                tmem_ld16x256_x16(t_base + sbuf, s);
                tmem_wait_ld();
            };
            load_s();
            float alpha[2];
            const bool rescale = softmax_block_rows<kPoly>(s, j, sl2, lw2, m, l, alpha, load_s);
            tmem_st16x128_x16(t_base + sbuf, s);  // P_j over the first 64 columns of S_j
            if (rescale) {
                // O must hold P_0..P_{j-1} V: wait for PV_{j-1}
                const int32_t pv = ring_pos_v(j - 1, n);
                const bool wv = mbar_wait(smem_u32(&bars->empty[pv % C::kStages]), (uint32_t)(pv / C::kStages) & 1u, kWaitNs, P.status, BSA_ERR_TIMEOUT);
                if (__any_sync(0xffffffffu, !wv)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                scale_o_rows<D>(t_base + kColO, alpha[0], alpha[1]);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(smem_u32(&bars->p_full[j % kSBuf]));
        }
        if (!ok) {
            if (lane == 0) set_abort(bars, P.status);
        } else {
            const float l_a = row_sum4(l[0]), l_b = row_sum4(l[1]);
            __nv_bfloat16* row_a = tok_ok[0] ? P.o + (bh * N + tok[0]) * D : nullptr;
            __nv_bfloat16* row_b = tok_ok[1] ? P.o + (bh * N + tok[1]) * D : nullptr;
            const int c = 2 * (lane & 3);
            if (n == 0) {
#pragma unroll
                for (int k = 0; k < D / 8; ++k) {
                    if (row_a) *reinterpret_cast<uint32_t*>(row_a + 8 * k + c) = 0u;
                    if (row_b) *reinterpret_cast<uint32_t*>(row_b + 8 * k + c) = 0u;
                }
                if ((lane & 3) == 0) {
                    if (row_a) P.lse[bh * N + tok[0]] = -INFINITY;
                    if (row_b) P.lse[bh * N + tok[1]] = -INFINITY;
                }
            } else {
                const int32_t pv = ring_pos_v(n - 1, n);
                const bool w = mbar_wait(smem_u32(&bars->empty[pv % C::kStages]), (uint32_t)(pv / C::kStages) & 1u, kWaitNs, P.status, BSA_ERR_TIMEOUT);
                if (__any_sync(0xffffffffu, !w)) {
                    if (lane == 0) set_abort(bars, P.status);
                } else {
                    tc_fence_after();
                    store_o_rows<D>(t_base + kColO, l_a > 0.0f ? 1.0f / l_a : 0.0f, l_b > 0.0f ? 1.0f / l_b : 0.0f,
                                    row_a, row_b);
                    if ((lane & 3) == 0) {
                        if (row_a) P.lse[bh * N + tok[0]] = l_a > 0.0f ? (m[0] + log2f(l_a)) * kLn2 : -INFINITY;
                        if (row_b) P.lse[bh * N + tok[1]] = l_b > 0.0f ? (m[1] + log2f(l_b)) * kLn2 : -INFINITY;
                    }
                }
            }
        }
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        const int qd = warp & 3;                 // TMEM lane quadrant of this warp
        const int r = qd * 32 + lane;            // row within the query tile
        const uint32_t t_lane = tmem + ((uint32_t)(qd * 32) << 16);
        const int32_t p = qb * 128 + r;
        int32_t tok = p;
        bool tok_ok = true;
        if constexpr (kGeom) tok = g0::query_token(P.geo, p);
        if (P.q_map != nullptr) {
            tok = P.q_map[bh * N + p];
            if (tok < 0 || tok >= N) {
                raise_status(P.status, BSA_ERR_BOUNDS);
                tok_ok = false;
            }
            // this warp's 32 query rows into the Q tile (row 0 stands in for
            // an invalid token; that row's output is not written)
            copy_rows32<D>(s_q, P.q, bh, N, qd, lane, tok_ok ? tok : 0);
            cp_async_arrive_noinc(smem_u32(&bars->q_full));
        }
        const float sl2 = P.scale_log2;
        const float* lw_row = P.log_w ? P.log_w + row * max_kv : nullptr;
        // quadrant visibility of the listed blocks: bit qd of entry j says
        // whether this warp's 32 rows see block j at all
        const uint8_t* qm_row = (kQuad && P.quad_mask != nullptr) ? P.quad_mask + row * max_kv : nullptr;
        float m = -INFINITY, l = 0.0f;
        bool ok = true;
        float lw_next = (lw_row && n > 0) ? lw_row[0] : 0.0f;
        // The row's quadrant masks, 32 at a time (lane e holds entry base + e),
        // loaded ahead so that no iteration waits on a global load before it
        // knows whether its warp sees the block.
        uint32_t qm_chunk = 0xFu;
        if constexpr (kQuad) qm_chunk = (qm_row != nullptr && lane < n) ? qm_row[lane] : 0xFu;
        for (int32_t j = 0; j < n; ++j) {
            const float lw2 = lw_next * kLog2e;
            lw_next = (lw_row && j + 1 < n) ? lw_row[j + 1] : 0.0f;
            if (kQuad && j > 0 && (j & 31) == 0)
                qm_chunk = (qm_row != nullptr && j + lane < n) ? qm_row[j + lane] : 0xFu;
            const uint32_t sbuf = (uint32_t)(j % kSBuf) * 128u;
            // Token mask: the key tokens of block j (column c of the tile is key
            // 128 kb + c, or kv_map of it), read before the wait for S_j.  A
            // row needs per-element masking only if some key of the block may
            // be dropped for it (a conservative test on the block's key range).
            int32_t kt[4] = {0, 0, 0, 0};  // with kv_map: keys of columns lane + 32 m
            int32_t kbase = 0;
            bool need_mask = false;
            uint32_t vis_w[4] = {~0u, ~0u, ~0u, ~0u};
            bool hidden = false;  // warp-uniform: no row of this warp sees block j
            if constexpr (kQuad) hidden = ((__shfl_sync(0xffffffffu, qm_chunk, j & 31) >> qd) & 1u) == 0u;
            if (kMask && !kGeom && !hidden) {
                int32_t kb = list[j];
                kb = (kb < 0 || kb >= nKB) ? 0 : kb;  // flagged by the producer
                int32_t kmin, kmax;
                if (P.kv_map != nullptr) {
                    const int32_t* km = P.kv_map + bh_kv * P.n_kv + (int64_t)kb * 128 + lane;
#pragma unroll
                    for (int x = 0; x < 4; ++x) kt[x] = km[32 * x];
                    kmin = __reduce_min_sync(0xffffffffu, min(min(kt[0], kt[1]), min(kt[2], kt[3])));
                    kmax = __reduce_max_sync(0xffffffffu, max(max(kt[0], kt[1]), max(kt[2], kt[3])));
                } else {
                    kbase = kb * 128;
                    kmin = kbase;
                    kmax = kbase + 127;
                }
                need_mask = kmax >= P.n_valid || (P.causal && kmax > tok) ||
                            (P.window > 0 && kmin <= tok - P.window && kmax >= P.sinks);
                // visibility of the 128 columns as four 32-bit words, built
                // before S_j arrives so that only the words stay live
                if (__any_sync(0xffffffffu, need_mask) && P.kv_map == nullptr) {
                    // contiguous keys kbase .. kbase + 127: the visible ones form
                    // at most two runs, [tok - window + 1, hi) and [0, min(sinks, hi))
                    // with hi = min(n_valid, tok + 1) (causal) or n_valid; each word
                    // is the union of the runs' bits in its 32 columns
                    const int32_t hi_g = P.causal ? min(P.n_valid, tok + 1) : P.n_valid;
                    int32_t a1 = -kbase, a2 = 0, b2 = 0;
                    if (P.window > 0) {
                        a1 = tok - P.window + 1 - kbase;
                        a2 = -kbase;
                        b2 = min(P.sinks, hi_g) - kbase;
                    }
                    const int32_t b1 = hi_g - kbase;
#pragma unroll
                    for (int x = 0; x < 4; ++x)
                        vis_w[x] = run_bits(a1 - 32 * x, b1 - 32 * x) | run_bits(a2 - 32 * x, b2 - 32 * x);
                } else if (__any_sync(0xffffffffu, need_mask)) {
                    const int32_t nv = P.n_valid, win = P.window, sk = P.sinks;
                    const bool causal = P.causal != 0;
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        uint32_t word = 0u;
#pragma unroll
                        for (int c = 0; c < 32; ++c) {
                            const int32_t jt = P.kv_map != nullptr ? __shfl_sync(0xffffffffu, kt[x], c)
                                                                   : kbase + 32 * x + c;
                            const bool vis = jt < nv && (!causal || jt <= tok) &&
                                             (win <= 0 || jt > tok - win || jt < sk);
                            word |= (uint32_t)vis << c;
                        }
                        vis_w[x] = word;
                    }
                } else {
                    need_mask = false;
                }
            }
            const int32_t pk = ring_pos_k(j);
            bool w = mbar_wait(smem_u32(&bars->empty[pk % C::kStages]), (uint32_t)(pk / C::kStages) & 1u, kWaitNs, P.status, BSA_ERR_TIMEOUT);
            if (__any_sync(0xffffffffu, !w || aborted(bars))) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (kQuad && hidden) {
                // P_j = 0 for these rows; m, l and O are unchanged
                uint32_t z[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) z[c] = 0u;
                tmem_st32(t_lane + sbuf + 0, z);
                tmem_st32(t_lane + sbuf + 32, z);
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(smem_u32(&bars->p_full[j % kSBuf]));
                continue;
            }
            uint32_t s[128];
            // S_j out of tensor memory, dropped keys set to -inf
            auto load_s = [&]() {
                tmem_ld32(t_lane + sbuf + 0, &s[0]);
                tmem_ld32(t_lane + sbuf + 32, &s[32]);
                tmem_ld32(t_lane + sbuf + 64, &s[64]);
                tmem_ld32(t_lane + sbuf + 96, &s[96]);
                tmem_wait_ld();
                if constexpr (kMask) {
                    if (__any_sync(0xffffffffu, need_mask)) {
                        const uint32_t ninf = __float_as_uint(-INFINITY);
#pragma unroll
                        for (int c = 0; c < 128; ++c) s[c] = ((vis_w[c >> 5] >> (c & 31)) & 1u) ? s[c] : ninf;
                    }
                }
            };
            load_s();
            float alpha;
            const bool rescale = softmax_block<kPoly, kMask>(s, j, sl2, lw2, m, l, alpha, load_s);
            tmem_st32(t_lane + sbuf + 0, &s[0]);
            tmem_st32(t_lane + sbuf + 32, &s[32]);
            if (rescale) {
                // O must hold P_0..P_{j-1} V: wait for PV_{j-1}
                const int32_t pv = ring_pos_v(j - 1, n);
                w = mbar_wait(smem_u32(&bars->empty[pv % C::kStages]), (uint32_t)(pv / C::kStages) & 1u, kWaitNs, P.status, BSA_ERR_TIMEOUT);
                if (__any_sync(0xffffffffu, !w)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < D; c += 32) {
                    uint32_t o[32];
                    tmem_ld32(t_lane + kColO + c, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tmem_st32(t_lane + kColO + c, o);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(smem_u32(&bars->p_full[j % kSBuf]));
        }
        if (!ok) {
            if (lane == 0) set_abort(bars, P.status);
        } else {
            __nv_bfloat16* orow = P.o + (bh * N + tok) * D;
            if (n == 0) {
                if (tok_ok) {
                    const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
                    for (int c = 0; c < D; c += 8) *reinterpret_cast<uint4*>(orow + c) = z;
                    P.lse[bh * N + tok] = -INFINITY;
                }
            } else {
                const int32_t pv = ring_pos_v(n - 1, n);
                const bool w = mbar_wait(smem_u32(&bars->empty[pv % C::kStages]), (uint32_t)(pv / C::kStages) & 1u, kWaitNs, P.status, BSA_ERR_TIMEOUT);
                if (__any_sync(0xffffffffu, !w)) {
                    if (lane == 0) set_abort(bars, P.status);
                } else {
                    tc_fence_after();
                    const float inv_l = l > 0.0f ? 1.0f / l : 0.0f;  // l = 0: every key dropped
#pragma unroll
                    for (int c = 0; c < D; c += 32) {
                        uint32_t o[32];
                        tmem_ld32(t_lane + kColO + c, o);
                        tmem_wait_ld();
                        uint32_t pk[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            pk[i] = pack_bf16(__uint_as_float(o[2 * i]) * inv_l,
                                              __uint_as_float(o[2 * i + 1]) * inv_l);
                        if (tok_ok) {
                            uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                        }
                    }
                    if (tok_ok) P.lse[bh * N + tok] = l > 0.0f ? (m + log2f(l)) * kLn2 : -INFINITY;
                }
            }
        }
    }

    cp_async_wait_all();  // no copies of this thread may outlive the block
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// ---------------------------------------------------------------- per-item blocks
// The geometry layers (Scatter, Gather 0) have short rows: 1 and 7-8 block
// pairs.  One thread block per row pays a launch, a prologue, the first
// tiles' DRAM round trip and an epilogue with the tensor core idle.  Here one
// block per SM walks several rows ("items") in wave order: the producer runs
// into the next item's Q (two Q buffers) and tiles while the current item
// computes, the MMA lane starts the next item's QK as soon as its tiles land,
// and the softmax warps hand O over (o_free) before they normalise and store
// it.  Ring and score-buffer positions continue across items.
struct ItemBarriers {
    uint64_t full[16];
    uint64_t empty[16];
    uint64_t q_full[2];
    uint64_t q_empty[2];
    uint64_t p_full[kSBuf];
    uint64_t o_free;
    uint64_t mma_done;
    uint32_t tmem_base;
    int32_t abort;
};

struct Item {
    int64_t bh, bh_kv, row;
    int32_t qb, n;
    int32_t n_raw;  // the count as read (n is clamped to [0, max_kv])
};

__device__ __forceinline__ void report_count(const Params& P, int32_t n) {
    if (n < 0 || n > P.max_kv) raise_status(P.status, n < 0 ? BSA_ERR_BOUNDS : BSA_ERR_OVERFLOW);
}

// Item f is execution slot f % nQB of head f / nQB.  false: a bad row order
// entry (every role skips the item alike; the producer reports it, and a bad
// count, with report_count once it reaches the item).  Nothing here branches
// on the count, so a role can decode the next item while the current one
// runs without waiting for the load.
__device__ __forceinline__ bool decode_item(const Params& P, int64_t f, Item& it, int64_t BH) {
    // BH > 0: heads interleaved, consecutive items are the same execution slot
    // of consecutive heads (see kInterleave); else head-major
    const int32_t nQB = P.nQB;
    it.bh = BH > 0 ? f % BH : f / nQB;
    const int32_t slot = (int32_t)(BH > 0 ? f / BH : f - it.bh * nQB);
    int32_t qb = slot;
    if (P.row_perm != nullptr) {
        qb = P.row_perm[it.bh * nQB + slot];
        if (qb < 0 || qb >= nQB) return false;
    }
    it.qb = qb;
    it.bh_kv = (it.bh / P.H) * (P.H / P.group) + (it.bh % P.H) / P.group;
    it.row = it.bh * nQB + qb;
    const int32_t n = P.kv_cnt[it.row];
    it.n_raw = n;
    it.n = n < 0 ? 0 : (n > P.max_kv ? P.max_kv : n);
    return true;
}

__device__ __forceinline__ bool items_aborted(const ItemBarriers* b) {
    return *reinterpret_cast<const volatile int32_t*>(&b->abort) != 0;
}
__device__ __forceinline__ void items_set_abort(ItemBarriers* b, int32_t* status) {
    *reinterpret_cast<volatile int32_t*>(&b->abort) = 1;
    raise_status(status, BSA_ERR_TIMEOUT);
}

// kQB Q buffers: two let the next row's Q load while the current row's
// products still read its Q, at the cost of one ring slot; with one, the next
// Q loads once the current row's last QK has run (the PVs do not read Q).
template <int D, int kQB>
struct ItemCfg {
    static constexpr int kStages = Cfg<D>::kStages + 1 - kQB;
    static constexpr int kData = Cfg<D>::kTile * (kQB + kStages);
};

template <int D, int kPoly, bool kMask, bool kGeom, bool kQuad, int kQB>
__global__ void __launch_bounds__(threads_for(false, kMask), 1) k_bsa_forward_items(const __grid_constant__ Params P, int64_t n_items) {
    static_assert(kQB == 1 || kQB == 2, "one or two Q buffers");
    using C = Cfg<D>;
    using IC = ItemCfg<D, kQB>;
    constexpr int S = IC::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s_q = smem_u32(smem);  // two Q buffers, then the K/V ring
    const uint32_t s_ring = s_q + kQB * C::kTile;
    ItemBarriers* bars = reinterpret_cast<ItemBarriers*>(smem + IC::kData);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int32_t N = P.N, max_kv = P.max_kv, nKB = kGeom ? P.n_kv / 128 : P.nQB;
    // wave w takes item w * G + b, or w * G + G - 1 - b on odd waves (zig-zag)
    const int64_t G = gridDim.x;
    auto item_of = [&](int64_t w) -> int64_t {
        return w * G + ((w & 1) ? (G - 1 - (int64_t)blockIdx.x) : (int64_t)blockIdx.x);
    };
    // The Gather 0 layer walks the heads interleaved (item f is execution slot
    // f / BH of head f % BH): a text query tile lists about three times the
    // tiles of an image tile, and head-major order hands some blocks two of
    // them and others none.  Elsewhere head-major order keeps a wave on
    // neighbouring rows of one head (DRAM pages and L2 reuse).
    constexpr bool kInterleave = kGeom && kQuad;
    const int64_t heads_il = kInterleave ? n_items / P.nQB : 0;

    if (*reinterpret_cast<const volatile int32_t*>(P.status) == BSA_ERR_TIMEOUT) return;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&bars->full[s]), 1);
            mbar_init(smem_u32(&bars->empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&bars->q_full[b]), 1);
            mbar_init(smem_u32(&bars->q_empty[b]), 1);
        }
        for (int s = 0; s < kSBuf; ++s) mbar_init(smem_u32(&bars->p_full[s]), 32 * softmax_warps(kMask));
        mbar_init(smem_u32(&bars->o_free), 32 * softmax_warps(kMask));
        mbar_init(smem_u32(&bars->mma_done), 1);
        bars->abort = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(&bars->tmem_base), kTmemCols);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        prefetch_tensormap(&P.map_k);
        prefetch_tensormap(&P.map_v);
        if constexpr (kGeom) {
            prefetch_tensormap(&P.map_ki);
            prefetch_tensormap(&P.map_vi);
            if (P.geo.nt > 0 || P.geo.scatter) {
                prefetch_tensormap(&P.map_kg);
                prefetch_tensormap(&P.map_vg);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ producer
        uint32_t t_glob = 0, qi = 0;
        uint32_t issued = 0, q_issued = 0;  // copies started (ring positions, Q loads)
        bool ok = true;
        // Items are decoded one ahead: the next item's count and first 64 list
        // entries (lane e: entries e, 32 + e) load while this item's copies
        // are issued, so that no item starts by waiting for them.
        Item next_it{};
        bool next_ok = item_of(0) < n_items && decode_item(P, item_of(0), next_it, heads_il);
        int32_t next_e0 = 0, next_e1 = 0;
        auto load_entries = [&]() {
            const int32_t* l = P.kv_idx + next_it.row * max_kv;
            next_e0 = next_ok && lane < max_kv ? l[lane] : 0;
            next_e1 = next_ok && 32 + lane < max_kv ? l[32 + lane] : 0;
        };
        load_entries();
        for (int64_t w = 0; ok; ++w) {
            if (item_of(w) >= n_items) break;
            const Item it = next_it;
            const bool it_ok = next_ok;
            const int32_t cur_e0 = next_e0, cur_e1 = next_e1;
            next_ok = item_of(w + 1) < n_items && decode_item(P, item_of(w + 1), next_it, heads_il);
            load_entries();
            // bad entries are reported here, once the item's values are needed
            if (!it_ok) {
                if (lane == 0) raise_status(P.status, BSA_ERR_BOUNDS);  // a row-order entry out of range
                continue;
            }
            if (lane == 0) report_count(P, it.n_raw);
            const int32_t n = it.n;
            if (n == 0) continue;
            const int32_t* list = P.kv_idx + it.row * max_kv;
            const uint32_t qbuf = qi % kQB;
            if (lane == 0) {
                // the buffer's previous item must be done with it
                if (qi >= (uint32_t)kQB && !mbar_wait(smem_u32(&bars->q_empty[qbuf]), (qi / kQB - 1u) & 1u, kWaitNs,
                                                      P.status, BSA_ERR_TIMEOUT))
                    ok = false;
                if (ok) {
                    mbar_arrive_expect_tx(smem_u32(&bars->q_full[qbuf]), C::kTile);
                    if constexpr (kGeom) geo_load_q(P, s_q + qbuf * C::kTile, smem_u32(&bars->q_full[qbuf]), it.bh, it.qb);
                    else tma_load_3d(s_q + qbuf * C::kTile, &P.map_q, 0, (int32_t)(it.bh * N) + it.qb * 128, 0,
                                     smem_u32(&bars->q_full[qbuf]));
                }
            }
            ok = __shfl_sync(0xffffffffu, (int)ok, 0) != 0;
            if (!ok) break;
            q_issued = qi + 1;
            // tiles in MMA consumption order: K_0 .. K_2, then V_i, K_{i+3}, then the last V.
            // The K and V streams each walk the list in increasing order through
            // their own 32-entry window, with the next window already loaded
            // (lane e holds entry base + e): every entry is read once, about 32
            // tiles before it is needed.
            auto checked = [&](int32_t e, int32_t kb) -> int32_t {
                kb = e < n ? kb : 0;
                if (kb < 0 || kb >= nKB) {
                    raise_status(P.status, BSA_ERR_BOUNDS);
                    kb = 0;  // keeps the pipeline in step; this row's result is unspecified
                }
                return kb;
            };
            auto fetch = [&](int32_t e) -> int32_t { return checked(e, e < n ? list[e] : 0); };
            int32_t k_base = 0, k_cur = checked(lane, cur_e0), k_nxt = checked(32 + lane, cur_e1);
            int32_t v_base = 0, v_cur = k_cur, v_nxt = k_nxt;
            auto stream_kb = [&](int32_t e, int32_t& base, int32_t& cur, int32_t& nxt) -> int32_t {
                while (e >= base + 32) {
                    base += 32;
                    cur = nxt;
                    nxt = fetch(base + 32 + lane);
                }
                return __shfl_sync(0xffffffffu, cur, e - base);
            };
            const int32_t lead = n < kSBuf ? n : kSBuf;
            const int32_t inter = 2 * (n - lead);
            for (int32_t t = 0; t < 2 * n; ++t) {
                const bool is_v = t >= lead && (t - lead >= inter || ((t - lead) & 1) == 0);
                int32_t e;
                if (t < lead) e = t;
                else if (t - lead < inter) e = ((t - lead) >> 1) + (is_v ? 0 : kSBuf);
                else e = (n - lead) + (t - lead - inter);
                const int32_t kb = is_v ? stream_kb(e, v_base, v_cur, v_nxt) : stream_kb(e, k_base, k_cur, k_nxt);
                const uint32_t pos = t_glob + (uint32_t)t;
                const uint32_t slot = pos % S;
                // every lane waits (warp-uniform control flow); one elected lane issues
                const bool wt = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->empty[slot]), ((pos / S) & 1u) ^ 1u,
                                                                  kWaitNs, P.status, BSA_ERR_TIMEOUT));
                if (!wt || items_aborted(bars)) {
                    ok = false;
                    break;
                }
                if (elect_one()) {
                    const uint32_t fb = smem_u32(&bars->full[slot]);
                    mbar_arrive_expect_tx(fb, C::kTile);
                    if constexpr (kGeom) geo_load_kv(P, s_ring + slot * C::kTile, fb, is_v, it.bh_kv, kb);
                    else tma_load_3d(s_ring + slot * C::kTile, is_v ? &P.map_v : &P.map_k, 0,
                                     (int32_t)(it.bh_kv * N) + kb * 128, 0, fb);
                }
                __syncwarp();
                issued = pos + 1;
            }
            if (!ok) break;
            t_glob += 2u * (uint32_t)n;
            ++qi;
        }
        if (!ok && lane == 0) items_set_abort(bars, P.status);
        // Drain: every issued copy must land before the block exits (older
        // copies were consumed before their buffers were reused).
        if (lane == 0) {
            for (uint32_t q = q_issued > (uint32_t)kQB ? q_issued - kQB : 0; q < q_issued; ++q)
                if (!mbar_wait(smem_u32(&bars->q_full[q % kQB]), (q / kQB) & 1u, kWaitNs, P.status, BSA_ERR_TIMEOUT))
                    raise_status(P.status, BSA_ERR_TIMEOUT);
            const uint32_t first = issued > (uint32_t)S ? issued - S : 0;
            for (uint32_t i = first; i < issued; ++i)
                if (!mbar_wait(smem_u32(&bars->full[i % S]), (i / S) & 1u, kWaitNs, P.status, BSA_ERR_TIMEOUT))
                    raise_status(P.status, BSA_ERR_TIMEOUT);
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp walks the items (warp-uniform control flow and
        // descriptor arithmetic); one elected lane issues each MMA group.
        const uint64_t dk = smem_desc_sw128(s_ring, 16, 1024);
        const uint64_t dv = smem_desc_sw128(s_ring, C::kBoxBytes, 1024);
        uint32_t pos = 0, g_glob = 0, qi = 0;  // ring position, score buffer count, items
        bool ok = true;
        auto wait_all = [&](uint32_t bar, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, mbar_wait(bar, parity, kWaitNs, P.status, BSA_ERR_TIMEOUT));
        };
        Item next_it{};  // decoded one ahead (see the producer)
        bool next_ok = item_of(0) < n_items && decode_item(P, item_of(0), next_it, heads_il);
        for (int64_t w = 0; ok; ++w) {
            if (item_of(w) >= n_items) break;
            const Item it = next_it;
            const bool it_ok = next_ok;
            next_ok = item_of(w + 1) < n_items && decode_item(P, item_of(w + 1), next_it, heads_il);
            if (!it_ok || it.n == 0) continue;
            const int32_t n = it.n;
            const uint32_t qbuf = qi % kQB;
            ok = wait_all(smem_u32(&bars->q_full[qbuf]), (qi / kQB) & 1u);
            if (!ok) break;
            tc_fence_after();
            const uint64_t dq = smem_desc_sw128(s_q + qbuf * C::kTile, 16, 1024);
            auto issue_qk = [&](int32_t j) -> bool {
                const uint32_t slot = pos % S;
                if (!wait_all(smem_u32(&bars->full[slot]), (pos / S) & 1u)) return false;
                tc_fence_after();
                const uint64_t ks = dk + (uint64_t)((slot * C::kTile) >> 4);
                const uint32_t d_col = ((g_glob + (uint32_t)j) % kSBuf) * 128u;
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = ((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4;
                        mma_ss(tmem + d_col, dq + off, ks + off, C::kIdescQK, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(smem_u32(&bars->empty[slot]));  // also signals S_j to the softmax
                    // one Q buffer: free once the row's last QK has run
                    if (kQB == 1 && j == n - 1) mma_commit(smem_u32(&bars->q_empty[0]));
                }
                __syncwarp();
                ++pos;
                return true;
            };
            for (int32_t j = 0; ok && j < n && j < kSBuf; ++j) ok = issue_qk(j);
            for (int32_t i = 0; ok && i < n; ++i) {
                const uint32_t gb = g_glob + (uint32_t)i;
                ok = wait_all(smem_u32(&bars->p_full[gb % kSBuf]), (gb / kSBuf) & 1u);
                // the first PV of an item overwrites O: the previous item's
                // epilogue must have read it out
                if (ok && i == 0 && qi > 0) ok = wait_all(smem_u32(&bars->o_free), (qi - 1u) & 1u);
                if (!ok) break;
                const uint32_t slot = pos % S;
                ok = wait_all(smem_u32(&bars->full[slot]), (pos / S) & 1u);
                if (!ok) break;
                tc_fence_after();
                const uint64_t vs = dv + (uint64_t)((slot * C::kTile) >> 4);
                const uint32_t p_col = (gb % kSBuf) * 128u;
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ts(tmem + kColO, tmem + p_col + kk * 8, vs + (uint64_t)(kk * 2048 >> 4), C::kIdescPV,
                               (i > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(smem_u32(&bars->empty[slot]));  // also signals PV_i to the softmax
                }
                __syncwarp();
                ++pos;
                // score buffer gb % 3 is free again once PV_i (issued above) has read P
                if (i + kSBuf < n) ok = issue_qk(i + kSBuf);
            }
            if (!ok) break;
            if (kQB == 2) {
                if (elect_one()) mma_commit(smem_u32(&bars->q_empty[qbuf]));  // once this item's MMAs ran
                __syncwarp();
            }
            g_glob += (uint32_t)n;
            ++qi;
        }
        if (!ok && lane == 0) items_set_abort(bars, P.status);
        // Drain: nothing of ours may still be running when TMEM is freed.
        if (elect_one()) mma_commit(smem_u32(&bars->mma_done));
        __syncwarp();
        if (!mbar_wait(smem_u32(&bars->mma_done), 0, kWaitNs, P.status, BSA_ERR_TIMEOUT) && lane == 0)
            raise_status(P.status, BSA_ERR_TIMEOUT);
        __syncwarp();
    } else if constexpr (!kMask) {
        // ------------------------------------------------ softmax + epilogue (row split)
        const int qd = warp & 3;
        const int half = (warp - kFirstSoftmaxWarp) >> 2;
        const int ra = qd * 32 + half * 16 + (lane >> 2), rb = ra + 8;
        const uint32_t t_base = tmem + ((uint32_t)(qd * 32 + half * 16) << 16);
        const float sl2 = P.scale_log2;
        uint32_t t_glob = 0, g_glob = 0;
        bool ok = true;
        Item next_it{};  // decoded one ahead (see the producer)
        bool next_ok = item_of(0) < n_items && decode_item(P, item_of(0), next_it, heads_il);
        // An item's normalised O waits in registers and is stored while the
        // next item's last PV runs, off the softmax warps' critical path.
        uint32_t pend[D / 4];
        __nv_bfloat16 *pend_a = nullptr, *pend_b = nullptr;
        bool pending = false;
        for (int64_t w = 0; ok; ++w) {
            if (item_of(w) >= n_items) break;
            const Item it = next_it;
            const bool it_ok = next_ok;
            next_ok = item_of(w + 1) < n_items && decode_item(P, item_of(w + 1), next_it, heads_il);
            if (!it_ok) continue;
            const int32_t n = it.n;
            const int32_t tok_a = kGeom ? g0::query_token(P.geo, it.qb * 128 + ra) : it.qb * 128 + ra;
            const int32_t tok_b = kGeom ? g0::query_token(P.geo, it.qb * 128 + rb) : it.qb * 128 + rb;
            __nv_bfloat16* row_a = P.o + (it.bh * N + tok_a) * D;
            __nv_bfloat16* row_b = P.o + (it.bh * N + tok_b) * D;
            const int c = 2 * (lane & 3);
            if (n == 0) {
#pragma unroll
                for (int k = 0; k < D / 8; ++k) {
                    *reinterpret_cast<uint32_t*>(row_a + 8 * k + c) = 0u;
                    *reinterpret_cast<uint32_t*>(row_b + 8 * k + c) = 0u;
                }
                if ((lane & 3) == 0) {
                    P.lse[it.bh * N + tok_a] = -INFINITY;
                    P.lse[it.bh * N + tok_b] = -INFINITY;
                }
                continue;
            }
            const float* lw_row = P.log_w ? P.log_w + it.row * max_kv : nullptr;
            const uint8_t* qm_row = (kQuad && P.quad_mask != nullptr) ? P.quad_mask + it.row * max_kv : nullptr;
            uint32_t qm_chunk = 0xFu;
            if constexpr (kQuad) qm_chunk = (qm_row != nullptr && lane < n) ? qm_row[lane] : 0xFu;
            float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.0f, 0.0f};
            float lw_next = lw_row ? lw_row[0] : 0.0f;
            for (int32_t j = 0; j < n; ++j) {
                const float lw2 = lw_next * kLog2e;
                lw_next = (lw_row && j + 1 < n) ? lw_row[j + 1] : 0.0f;
                if (kQuad && j > 0 && (j & 31) == 0)
                    qm_chunk = (qm_row != nullptr && j + lane < n) ? qm_row[j + lane] : 0xFu;
                bool hidden = false;  // warp-uniform: no row of this quadrant sees block j
                if constexpr (kQuad) hidden = ((__shfl_sync(0xffffffffu, qm_chunk, j & 31) >> qd) & 1u) == 0u;
                const uint32_t gb = g_glob + (uint32_t)j;
                const uint32_t sbuf = (gb % kSBuf) * 128u;
                const uint32_t pk = t_glob + (uint32_t)ring_pos_k(j);
                const bool wt = mbar_wait(smem_u32(&bars->empty[pk % S]), (pk / S) & 1u, kWaitNs, P.status, BSA_ERR_TIMEOUT);
                if (__any_sync(0xffffffffu, !wt || items_aborted(bars))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (kQuad && hidden) {
                    store_p_zero(t_base + sbuf);
                    tc_fence_before();
                    mbar_arrive(smem_u32(&bars->p_full[gb % kSBuf]));
                    continue;
                }
                uint32_t s[64];
                auto load_s = [&]() {
                    tmem_ld16x256_x16(t_base + sbuf, s);
                    tmem_wait_ld();
                };
                load_s();
                float alpha[2];
                const bool rescale = softmax_block_rows<kPoly>(s, j, sl2, lw2, m, l, alpha, load_s);
                tmem_st16x128_x16(t_base + sbuf, s);
                if (rescale) {
                    // O must hold P_0..P_{j-1} V: wait for PV_{j-1}
                    const uint32_t pv = t_glob + (uint32_t)ring_pos_v(j - 1, n);
                    const bool wv = mbar_wait(smem_u32(&bars->empty[pv % S]), (pv / S) & 1u, kWaitNs, P.status, BSA_ERR_TIMEOUT);
                    if (__any_sync(0xffffffffu, !wv)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    scale_o_rows<D>(t_base + kColO, alpha[0], alpha[1]);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(smem_u32(&bars->p_full[gb % kSBuf]));
            }
            if (!ok) break;
            // Epilogue: the previous item's O leaves while PV_{n-1} runs; once
            // it has run, read O out of tensor memory, hand the accumulator to
            // the next item (o_free) and keep the normalised rows for later.
            if (pending) store_packed_pairs<D>(pend, pend_a, pend_b);
            {
                const uint32_t pv = t_glob + (uint32_t)ring_pos_v(n - 1, n);
                const bool wt = mbar_wait(smem_u32(&bars->empty[pv % S]), (pv / S) & 1u, kWaitNs, P.status, BSA_ERR_TIMEOUT);
                if (__any_sync(0xffffffffu, !wt)) {
                    ok = false;
                    break;
                }
            }
            tc_fence_after();
            const float l_a = row_sum4(l[0]), l_b = row_sum4(l[1]);
            const float inv_a = l_a > 0.0f ? 1.0f / l_a : 0.0f, inv_b = l_b > 0.0f ? 1.0f / l_b : 0.0f;
            uint32_t o[D / 2];
            if constexpr (D == 128) tmem_ld16x256_x16(t_base + kColO, o);
            else tmem_ld16x256_x8(t_base + kColO, o);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(smem_u32(&bars->o_free));
            pack_o_pairs<D>(o, inv_a, inv_b, pend);
            pend_a = row_a;
            pend_b = row_b;
            pending = true;
            if ((lane & 3) == 0) {
                P.lse[it.bh * N + tok_a] = l_a > 0.0f ? (m[0] + log2f(l_a)) * kLn2 : -INFINITY;
                P.lse[it.bh * N + tok_b] = l_b > 0.0f ? (m[1] + log2f(l_b)) * kLn2 : -INFINITY;
            }
            t_glob += 2u * (uint32_t)n;
            g_glob += (uint32_t)n;
        }
        if (ok && pending) store_packed_pairs<D>(pend, pend_a, pend_b);
        if (!ok && lane == 0) items_set_abort(bars, P.status);
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        const int qd = warp & 3;                 // TMEM lane quadrant of this warp
        const int r = qd * 32 + lane;            // row within the query tile
        const uint32_t t_lane = tmem + ((uint32_t)(qd * 32) << 16);
        const float sl2 = P.scale_log2;
        uint32_t t_glob = 0, g_glob = 0;
        bool ok = true;
        for (int64_t w = 0; ok; ++w) {
            const int64_t f = item_of(w);
            if (f >= n_items) break;
            Item it;
            if (!decode_item(P, f, it, heads_il)) continue;
            const int32_t n = it.n;
            const int32_t tok = kGeom ? g0::query_token(P.geo, it.qb * 128 + r) : it.qb * 128 + r;
            __nv_bfloat16* orow = P.o + (it.bh * N + tok) * D;
            if (n == 0) {
                const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int c = 0; c < D; c += 8) *reinterpret_cast<uint4*>(orow + c) = z;
                P.lse[it.bh * N + tok] = -INFINITY;
                continue;
            }
            const float* lw_row = P.log_w ? P.log_w + it.row * max_kv : nullptr;
            const uint8_t* qm_row = (kQuad && P.quad_mask != nullptr) ? P.quad_mask + it.row * max_kv : nullptr;
            const int32_t* list = P.kv_idx + it.row * max_kv;
            float m = -INFINITY, l = 0.0f;
            float lw_next = lw_row ? lw_row[0] : 0.0f;
            uint32_t qm_chunk = 0xFu;
            if constexpr (kQuad) qm_chunk = (qm_row != nullptr && lane < n) ? qm_row[lane] : 0xFu;
            for (int32_t j = 0; j < n; ++j) {
                const float lw2 = lw_next * kLog2e;
                lw_next = (lw_row && j + 1 < n) ? lw_row[j + 1] : 0.0f;
                if (kQuad && j > 0 && (j & 31) == 0)
                    qm_chunk = (qm_row != nullptr && j + lane < n) ? qm_row[j + lane] : 0xFu;
                const uint32_t gb = g_glob + (uint32_t)j;
                const uint32_t sbuf = (gb % kSBuf) * 128u;
                bool hidden = false;  // warp-uniform: no row of this warp sees block j
                if constexpr (kQuad) hidden = ((__shfl_sync(0xffffffffu, qm_chunk, j & 31) >> qd) & 1u) == 0u;
                // Token mask of block j (contiguous keys 128 kb ..): visibility
                // words from at most two runs, built before S_j arrives
                bool need_mask = false;
                uint32_t vis_w[4] = {~0u, ~0u, ~0u, ~0u};
                if (kMask && !kGeom) {
                    int32_t kb = list[j];
                    kb = (kb < 0 || kb >= nKB) ? 0 : kb;  // flagged by the producer
                    const int32_t kbase = kb * 128, kmax = kbase + 127;
                    need_mask = kmax >= P.n_valid || (P.causal && kmax > tok) ||
                                (P.window > 0 && kbase <= tok - P.window && kmax >= P.sinks);
                    if (__any_sync(0xffffffffu, need_mask)) {
                        const int32_t hi_g = P.causal ? min(P.n_valid, tok + 1) : P.n_valid;
                        int32_t a1 = -kbase, a2 = 0, b2 = 0;
                        if (P.window > 0) {
                            a1 = tok - P.window + 1 - kbase;
                            a2 = -kbase;
                            b2 = min(P.sinks, hi_g) - kbase;
                        }
                        const int32_t b1 = hi_g - kbase;
#pragma unroll
                        for (int x = 0; x < 4; ++x)
                            vis_w[x] = run_bits(a1 - 32 * x, b1 - 32 * x) | run_bits(a2 - 32 * x, b2 - 32 * x);
                    } else {
                        need_mask = false;
                    }
                }
                const uint32_t pk = t_glob + (uint32_t)ring_pos_k(j);
                bool wt = mbar_wait(smem_u32(&bars->empty[pk % S]), (pk / S) & 1u, kWaitNs, P.status, BSA_ERR_TIMEOUT);
                if (__any_sync(0xffffffffu, !wt || items_aborted(bars))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (kQuad && hidden) {
                    // P_j = 0 for these rows; m, l and O are unchanged
                    uint32_t z[32];
#pragma unroll
                    for (int c = 0; c < 32; ++c) z[c] = 0u;
                    tmem_st32(t_lane + sbuf + 0, z);
                    tmem_st32(t_lane + sbuf + 32, z);
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(smem_u32(&bars->p_full[gb % kSBuf]));
                    continue;
                }
                uint32_t s[128];
                // S_j out of tensor memory, dropped keys set to -inf
                auto load_s = [&]() {
                    tmem_ld32(t_lane + sbuf + 0, &s[0]);
                    tmem_ld32(t_lane + sbuf + 32, &s[32]);
                    tmem_ld32(t_lane + sbuf + 64, &s[64]);
                    tmem_ld32(t_lane + sbuf + 96, &s[96]);
                    tmem_wait_ld();
                    if constexpr (kMask && !kGeom) {
                        if (__any_sync(0xffffffffu, need_mask)) {
                            const uint32_t ninf = __float_as_uint(-INFINITY);
#pragma unroll
                            for (int c = 0; c < 128; ++c) s[c] = ((vis_w[c >> 5] >> (c & 31)) & 1u) ? s[c] : ninf;
                        }
                    }
                };
                load_s();
                float alpha;
                const bool rescale = softmax_block<kPoly, kMask>(s, j, sl2, lw2, m, l, alpha, load_s);
                tmem_st32(t_lane + sbuf + 0, &s[0]);
                tmem_st32(t_lane + sbuf + 32, &s[32]);
                if (rescale) {
                    // O must hold P_0..P_{j-1} V: wait for PV_{j-1}
                    const uint32_t pv = t_glob + (uint32_t)ring_pos_v(j - 1, n);
                    wt = mbar_wait(smem_u32(&bars->empty[pv % S]), (pv / S) & 1u, kWaitNs, P.status, BSA_ERR_TIMEOUT);
                    if (__any_sync(0xffffffffu, !wt)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < D; c += 32) {
                        uint32_t o[32];
                        tmem_ld32(t_lane + kColO + c, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st32(t_lane + kColO + c, o);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(smem_u32(&bars->p_full[gb % kSBuf]));
            }
            if (!ok) break;
            // Epilogue: once PV_{n-1} has run, read O out of tensor memory, hand
            // the accumulator to the next item (o_free), then normalise and
            // store while the next item's products proceed.
            {
                const uint32_t pv = t_glob + (uint32_t)ring_pos_v(n - 1, n);
                const bool wt = mbar_wait(smem_u32(&bars->empty[pv % S]), (pv / S) & 1u, kWaitNs, P.status, BSA_ERR_TIMEOUT);
                if (__any_sync(0xffffffffu, !wt)) {
                    ok = false;
                    break;
                }
            }
            tc_fence_after();
            const float inv_l = l > 0.0f ? 1.0f / l : 0.0f;  // l = 0: every key dropped
            if constexpr (kQB == 2) {
                // short rows: read all of O, hand the accumulator over, then store
                uint32_t o[D];
#pragma unroll
                for (int c = 0; c < D; c += 32) tmem_ld32(t_lane + kColO + c, &o[c]);
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(smem_u32(&bars->o_free));
#pragma unroll
                for (int c = 0; c < D; c += 8) {
                    uint4 v4;
                    v4.x = pack_bf16(__uint_as_float(o[c + 0]) * inv_l, __uint_as_float(o[c + 1]) * inv_l);
                    v4.y = pack_bf16(__uint_as_float(o[c + 2]) * inv_l, __uint_as_float(o[c + 3]) * inv_l);
                    v4.z = pack_bf16(__uint_as_float(o[c + 4]) * inv_l, __uint_as_float(o[c + 5]) * inv_l);
                    v4.w = pack_bf16(__uint_as_float(o[c + 6]) * inv_l, __uint_as_float(o[c + 7]) * inv_l);
                    *reinterpret_cast<uint4*>(orow + c) = v4;
                }
            } else {
                // 32 columns at a time (fewer live registers), then the hand-over
#pragma unroll
                for (int c = 0; c < D; c += 32) {
                    uint32_t o[32];
                    tmem_ld32(t_lane + kColO + c, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; i += 8) {
                        uint4 v4;
                        v4.x = pack_bf16(__uint_as_float(o[i + 0]) * inv_l, __uint_as_float(o[i + 1]) * inv_l);
                        v4.y = pack_bf16(__uint_as_float(o[i + 2]) * inv_l, __uint_as_float(o[i + 3]) * inv_l);
                        v4.z = pack_bf16(__uint_as_float(o[i + 4]) * inv_l, __uint_as_float(o[i + 5]) * inv_l);
                        v4.w = pack_bf16(__uint_as_float(o[i + 6]) * inv_l, __uint_as_float(o[i + 7]) * inv_l);
                        *reinterpret_cast<uint4*>(orow + c + i) = v4;
                    }
                }
                tc_fence_before();
                mbar_arrive(smem_u32(&bars->o_free));
            }
            P.lse[it.bh * N + tok] = l > 0.0f ? (m + log2f(l)) * kLn2 : -INFINITY;
            t_glob += 2u * (uint32_t)n;
            g_glob += (uint32_t)n;
        }
        if (!ok && lane == 0) items_set_abort(bars, P.status);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

// [rows, D] as (64 columns, rows, D/64 halves) with a 64 x 128 x D/64 box.
bool encode_tile_map(CUtensorMap* map, const void* base, uint64_t rows, int D) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(D / 64)};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, 128};
    cuuint32_t box[3] = {64, 128, (cuuint32_t)(D / 64)};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Gather 0 views of a [heads, N, D] tensor whose tokens n_text .. N-1 are an
// img_h x img_w image: (64 columns, x, y, D/64 halves, head) with a
// 64 x bx x by x D/64 x 1 box, or with group = true the Scatter groups
// (64, g, t, D/64, head) for token n_text + t*groups + g, box 64 x 1 x 128.
bool encode_image_map(CUtensorMap* map, const void* base, uint64_t heads, int32_t N, int D,
                      const g0::Geom& g, bool group, uint32_t bx, uint32_t by) {
    auto enc = get_encode();
    if (!enc) return false;
    const uint64_t row = (uint64_t)D * 2;
    const void* img = static_cast<const uint8_t*>(base) + (uint64_t)g.nt * row;
    cuuint64_t dims[5] = {64, (cuuint64_t)(group ? g.groups : g.w), (cuuint64_t)(group ? g.hw / g.groups : g.h),
                          (cuuint64_t)(D / 64), (cuuint64_t)heads};
    cuuint64_t strides[4] = {row, (cuuint64_t)(group ? g.groups : g.w) * row, 128, (cuuint64_t)N * row};
    cuuint32_t box[5] = {64, group ? 1u : bx, group ? 128u : by, (cuuint32_t)(D / 64), 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(img), dims, strides, box,
                     estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int D>
size_t smem_bytes() {
    return 1024 + Cfg<D>::kData + sizeof(Barriers);
}

template <int D, int kPoly, bool kCrm, bool kGather, bool kMask, bool kGeom = false, bool kQuad = false>
cudaError_t prepare_kernel() {
    // Per device: opt in to the large dynamic shared-memory carve-out.
    static int done[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && done[dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(k_bsa_forward<D, kPoly, kCrm, kGather, kMask, kGeom, kQuad>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem_bytes<D>());
    if (e == cudaSuccess && dev < 64) done[dev] = 1;
    return e;
}

// Per-item blocks on the tile path pay off for short rows only (a wave of
// long rows keeps every SM busy on its own, and the per-item kernel's ring
// is one slot shorter).  A sliding window bounds a row by construction: with
// only blocks that hold a visible key listed, a row has at most
// (window + 254) / 128 window blocks plus the sink blocks.
constexpr int32_t kShortRowBlocks = 16;
bool items_tile_choice(const ForwardArgs& a) {
    const bsa_schedule sched = forward_options().schedule;
    if (sched != BSA_SCHEDULE_AUTO) return sched == BSA_SCHEDULE_PER_ITEM;
    if (!a.masked || a.window <= 0) return false;
    const int64_t bound = ((int64_t)a.window + 254) / 128 + ((int64_t)a.sinks + 127) / 128;
    return bound <= kShortRowBlocks;
}

// The geometry layers (Scatter, Gather 0) run per-item blocks unless one
// block per row is asked for.
bool items_geometry() { return forward_options().schedule != BSA_SCHEDULE_PER_ROW; }

template <int D, bool kMask, bool kGeom, bool kQuad, int kQB>
bsa_status launch_items(const Params& P, int64_t n_items, cudaStream_t stream) {
    const size_t smem = 1024 + ItemCfg<D, kQB>::kData + sizeof(ItemBarriers);
    static int done[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return BSA_ERR_CUDA;
    if (dev >= 64 || !done[dev]) {
        if (cudaFuncSetAttribute(k_bsa_forward_items<D, kDefaultPoly, kMask, kGeom, kQuad, kQB>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return BSA_ERR_CUDA;
        if (dev < 64) done[dev] = 1;
    }
    const int32_t resident = forward_resident_ctas(D);
    if (resident <= 0) return BSA_ERR_CUDA;
    const unsigned grid = (unsigned)(n_items < resident ? n_items : resident);
    k_bsa_forward_items<D, kDefaultPoly, kMask, kGeom, kQuad, kQB><<<grid, threads_for(false, kMask), smem, stream>>>(P, n_items);
    return cudaGetLastError() == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}

template <int D, int kPoly, bool kCrm, bool kGather, bool kMask = false, bool kGeom = false, bool kQuad = false>
bsa_status launch_dp(const Params& P, unsigned grid_x, unsigned grid_y, cudaStream_t stream) {
    if (prepare_kernel<D, kPoly, kCrm, kGather, kMask, kGeom, kQuad>() != cudaSuccess) return BSA_ERR_CUDA;
    k_bsa_forward<D, kPoly, kCrm, kGather, kMask, kGeom, kQuad>
        <<<dim3(grid_x, grid_y), threads_for(kGather, kMask), smem_bytes<D>(), stream>>>(P);
    return cudaGetLastError() == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}

template <int D>
bsa_status launch_d(const ForwardArgs& a, int32_t* status, cudaStream_t stream) {
    Params P;
    memset(&P, 0, sizeof(P));
    const int32_t H_kv = a.H_kv > 0 ? a.H_kv : a.H;
    const uint64_t rows = (uint64_t)a.B * a.H * a.N, kv_rows = (uint64_t)a.B * H_kv * a.N;
    bool ok = encode_tile_map(&P.map_q, a.q, rows, D) && encode_tile_map(&P.map_k, a.k, kv_rows, D) &&
              encode_tile_map(&P.map_v, a.v, kv_rows, D);
    if (!ok) return BSA_ERR_CUDA;
    P.q = static_cast<const __nv_bfloat16*>(a.q);
    P.k = static_cast<const __nv_bfloat16*>(a.k);
    P.v = static_cast<const __nv_bfloat16*>(a.v);
    P.kv_idx = a.kv_idx;
    P.kv_cnt = a.kv_cnt;
    P.log_w = a.log_w;
    P.q_map = a.q_map;
    P.kv_map = a.kv_map;
    P.quad_mask = a.quad_mask;
    P.row_perm = a.row_perm;
    P.crm = a.crm;
    P.crm_words = a.crm_words;
    P.o = static_cast<__nv_bfloat16*>(a.o);
    P.lse = a.lse;
    P.status = status;
    P.N = a.N;
    P.nQB = a.N / 128;
    P.max_kv = a.max_kv;
    P.n_kv = a.n_kv > 0 ? a.n_kv : a.N;
    P.H = a.H;
    P.group = a.H / H_kv;
    P.causal = a.causal;
    P.n_valid = a.n_valid > 0 ? a.n_valid : a.N;
    P.window = a.window;
    P.sinks = a.sinks;
    const float scale = a.scale > 0.f ? a.scale : 1.0f / sqrtf((float)D);
    P.scale_log2 = scale * kLog2e;
    const unsigned gx = (unsigned)P.nQB, gy = (unsigned)(a.B * a.H);
    if (a.gather0 != nullptr) {
        // Gather 0 geometry mode: tiles are TMA boxes of the image views
        const Gather0Geom& q0 = *a.gather0;
        const g0::Geom g = g0::make(q0.img_h, q0.img_w, q0.n_text, q0.groups, q0.N, q0.N_kv);
        P.geo = g;
        P.n_kv = g.N_kv;
        P.q_map = nullptr;
        P.kv_map = nullptr;
        const uint64_t qh = (uint64_t)a.B * a.H, kh = (uint64_t)a.B * H_kv;
        ok = encode_image_map(&P.map_qi, a.q, qh, a.N, D, g, false, 8, 16) &&
             encode_image_map(&P.map_ki, a.k, kh, a.N, D, g, false, 16, 8) &&
             encode_image_map(&P.map_vi, a.v, kh, a.N, D, g, false, 16, 8);
        if (ok && g.nt > 0)
            ok = encode_image_map(&P.map_kg, a.k, kh, a.N, D, g, true, 0, 0) &&
                 encode_image_map(&P.map_vg, a.v, kh, a.N, D, g, true, 0, 0);
        if (!ok) return BSA_ERR_CUDA;
        // no token masks in this mode: the row-split softmax with quadrant masks;
        // rows of about 7 tiles keep the full six-slot ring and one Q buffer
        if (items_geometry()) return launch_items<D, false, true, true, 1>(P, (int64_t)gx * gy, stream);
        return launch_dp<D, kDefaultPoly, false, false, false, true, true>(P, gx, gy, stream);
    }
    if (a.scatter_R > 0) {
        // Scatter geometry mode: every query and key/value tile is 128 tokens
        // of one group at stride R, one TMA box each
        const g0::Geom g = g0::make_scatter(a.N, a.scatter_R);
        P.geo = g;
        P.n_kv = g.N_kv;
        P.q_map = nullptr;
        P.kv_map = nullptr;
        const uint64_t qh = (uint64_t)a.B * a.H, kh = (uint64_t)a.B * H_kv;
        ok = encode_image_map(&P.map_qg, a.q, qh, a.N, D, g, true, 0, 0) &&
             encode_image_map(&P.map_kg, a.k, kh, a.N, D, g, true, 0, 0) &&
             encode_image_map(&P.map_vg, a.v, kh, a.N, D, g, true, 0, 0);
        if (!ok) return BSA_ERR_CUDA;
        if (items_geometry()) return launch_items<D, false, true, false, 2>(P, (int64_t)gx * gy, stream);
        return launch_dp<D, kDefaultPoly, false, false, false, true, false>(P, gx, gy, stream);
    }
    const bool crm = a.crm != nullptr, gather = a.kv_map != nullptr;
    if (a.masked) {
        if (crm) return BSA_ERR_UNSUPPORTED;
        const bool token_mask = a.causal || a.window > 0 || P.n_valid < a.N;
        if (gather && P.quad_mask != nullptr)
            return token_mask ? launch_dp<D, kDefaultPoly, false, true, true, false, true>(P, gx, gy, stream)
                              : launch_dp<D, kDefaultPoly, false, true, false, false, true>(P, gx, gy, stream);
        if (P.quad_mask != nullptr) return BSA_ERR_UNSUPPORTED;  // packed tiles need kv_map
        if (!gather && P.q_map == nullptr && items_tile_choice(a))
            return launch_items<D, true, false, false, 1>(P, (int64_t)gx * gy, stream);
        return gather ? launch_dp<D, kDefaultPoly, false, true, true>(P, gx, gy, stream)
                      : launch_dp<D, kDefaultPoly, false, false, true>(P, gx, gy, stream);
    }
    if (!gather && !crm && P.q_map == nullptr && items_tile_choice(a))
        return launch_items<D, false, false, false, 1>(P, (int64_t)gx * gy, stream);
    if (gather)
        return crm ? launch_dp<D, kDefaultPoly, true, true>(P, gx, gy, stream)
                   : launch_dp<D, kDefaultPoly, false, true>(P, gx, gy, stream);
    if (crm) return launch_dp<D, kDefaultPoly, true, false>(P, gx, gy, stream);
    return forward_options().exp2_fma == 2 ? launch_dp<D, 2, false, false>(P, gx, gy, stream)
                                           : launch_dp<D, 0, false, false>(P, gx, gy, stream);
}

template <int D>
int32_t occupancy() {
    int per_sm = 0;
    // every instantiation holds one block per SM (shared memory bound)
    if (prepare_kernel<D, kDefaultPoly, false, false, false>() != cudaSuccess) return -1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_bsa_forward<D, kDefaultPoly, false, false, false, false, false>,
                                                      threads_for(false, false),
                                                      smem_bytes<D>()) != cudaSuccess)
        return -1;
    return per_sm;
}

}  // namespace

bsa_forward_options& forward_options() {
    thread_local bsa_forward_options opts{BSA_SCHEDULE_AUTO, 0};
    return opts;
}

bsa_status launch_forward(const ForwardArgs& a, int32_t* status, cudaStream_t stream) {
    if (a.D == 128) return launch_d<128>(a, status, stream);
    if (a.D == 64) return launch_d<64>(a, status, stream);
    return BSA_ERR_UNSUPPORTED;
}

int32_t forward_resident_ctas(int32_t D) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    const int32_t per_sm = D == 128 ? occupancy<128>() : (D == 64 ? occupancy<64>() : -1);
    return per_sm > 0 ? sms * per_sm : -1;
}

}  // namespace bsa
