"""Block-sparse attention oracle (fp64 CPU reference).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  The product path (the CUDA library and
its binding) never imports this package, and this package never imports the
product path.  Every function wraps the plain C in ``bsa_oracle.c`` through
ctypes and takes/returns numpy arrays.  The passages each function follows are
listed at the top of ``bsa_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bsa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

# -ffp-contract=off: the sampler's integer decisions come from fp64 sums that
# must round exactly as written (no fused multiply-add), on x86 and on Arm.
CFLAGS = ["-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-std=c11"]


def build(force: bool = False) -> str:
    """Compile bsa_oracle.c into liboracle.so next to it (gcc, no GPU)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        # ORACLE_LIB_OVERRIDE: a library built from a deliberately altered copy
        # of bsa_oracle.c, used by the tests that check the pins catch it
        override = os.environ.get("ORACLE_LIB_OVERRIDE")
        if not override:
            build()
        lib = ctypes.CDLL(override or _LIB)
        P = ctypes.c_void_p
        i32, i64, f32, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_double
        lib.oracle_index_mask_u8.argtypes = [P, i64, i32, P, P, i32]
        lib.oracle_index_mask_u8.restype = i64
        lib.oracle_index_threshold.argtypes = [P, i64, i32, f32, P, P, i32]
        lib.oracle_index_threshold.restype = i64
        lib.oracle_index_topk.argtypes = [P, i64, i32, P, i32, P, P, i32]
        lib.oracle_index_topk.restype = i64
        lib.oracle_reorder_rows.argtypes = [P, P, i64, i32, i32, P]
        lib.oracle_reorder_rows.restype = None
        lib.oracle_sample_blocks.argtypes = [P, i64, i32, P, P, i32, i32, P, P, P, P, i32]
        lib.oracle_sample_blocks.restype = i64
        lib.oracle_attention.argtypes = [P, P, P, i32, i32, i32, i32, i32, P, P, i32, P, P, P,
                                         i32, i32, i32, i32, f64, P, i64, P, P, P]
        lib.oracle_attention.restype = None
        lib.oracle_crm_rows.argtypes = [i32, P, i64, i32, f32, P, i32]
        lib.oracle_crm_rows.restype = None
        lib.oracle_upscale_threshold.argtypes = [P, i64, i32, i32, i32, i32, P]
        lib.oracle_upscale_threshold.restype = None
        lib.oracle_block_scores.argtypes = [P, P, i32, i32, i32, i32, P, P, f64, i32, P]
        lib.oracle_block_scores.restype = None
        lib.oracle_spectral_order.argtypes = [P, P, i32, i64, i32, i32, i32, P, P, P, P]
        lib.oracle_spectral_order.restype = None
        lib.oracle_gather0_set.argtypes = [i32, i32, i32, i32, i64, P, P, P]
        lib.oracle_gather0_set.restype = i64
        lib.oracle_attention_set.argtypes = [P, P, P, i32, i32, i64, i64, i64, P, i64, P, f64, P, P]
        lib.oracle_attention_set.restype = None
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = i32
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def index_mask(mask, max_kv=None):
    """mask uint8 [rows, nKB] -> (kv_idx int32 [rows, max_kv], kv_cnt int32 [rows], n_overflow)."""
    mask = _c(mask, np.uint8)
    rows, nkb = mask.shape
    max_kv = nkb if max_kv is None else int(max_kv)
    idx = np.empty((rows, max_kv), np.int32)
    cnt = np.empty(rows, np.int32)
    ov = _load().oracle_index_mask_u8(_ptr(mask), rows, nkb, _ptr(idx), _ptr(cnt), max_kv)
    return idx, cnt, int(ov)


def index_threshold(T, p, max_kv=None):
    """Threshold map fp32 [rows, nKB], keep T <= p (fp32) -> (kv_idx, kv_cnt, n_overflow)."""
    T = _c(T, np.float32)
    rows, nkb = T.shape
    max_kv = nkb if max_kv is None else int(max_kv)
    idx = np.empty((rows, max_kv), np.int32)
    cnt = np.empty(rows, np.int32)
    ov = _load().oracle_index_threshold(_ptr(T), rows, nkb, float(np.float32(p)), _ptr(idx),
                                        _ptr(cnt), max_kv)
    return idx, cnt, int(ov)


def index_topk(scores, k, max_kv=None):
    """Top-k per row (score desc, ties to the lower block), listed in ascending block order.

    ``k`` is an int or an int32 array [rows]."""
    scores = _c(scores, np.float32)
    rows, nkb = scores.shape
    if np.isscalar(k):
        kpr, kc = None, int(k)
        kmax = kc
    else:
        kpr, kc = _c(k, np.int32), 0
        kmax = int(kpr.max()) if rows else 0
    max_kv = min(nkb, kmax) if max_kv is None else int(max_kv)
    max_kv = max(max_kv, 1)
    idx = np.empty((rows, max_kv), np.int32)
    cnt = np.empty(rows, np.int32)
    ov = _load().oracle_index_topk(_ptr(scores), rows, nkb, _ptr(kpr), kc, _ptr(idx), _ptr(cnt),
                                   max_kv)
    return idx, cnt, int(ov)


def reorder_rows(kv_cnt, wave, order_in=None):
    """kv_cnt int32 [heads, nQB] -> row_perm int32 [heads, nQB] (WaveAlign stage 2)."""
    kv_cnt = _c(kv_cnt, np.int32)
    heads, nqb = kv_cnt.shape
    order_in = _c(order_in, np.int32)
    perm = np.empty((heads, nqb), np.int32)
    _load().oracle_reorder_rows(_ptr(kv_cnt), _ptr(order_in), heads, nqb, int(wave), _ptr(perm))
    return perm


def sample_blocks(scores, exact_idx, exact_cnt, m, u, max_kv, nkb=None):
    """Exact list + PPSWOR/systematic-PPS sample -> (kv_idx, kv_cnt, log_w, n_overflow).

    scores None selects the uniform sampler (pass nkb and rows via exact_cnt)."""
    if scores is None:
        rows = len(exact_cnt)
    else:
        scores = _c(scores, np.float32)
        rows, nkb = scores.shape
    exact_idx = _c(exact_idx, np.int32)
    exact_cnt = _c(exact_cnt, np.int32)
    u = _c(u, np.float64)
    idx = np.empty((rows, max_kv), np.int32)
    cnt = np.empty(rows, np.int32)
    lw = np.empty((rows, max_kv), np.float32)
    ov = _load().oracle_sample_blocks(_ptr(scores), rows, int(nkb), _ptr(exact_idx), _ptr(exact_cnt),
                                      exact_idx.shape[1], int(m), _ptr(u), _ptr(idx), _ptr(cnt),
                                      _ptr(lw), int(max_kv))
    return idx, cnt, lw, int(ov)


def crm_rows(src, p=None):
    """CRM rows: uint32 [rows, ceil(nKB/32)], bit i of word w = block 32w+i kept.
    src uint8 mask (nonzero keeps) or fp32 threshold map with p (T <= p keeps)."""
    src = np.ascontiguousarray(src)
    rows, nkb = src.shape
    nw = (nkb + 31) // 32
    out = np.empty((rows, nw), np.uint32)
    mode = 0 if src.dtype == np.uint8 else 1
    if mode == 1:
        src = src.astype(np.float32)
    _load().oracle_crm_rows(mode, _ptr(src), rows, nkb, float(np.float32(p or 0.0)), _ptr(out), nw)
    return out


def upscale_threshold(T, Ut, Vt):
    """Threshold maps fp32 [heads, Ub, Vb] -> [heads, Ut, Vt] (eq. 7 reading)."""
    T = _c(T, np.float32)
    heads, ub, vb = T.shape
    out = np.empty((heads, Ut, Vt), np.float32)
    _load().oracle_upscale_threshold(_ptr(T), heads, ub, vb, int(Ut), int(Vt), _ptr(out))
    return out


def block_scores(q, k, q_map=None, kv_map=None, scale=0.0, mode=0):
    """Scores [B*H*nQB, nKB] (fp64) from the block means of Q and K (mode 0:
    scaled dot product, mode 1: its exponential, the centroid score)."""
    q, k = _as_u16(q), _as_u16(k)
    B, H, N, D = q.shape
    nb = N // 128
    out = np.empty((B * H * nb, nb), np.float64)
    _load().oracle_block_scores(_ptr(q), _ptr(k), B, H, N, D, _ptr(_c(q_map, np.int32)),
                                _ptr(_c(kv_map, np.int32)), float(scale), int(mode), _ptr(out))
    return out


def spectral_order(kv_idx, kv_cnt, n_kb, x0, iters):
    """WaveAlign stage 1 per head: (X [heads, nQB, 2], angle [heads, nQB], order [heads, nQB]).

    kv_idx [heads*nQB, max_kv], kv_cnt [heads*nQB]; x0 fp64 [heads, nQB, 2]."""
    kv_idx = _c(kv_idx, np.int32)
    kv_cnt = _c(kv_cnt, np.int32)
    x0 = _c(x0, np.float64)
    heads, nqb = x0.shape[0], x0.shape[1]
    X = np.empty((heads, nqb, 2), np.float64)
    ang = np.empty((heads, nqb), np.float64)
    order = np.empty((heads, nqb), np.int32)
    _load().oracle_spectral_order(_ptr(kv_idx), _ptr(kv_cnt), kv_idx.shape[1], heads, nqb,
                                  int(n_kb), int(iters), _ptr(x0), _ptr(X), _ptr(ang),
                                  _ptr(order))
    return X, ang, order


def attention(q, k, v, kv_idx, kv_cnt, log_w=None, q_map=None, kv_map=None, scale=0.0,
              sel=None, causal=False, n_valid=0, window=0, sinks=0):
    """Block-sparse attention from the definition, fp64.

    q: uint16 bf16 bit patterns [B, H, N, D] (or a torch bf16 tensor on CPU);
    k, v: [B, H_kv, N, D] with H a multiple of H_kv (grouped heads).
    kv_idx [B*H*nQB, max_kv], kv_cnt [B*H*nQB]; log_w like kv_idx or None;
    q_map int32 [B*H, N] or None; kv_map int32 [B*H_kv, N] or None.
    Token mask: key j is dropped for query i unless j < n_valid (n_valid <= 0:
    N), (not causal or j <= i) and (window <= 0 or j > i - window or j < sinks).
    ``sel`` lists the flat query blocks (bh * nQB + qb) to evaluate (all when None).
    Returns (O fp64 [nsel*128, D], LSE fp64 [nsel*128], tok int32 [nsel*128]),
    where row x belongs to original query token tok[x] of head sel[x // 128] // nQB.
    """
    q, k, v = (_as_u16(t) for t in (q, k, v))
    B, H, N, D = q.shape
    H_kv = k.shape[1]
    if H % H_kv or k.shape != v.shape or k.shape[0] != B or k.shape[2:] != (N, D):
        raise ValueError("attention: k, v must be [B, H_kv, N, D] with H a multiple of H_kv")
    nqb = N // 128
    kv_idx = _c(kv_idx, np.int32)
    kv_cnt = _c(kv_cnt, np.int32)
    max_kv = kv_idx.shape[1]
    log_w = _c(log_w, np.float32)
    q_map = _c(q_map, np.int32)
    kv_map = _c(kv_map, np.int32)
    sel = np.arange(B * H * nqb, dtype=np.int64) if sel is None else _c(sel, np.int64)
    n = sel.shape[0]
    O = np.empty((n * 128, D), np.float64)
    L = np.empty(n * 128, np.float64)
    tok = np.empty(n * 128, np.int32)
    _load().oracle_attention(_ptr(q), _ptr(k), _ptr(v), B, H, H_kv, N, D, _ptr(kv_idx),
                             _ptr(kv_cnt), max_kv, _ptr(log_w), _ptr(q_map), _ptr(kv_map),
                             int(bool(causal)), int(n_valid), int(window), int(sinks),
                             float(scale), _ptr(sel), n, _ptr(O), _ptr(L), _ptr(tok))
    return O, L, tok


def gather0_sets(img_h, img_w, n_text, groups):
    """Query and key token sets of the INTRA Gather 0 layer.

    Returns a list of (q_tok, k_tok) int32 arrays: the img_h*img_w/64 image
    CQS in the page's order (8 x 8 query patch; text keys, then the clamped
    16 x 16 window), then, when n_text > 0, the text queries of each of the
    ``groups`` Scatter groups (text keys, then the group's image tokens).
    """
    hw = img_h * img_w
    n_sets = hw // 64 + (groups if n_text > 0 else 0)
    per = n_text // groups if n_text > 0 else 0
    qcap = max(64, per)
    kcap = n_text + max(256, hw // groups if n_text > 0 else 0)
    lib = _load()
    out = []
    for sidx in range(n_sets):
        qt = np.empty(qcap, np.int32)
        kt = np.empty(kcap, np.int32)
        nq = np.zeros(1, np.int64)
        nk = lib.oracle_gather0_set(img_h, img_w, n_text, groups, sidx, _ptr(qt), _ptr(nq), _ptr(kt))
        if nk < 0:
            raise ValueError("gather0_sets: set index out of range")
        out.append((qt[: int(nq[0])].copy(), kt[:nk].copy()))
    return out


def attention_set(q, k, v, bh, q_tok, k_tok, scale=0.0):
    """Softmax attention of query tokens q_tok of query head bh (flat b*H + h)
    over key tokens k_tok, fp64.  q [B, H, N, D], k/v [B, H_kv, N, D] (bf16
    bit patterns or CPU bf16 tensors).  Returns (O [nq, D], LSE [nq])."""
    q, k, v = (_as_u16(t) for t in (q, k, v))
    B, H, N, D = q.shape
    H_kv = k.shape[1]
    kvh = (bh // H) * H_kv + (bh % H) // (H // H_kv)
    q_tok = _c(q_tok, np.int32)
    k_tok = _c(k_tok, np.int32)
    O = np.empty((q_tok.shape[0], D), np.float64)
    L = np.empty(q_tok.shape[0], np.float64)
    _load().oracle_attention_set(_ptr(q), _ptr(k), _ptr(v), N, D, int(bh), int(kvh),
                                 q_tok.shape[0], _ptr(q_tok), k_tok.shape[0], _ptr(k_tok),
                                 float(scale), _ptr(O), _ptr(L))
    return O, L


def gather0_attention(q, k, v, img_h, img_w, n_text, groups, scale=0.0, heads=None, sets=None):
    """The INTRA Gather 0 layer from its definition, fp64.

    q [B, H, N, D] with N = n_text + img_h*img_w; k, v [B, H_kv, N, D].
    ``heads`` lists flat query heads (all when None) and ``sets`` indexes
    gather0_sets (all when None).  Returns (O [len(heads), N, D], LSE
    [len(heads), N]); rows of query tokens outside the chosen sets are NaN.
    """
    q_u = _as_u16(q)
    B, H, N, D = q_u.shape
    all_sets = gather0_sets(img_h, img_w, n_text, groups)
    chosen = range(len(all_sets)) if sets is None else sets
    heads = range(B * H) if heads is None else heads
    O = np.full((len(heads), N, D), np.nan)
    L = np.full((len(heads), N), np.nan)
    for hi, bh in enumerate(heads):
        for sidx in chosen:
            qt, kt = all_sets[sidx]
            o, lse = attention_set(q_u, k, v, bh, qt, kt, scale)
            O[hi, qt] = o
            L[hi, qt] = lse
    return O, L


def _as_u16(t):
    if hasattr(t, "view") and hasattr(t, "dtype") and "bfloat16" in str(t.dtype):
        t = t.contiguous().view(__import__("torch").int16).numpy()
    return np.ascontiguousarray(t).view(np.uint16)
