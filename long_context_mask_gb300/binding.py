"""ctypes binding of libbsa.so (argument marshalling only).

Names mirror the C-ABI in include/bsa.h.  Tensors are torch CUDA tensors; the
binding passes their device pointers, their sizes and the current CUDA
stream.  No arithmetic of the method happens here.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(HERE, "libbsa.so")

BLOCK = 128
IDX_MASK_U8, IDX_THRESHOLD_F32, IDX_TOPK_F32 = 0, 1, 2

STATUS_NAMES = {0: "BSA_OK", 1: "BSA_ERR_INVALID_ARG", 2: "BSA_ERR_UNSUPPORTED",
                3: "BSA_ERR_OVERFLOW", 4: "BSA_ERR_CUDA", 5: "BSA_ERR_TIMEOUT",
                6: "BSA_ERR_BOUNDS"}

EXPORTS = ("bsa_build_index", "bsa_build_crm", "bsa_forward_crm", "bsa_upscale_threshold",
           "bsa_block_scores", "bsa_block_scores_workspace_size",
           "bsa_reorder_rows", "bsa_reorder_guard", "bsa_set_forward_options", "bsa_spectral_order",
           "bsa_spectral_order_workspace_size", "bsa_spectral_order_noalloc", "bsa_sample_blocks",
           "bsa_forward", "bsa_forward_masked", "bsa_forward_packed", "bsa_gather_rows",
           "bsa_gather0_sizes", "bsa_gather0_layout", "bsa_forward_gather0",
           "bsa_forward_scatter",
           "bsa_device_status", "bsa_resident_ctas", "bsa_status_string", "bsa_selftest_exp2",
           "bsa_selftest_wait_timeout")


class BsaError(RuntimeError):
    def __init__(self, call: str, code: int):
        super().__init__(f"{call} failed: {STATUS_NAMES.get(code, code)}")
        self.code = code


_lib = None


def lib_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libbsa.so (raises if it was not built: there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"libbsa.so not found at {_LIB_PATH}; run __graft_entry__.build()")
    lib = ctypes.CDLL(_LIB_PATH)
    P, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    lib.bsa_build_index.argtypes = [i32, P, i64, i32, f32, P, i32, P, P, i32, P]
    lib.bsa_reorder_rows.argtypes = [P, P, i64, i32, i32, P, P]
    lib.bsa_build_crm.argtypes = [i32, P, i64, i32, f32, P, i32, P]
    lib.bsa_build_crm.restype = i32
    lib.bsa_forward_crm.argtypes = [P, P, P, i32, i32, i32, i32, P, i32, P, P, P, f32, P, P, P]
    lib.bsa_forward_crm.restype = i32
    lib.bsa_upscale_threshold.argtypes = [P, i64, i32, i32, i32, i32, P, P]
    lib.bsa_upscale_threshold.restype = i32
    lib.bsa_gather_rows.argtypes = [P, P, i64, i32, i32, P, P]
    lib.bsa_gather_rows.restype = i32
    lib.bsa_block_scores.argtypes = [P, P, i32, i32, i32, i32, P, P, f32, i32, P, ctypes.c_size_t,
                                     P, P]
    lib.bsa_block_scores.restype = i32
    lib.bsa_block_scores_workspace_size.argtypes = [i32, i32, i32, i32]
    lib.bsa_block_scores_workspace_size.restype = ctypes.c_size_t
    lib.bsa_sample_blocks.argtypes = [P, i64, i32, P, P, i32, i32, P, P, P, P, i32, P]
    lib.bsa_spectral_order.argtypes = [P, P, i32, i64, i32, i32, i32, P, P, ctypes.c_size_t, P, P,
                                       P, P]
    lib.bsa_spectral_order_workspace_size.argtypes = [i64, i32, i32]
    lib.bsa_spectral_order_workspace_size.restype = ctypes.c_size_t
    lib.bsa_spectral_order_noalloc.argtypes = [P, P, i32, i64, i32, i32, i32, P, P, P, P, P]
    lib.bsa_spectral_order_noalloc.restype = i32
    lib.bsa_forward.argtypes = [P, P, P, i32, i32, i32, i32, P, P, i32, P, P, P, P, f32, P, P, P]
    lib.bsa_forward_masked.argtypes = [P, P, P, i32, i32, i32, i32, i32, P, P, i32, P, P, P, P,
                                       i32, i32, i32, i32, f32, P, P, P]
    lib.bsa_forward_masked.restype = i32
    lib.bsa_forward_packed.argtypes = [P, P, P, i32, i32, i32, i32, i32, P, P, i32, P, P, P, i32, P,
                                       P, i32, i32, i32, i32, f32, P, P, P]
    lib.bsa_forward_packed.restype = i32
    lib.bsa_gather0_sizes.argtypes = [i32, i32, i32, i32, ctypes.POINTER(i32), ctypes.POINTER(i32),
                                      ctypes.POINTER(i32)]
    lib.bsa_gather0_sizes.restype = i32
    lib.bsa_gather0_layout.argtypes = [i32, i32, i32, i32, i64, P, P, P, P, P, i32, P]
    lib.bsa_gather0_layout.restype = i32
    lib.bsa_forward_gather0.argtypes = [P, P, P, i32, i32, i32, i32, i32, i32, i32, i32, P, P, P, i32,
                                        P, f32, P, P, P]
    lib.bsa_forward_gather0.restype = i32
    lib.bsa_forward_scatter.argtypes = [P, P, P, i32, i32, i32, i32, i32, i32, P, P, i32, P, P, f32, P, P, P]
    lib.bsa_forward_scatter.restype = i32
    lib.bsa_set_forward_options.argtypes = [P]
    lib.bsa_set_forward_options.restype = i32
    lib.bsa_reorder_guard.argtypes = [P, P]
    lib.bsa_reorder_guard.restype = i32
    lib.bsa_device_status.argtypes = [P, ctypes.POINTER(i32)]
    lib.bsa_resident_ctas.argtypes = [i32]
    lib.bsa_status_string.argtypes = [i32]
    lib.bsa_status_string.restype = ctypes.c_char_p
    lib.bsa_selftest_exp2.argtypes = [P, P, P, P, i64, P]
    lib.bsa_selftest_wait_timeout.argtypes = [i64, P]
    for name in ("bsa_build_index", "bsa_reorder_rows", "bsa_spectral_order", "bsa_sample_blocks",
                 "bsa_forward",
                 "bsa_device_status", "bsa_resident_ctas", "bsa_selftest_exp2",
                 "bsa_selftest_wait_timeout"):
        getattr(lib, name).restype = i32
    _lib = lib
    return lib


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(call, code):
    if code != 0:
        raise BsaError(call, code)


def _dtype(t, name, *dtypes):
    if t is not None and t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtypes}")


# The library takes plain pointers, so it cannot see how large a buffer is:
# the checks below reject, before any launch, a buffer smaller than what the
# kernels read or write, an index array of another width, and tensors on
# different devices.  A larger buffer is accepted (only its leading part is
# used).

def _rows(t, name, rows, dtype, cols=None):
    """A 2-D array of `dtype` with at least `rows` rows (and exactly `cols`
    columns when given, i.e. sharing another array's row stride)."""
    if t is None:
        return
    _dtype(t, name, dtype)
    if t.dim() != 2 or t.shape[0] < rows or (cols is not None and t.shape[1] != cols):
        want = "any" if cols is None else cols
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected [>= {rows}, {want}]")


def _flat(t, name, n, dtype):
    """An array of `dtype` with at least `n` entries."""
    if t is None:
        return
    _dtype(t, name, dtype)
    if t.numel() < n:
        raise ValueError(f"{name}: {t.numel()} entries, expected >= {n}")


def _current_device(dev):
    """The library launches on, and keeps its status word for, the current
    CUDA device: tensors elsewhere would be read by another device's kernels."""
    import torch
    if dev.type == "cuda" and dev.index is not None and dev.index != torch.cuda.current_device():
        raise ValueError(f"tensors on {dev} but the current device is cuda:{torch.cuda.current_device()}: "
                         "call torch.cuda.set_device first")


def _same_device(ref, *ts):
    for t in ts:
        if t is not None and t.device != ref.device:
            raise ValueError(f"tensors on {t.device} and {ref.device}: all must be on one device")
    _current_device(ref.device)


def _lists(B, H, N, kv_idx, kv_cnt, log_w=None, row_perm=None, lse=None):
    """The per-row block lists of a forward over B*H heads of N tokens."""
    import torch
    if kv_idx is None or kv_cnt is None:
        raise ValueError("kv_idx and kv_cnt are required")
    rows = B * H * (N // BLOCK)
    _rows(kv_idx, "kv_idx", rows, torch.int32)
    _flat(kv_cnt, "kv_cnt", rows, torch.int32)
    _rows(log_w, "log_w", rows, torch.float32, cols=kv_idx.shape[1])
    _flat(row_perm, "row_perm", rows, torch.int32)
    _flat(lse, "lse", B * H * N, torch.float32)


def build_index(mode: int, src, kv_idx, kv_cnt, *, p: float = 0.0, k_per_row=None,
                k_const: int = 0, stream=None):
    """Fill kv_idx [rows, max_kv] / kv_cnt [rows] from src [rows, nKB] (see bsa.h)."""
    import torch
    _dtype(src, "src", torch.uint8 if mode == IDX_MASK_U8 else torch.float32)
    _dtype(kv_idx, "kv_idx", torch.int32)
    _dtype(kv_cnt, "kv_cnt", torch.int32)
    _dtype(k_per_row, "k_per_row", torch.int32)
    rows, nkb = src.shape
    _rows(kv_idx, "kv_idx", rows, torch.int32)
    _flat(kv_cnt, "kv_cnt", rows, torch.int32)
    _flat(k_per_row, "k_per_row", rows, torch.int32)
    _same_device(src, kv_idx, kv_cnt, k_per_row)
    code = load_library().bsa_build_index(mode, _ptr(src), rows, nkb, float(p), _ptr(k_per_row),
                                          int(k_const), _ptr(kv_idx), _ptr(kv_cnt),
                                          kv_idx.shape[1], _stream(stream))
    _check("bsa_build_index", code)


SCORE_MEAN_DOT, SCORE_CENTROID_EXP = 0, 1


def block_scores(q, k, scores, *, q_map=None, kv_map=None, scale: float = 0.0,
                 mode: int = SCORE_MEAN_DOT, workspace=None, stream=None):
    """scores [B*H*nQB, nKB] fp32 from the block means of Q and K (see bsa.h)."""
    import torch
    _dtype(q, "q", torch.bfloat16)
    _dtype(k, "k", torch.bfloat16)
    _dtype(scores, "scores", torch.float32)
    B, H, N, D = q.shape
    if k.shape != q.shape:
        raise ValueError("q and k must share the shape [B, H, N, D]")
    _flat(scores, "scores", B * H * (N // BLOCK) * (N // BLOCK), torch.float32)
    _flat(q_map, "q_map", B * H * N, torch.int32)
    _flat(kv_map, "kv_map", B * H * N, torch.int32)
    _same_device(q, k, scores, q_map, kv_map, workspace)
    lib = load_library()
    need = int(lib.bsa_block_scores_workspace_size(B, H, N, D))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    nbytes = workspace.numel() * workspace.element_size()
    code = lib.bsa_block_scores(_ptr(q), _ptr(k), B, H, N, D, _ptr(q_map), _ptr(kv_map),
                                float(scale), int(mode), _ptr(workspace), nbytes, _ptr(scores),
                                _stream(stream))
    _check("bsa_block_scores", code)


def build_crm(mode: int, src, words, *, p: float = 0.0, stream=None):
    """CRM rows (uint32 [rows, n_words], viewed as int32 in torch) from a mask /
    threshold map [rows, nKB]."""
    import torch
    _dtype(src, "src", torch.uint8 if mode == IDX_MASK_U8 else torch.float32)
    _dtype(words, "words", torch.int32)
    rows, nkb = src.shape
    _rows(words, "words", rows, torch.int32)
    _same_device(src, words)
    _check("bsa_build_crm", load_library().bsa_build_crm(mode, _ptr(src), rows, nkb, float(p),
                                                         _ptr(words), words.shape[1],
                                                         _stream(stream)))


def forward_crm(q, k, v, crm, o, lse, *, q_map=None, kv_map=None, row_perm=None,
                scale: float = 0.0, stream=None):
    """bsa_forward with CRM rows (int32-viewed uint32 [B*H*nQB, n_words])."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o")):
        _dtype(t, n, torch.bfloat16)
    _dtype(crm, "crm", torch.int32)
    B, H, N, D = q.shape
    if k.shape != q.shape or v.shape != q.shape or o.shape != q.shape:
        raise ValueError("q, k, v, o must share the shape [B, H, N, D]")
    _rows(crm, "crm", B * H * (N // BLOCK), torch.int32)
    _flat(q_map, "q_map", B * H * N, torch.int32)
    _flat(kv_map, "kv_map", B * H * N, torch.int32)
    _flat(row_perm, "row_perm", B * H * (N // BLOCK), torch.int32)
    _flat(lse, "lse", B * H * N, torch.float32)
    _same_device(q, k, v, crm, o, lse, q_map, kv_map, row_perm)
    code = load_library().bsa_forward_crm(_ptr(q), _ptr(k), _ptr(v), B, H, N, D, _ptr(crm),
                                          crm.shape[1], _ptr(q_map), _ptr(kv_map), _ptr(row_perm),
                                          float(scale), _ptr(o), _ptr(lse), _stream(stream))
    _check("bsa_forward_crm", code)


def upscale_threshold(T_base, T_target, *, stream=None):
    """[heads, Ub, Vb] -> [heads, Ut, Vt] threshold maps (eq. 7)."""
    import torch
    _dtype(T_base, "T_base", torch.float32)
    _dtype(T_target, "T_target", torch.float32)
    heads, ub, vb = T_base.shape
    h_out, ut, vt = T_target.shape
    if h_out != heads:
        raise ValueError("T_base and T_target must hold the same number of heads")
    _same_device(T_base, T_target)
    _check("bsa_upscale_threshold", load_library().bsa_upscale_threshold(
        _ptr(T_base), heads, ub, vb, ut, vt, _ptr(T_target), _stream(stream)))


def gather_rows(src, map, dst=None, *, stream=None):
    """dst[h, p] = src[h, map[h, p]] for bf16 [..., N, D] rows (tokens permuted in HBM)."""
    import torch
    _dtype(src, "src", torch.bfloat16)
    _dtype(map, "map", torch.int32)
    N, D = src.shape[-2], src.shape[-1]
    heads = src.numel() // (N * D)
    if dst is None:
        dst = torch.empty_like(src)
    _dtype(dst, "dst", torch.bfloat16)
    if map.numel() != heads * N or dst.shape != src.shape:
        raise ValueError("gather_rows: map must hold heads * N entries and dst match src")
    _same_device(src, map, dst)
    _check("bsa_gather_rows", load_library().bsa_gather_rows(_ptr(src), _ptr(map), heads, N, D,
                                                             _ptr(dst), _stream(stream)))
    return dst


def reorder_rows(kv_cnt, wave: int, row_perm, *, order_in=None, stream=None):
    """row_perm [heads, nQB] from kv_cnt [heads, nQB] (WaveAlign stage 2)."""
    import torch
    _dtype(kv_cnt, "kv_cnt", torch.int32)
    _dtype(row_perm, "row_perm", torch.int32)
    _dtype(order_in, "order_in", torch.int32)
    heads, nqb = kv_cnt.shape
    _flat(row_perm, "row_perm", heads * nqb, torch.int32)
    _flat(order_in, "order_in", heads * nqb, torch.int32)
    _same_device(kv_cnt, row_perm, order_in)
    code = load_library().bsa_reorder_rows(_ptr(kv_cnt), _ptr(order_in), heads, nqb, int(wave),
                                           _ptr(row_perm), _stream(stream))
    _check("bsa_reorder_rows", code)


def _spectral_args(heads, nqb, kv_idx, kv_cnt, x0, x_out, angle):
    import torch
    _rows(kv_idx, "kv_idx", heads * nqb, torch.int32)
    _flat(kv_cnt, "kv_cnt", heads * nqb, torch.int32)
    _flat(x0, "x0", heads * nqb * 2, torch.float32)
    _flat(x_out, "x_out", heads * nqb * 2, torch.float32)
    _flat(angle, "angle", heads * nqb, torch.float32)


def spectral_order_workspace_size(heads: int, nqb: int, nkb: int) -> int:
    return int(load_library().bsa_spectral_order_workspace_size(heads, nqb, nkb))


def spectral_order(kv_idx, kv_cnt, n_kb: int, x0, order, *, workspace=None, x_out=None,
                   angle=None, iters: int = 10, stream=None):
    """Row order from the rank-2 centered-mask embedding (WaveAlign section IV-C).

    kv_idx [heads*nQB, max_kv], kv_cnt [heads*nQB]; x0 fp32 [heads, nQB, 2];
    order int32 [heads, nQB] out (optional x_out like x0, angle [heads, nQB]).
    ``workspace`` is a CUDA tensor of at least spectral_order_workspace_size()
    bytes (allocated here through torch when omitted)."""
    import torch
    _dtype(x0, "x0", torch.float32)
    _dtype(order, "order", torch.int32)
    heads, nqb = order.shape
    _spectral_args(heads, nqb, kv_idx, kv_cnt, x0, x_out, angle)
    _same_device(order, kv_idx, kv_cnt, x0, x_out, angle, workspace)
    need = spectral_order_workspace_size(heads, nqb, n_kb)
    if workspace is None:
        workspace = torch.empty(max(need, 8), dtype=torch.uint8, device=order.device)
    nbytes = workspace.numel() * workspace.element_size()
    code = load_library().bsa_spectral_order(_ptr(kv_idx), _ptr(kv_cnt), kv_idx.shape[1], heads,
                                             nqb, int(n_kb), int(iters), _ptr(x0),
                                             _ptr(workspace), nbytes, _ptr(x_out), _ptr(angle),
                                             _ptr(order), _stream(stream))
    _check("bsa_spectral_order", code)


NOALLOC_SCRATCH_BYTES = 4 << 20


def spectral_order_noalloc(kv_idx, kv_cnt, n_kb: int, x0, order, *, x_out=None, angle=None,
                           iters: int = 10, stream=None):
    """spectral_order for callers that cannot allocate device memory: the
    library's own fixed scratch array replaces the workspace (see bsa.h)."""
    import torch
    _dtype(x0, "x0", torch.float32)
    _dtype(order, "order", torch.int32)
    heads, nqb = order.shape
    _spectral_args(heads, nqb, kv_idx, kv_cnt, x0, x_out, angle)
    _same_device(order, kv_idx, kv_cnt, x0, x_out, angle)
    code = load_library().bsa_spectral_order_noalloc(_ptr(kv_idx), _ptr(kv_cnt), kv_idx.shape[1],
                                                     heads, nqb, int(n_kb), int(iters), _ptr(x0),
                                                     _ptr(x_out), _ptr(angle), _ptr(order),
                                                     _stream(stream))
    _check("bsa_spectral_order_noalloc", code)


class GuardArgs(ctypes.Structure):
    _fields_ = [("heads", ctypes.c_int64), ("kv_heads", ctypes.c_int64), ("nQB", ctypes.c_int32),
                ("nKB", ctypes.c_int32), ("D", ctypes.c_int32), ("listed_blocks", ctypes.c_int64),
                ("l2_bytes", ctypes.c_double), ("tensor_tflops", ctypes.c_double),
                ("hbm_gbs", ctypes.c_double), ("wave_ms", ctypes.c_double),
                ("spectral_ms", ctypes.c_double)]


class GuardResult(ctypes.Structure):
    _fields_ = [("order", ctypes.c_int32), ("kv_head_bytes", ctypes.c_double),
                ("kv_cache_bytes", ctypes.c_double), ("miss_fraction", ctypes.c_double),
                ("t_input_ms", ctypes.c_double), ("t_wave_ms", ctypes.c_double),
                ("t_spectral_ms", ctypes.c_double), ("wave_cost_ms", ctypes.c_double),
                ("spectral_cost_ms", ctypes.c_double)]


class ForwardOptions(ctypes.Structure):
    _fields_ = [("schedule", ctypes.c_int32), ("exp2_fma", ctypes.c_int32)]


SCHEDULES = {"auto": 0, "per_row": 1, "per_item": 2}


def set_forward_options(schedule: str = "auto", exp2_fma: int = 0):
    """bsa_set_forward_options for this host thread: the launch schedule of
    later forward calls ("auto", "per_row", "per_item") and how many
    exponentials of every 8 the plain tile path takes on the FMA pipe (0, 2)."""
    o = ForwardOptions(SCHEDULES[schedule], int(exp2_fma))
    _check("bsa_set_forward_options", load_library().bsa_set_forward_options(ctypes.byref(o)))


ORDER_NAMES = {0: "input", 1: "wave", 2: "spectral"}


def reorder_guard(*, heads: int, nqb: int, nkb: int, D: int, listed_blocks: int, kv_heads=None,
                  l2_bytes: float = 0.0, tensor_tflops: float = 0.0, hbm_gbs: float = 0.0,
                  wave_ms: float = -1.0, spectral_ms: float = -1.0) -> dict:
    """bsa_reorder_guard: which row order pays for this forward call ("input",
    "wave" or "spectral") and the estimates behind the choice (see bsa.h)."""
    a = GuardArgs(heads, heads if kv_heads is None else kv_heads, nqb, nkb, D, int(listed_blocks),
                  float(l2_bytes), float(tensor_tflops), float(hbm_gbs), float(wave_ms),
                  float(spectral_ms))
    r = GuardResult()
    _check("bsa_reorder_guard", load_library().bsa_reorder_guard(ctypes.byref(a), ctypes.byref(r)))
    out = {f: getattr(r, f) for f, _ in GuardResult._fields_}
    out["order"] = ORDER_NAMES[r.order]
    return out


def sample_blocks(scores, exact_idx, exact_cnt, m: int, u, kv_idx, kv_cnt, log_w, *, nkb=None,
                  stream=None):
    """Exact list + PPSWOR sample with log-weights (InstaGen section 3.2.1).
    scores None selects the uniform sampler (then pass nkb)."""
    import torch
    _dtype(scores, "scores", torch.float32)
    _dtype(u, "u", torch.float64)
    if scores is None:
        rows = exact_cnt.shape[0]
        if nkb is None:
            raise ValueError("sample_blocks: pass nkb with the uniform sampler (scores None)")
    else:
        rows, nkb = scores.shape
    _rows(exact_idx, "exact_idx", rows, torch.int32)
    _flat(exact_cnt, "exact_cnt", rows, torch.int32)
    _flat(u, "u", rows, torch.float64)
    if kv_idx is None or kv_cnt is None or log_w is None:
        raise ValueError("kv_idx, kv_cnt and log_w are required")
    _rows(kv_idx, "kv_idx", rows, torch.int32)
    _flat(kv_cnt, "kv_cnt", rows, torch.int32)
    _rows(log_w, "log_w", rows, torch.float32, cols=kv_idx.shape[1])
    _same_device(exact_idx, scores, exact_cnt, u, kv_idx, kv_cnt, log_w)
    code = load_library().bsa_sample_blocks(_ptr(scores), rows, nkb, _ptr(exact_idx),
                                            _ptr(exact_cnt), exact_idx.shape[1], int(m), _ptr(u),
                                            _ptr(kv_idx), _ptr(kv_cnt), _ptr(log_w),
                                            kv_idx.shape[1], _stream(stream))
    _check("bsa_sample_blocks", code)


def forward(q, k, v, kv_idx, kv_cnt, o, lse, *, log_w=None, q_map=None, kv_map=None,
            row_perm=None, scale: float = 0.0, stream=None):
    """Block-sparse attention forward: fills o [B,H,N,D] bf16 and lse [B,H,N] fp32."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o")):
        _dtype(t, n, torch.bfloat16)
    _dtype(lse, "lse", torch.float32)
    _dtype(log_w, "log_w", torch.float32)
    B, H, N, D = q.shape
    if k.shape != q.shape or v.shape != q.shape or o.shape != q.shape:
        raise ValueError("q, k, v, o must share the shape [B, H, N, D]")
    _lists(B, H, N, kv_idx, kv_cnt, log_w, row_perm, lse)
    _flat(q_map, "q_map", B * H * N, torch.int32)
    _flat(kv_map, "kv_map", B * H * N, torch.int32)
    _same_device(q, k, v, o, lse, kv_idx, kv_cnt, log_w, q_map, kv_map, row_perm)
    code = load_library().bsa_forward(_ptr(q), _ptr(k), _ptr(v), B, H, N, D, _ptr(kv_idx),
                                      _ptr(kv_cnt), kv_idx.shape[1], _ptr(log_w), _ptr(q_map),
                                      _ptr(kv_map), _ptr(row_perm), float(scale), _ptr(o),
                                      _ptr(lse), _stream(stream))
    _check("bsa_forward", code)


def forward_masked(q, k, v, kv_idx, kv_cnt, o, lse, *, causal: bool = False, n_valid: int = 0,
                   window: int = 0, sinks: int = 0, log_w=None, q_map=None, kv_map=None,
                   row_perm=None, scale: float = 0.0, stream=None):
    """bsa_forward with grouped K/V heads (k, v [B, H_kv, N, D]) and a token mask (see bsa.h)."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o")):
        _dtype(t, n, torch.bfloat16)
    _dtype(lse, "lse", torch.float32)
    _dtype(log_w, "log_w", torch.float32)
    B, H, N, D = q.shape
    H_kv = k.shape[1]
    if k.shape != (B, H_kv, N, D) or v.shape != k.shape or o.shape != q.shape:
        raise ValueError("q, o [B, H, N, D]; k, v [B, H_kv, N, D]")
    _lists(B, H, N, kv_idx, kv_cnt, log_w, row_perm, lse)
    _flat(q_map, "q_map", B * H * N, torch.int32)
    _flat(kv_map, "kv_map", B * H_kv * N, torch.int32)
    _same_device(q, k, v, o, lse, kv_idx, kv_cnt, log_w, q_map, kv_map, row_perm)
    code = load_library().bsa_forward_masked(
        _ptr(q), _ptr(k), _ptr(v), B, H, H_kv, N, D, _ptr(kv_idx), _ptr(kv_cnt), kv_idx.shape[1],
        _ptr(log_w), _ptr(q_map), _ptr(kv_map), _ptr(row_perm), int(bool(causal)), int(n_valid),
        int(window), int(sinks), float(scale), _ptr(o), _ptr(lse), _stream(stream))
    _check("bsa_forward_masked", code)


def forward_packed(q, k, v, kv_idx, kv_cnt, kv_map, o, lse, *, quad_mask=None, causal: bool = False,
                   n_valid: int = 0, window: int = 0, sinks: int = 0, log_w=None, q_map=None,
                   row_perm=None, scale: float = 0.0, stream=None):
    """bsa_forward_masked over key tiles packed through kv_map [B*H_kv, N_kv]
    (tokens may repeat across tiles) with optional quad_mask uint8
    [B*H*nQB, max_kv] (see bsa.h)."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o")):
        _dtype(t, n, torch.bfloat16)
    _dtype(lse, "lse", torch.float32)
    _dtype(log_w, "log_w", torch.float32)
    _dtype(quad_mask, "quad_mask", torch.uint8)
    B, H, N, D = q.shape
    H_kv = k.shape[1]
    if k.shape != (B, H_kv, N, D) or v.shape != k.shape or o.shape != q.shape:
        raise ValueError("q, o [B, H, N, D]; k, v [B, H_kv, N, D]")
    if kv_map is None:
        raise ValueError("forward_packed needs kv_map")
    N_kv = kv_map.shape[-1]
    if quad_mask is not None and tuple(quad_mask.shape) != tuple(kv_idx.shape):
        raise ValueError("quad_mask must have kv_idx's shape")
    _lists(B, H, N, kv_idx, kv_cnt, log_w, row_perm, lse)
    _flat(q_map, "q_map", B * H * N, torch.int32)
    _flat(kv_map, "kv_map", B * H_kv * N_kv, torch.int32)
    _same_device(q, k, v, o, lse, kv_idx, kv_cnt, log_w, q_map, kv_map, quad_mask, row_perm)
    code = load_library().bsa_forward_packed(
        _ptr(q), _ptr(k), _ptr(v), B, H, H_kv, N, D, _ptr(kv_idx), _ptr(kv_cnt), kv_idx.shape[1],
        _ptr(log_w), _ptr(q_map), _ptr(kv_map), int(N_kv), _ptr(quad_mask), _ptr(row_perm),
        int(bool(causal)), int(n_valid), int(window), int(sinks), float(scale), _ptr(o), _ptr(lse),
        _stream(stream))
    _check("bsa_forward_packed", code)


def gather0_sizes(img_h: int, img_w: int, n_text: int = 0, groups: int = 1):
    """(N, N_kv, max_kv) of the INTRA Gather 0 layout (host only)."""
    N, N_kv, mk = ctypes.c_int32(0), ctypes.c_int32(0), ctypes.c_int32(0)
    _check("bsa_gather0_sizes", load_library().bsa_gather0_sizes(
        img_h, img_w, n_text, groups, ctypes.byref(N), ctypes.byref(N_kv), ctypes.byref(mk)))
    return N.value, N_kv.value, mk.value


def gather0_layout(img_h: int, img_w: int, n_text: int, groups: int, heads: int, *, device=None,
                   stream=None):
    """The INTRA Gather 0 layer's q_map [heads, N], kv_map [heads, N_kv],
    kv_idx / quad_mask [heads*N/128, max_kv] and kv_cnt, built on the GPU."""
    import torch
    N, N_kv, max_kv = gather0_sizes(img_h, img_w, n_text, groups)
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    _current_device(dev)
    rows = heads * (N // BLOCK)
    q_map = torch.empty((heads, N), dtype=torch.int32, device=dev)
    kv_map = torch.empty((heads, N_kv), dtype=torch.int32, device=dev)
    kv_idx = torch.empty((rows, max_kv), dtype=torch.int32, device=dev)
    kv_cnt = torch.empty(rows, dtype=torch.int32, device=dev)
    quad_mask = torch.empty((rows, max_kv), dtype=torch.uint8, device=dev)
    _check("bsa_gather0_layout", load_library().bsa_gather0_layout(
        img_h, img_w, n_text, groups, heads, _ptr(q_map), _ptr(kv_map), _ptr(kv_idx), _ptr(kv_cnt),
        _ptr(quad_mask), max_kv, _stream(stream)))
    return q_map, kv_map, kv_idx, kv_cnt, quad_mask


def forward_gather0(q, k, v, img_h: int, img_w: int, n_text: int, groups: int, kv_idx, kv_cnt, o, lse,
                    *, quad_mask=None, row_perm=None, scale: float = 0.0, stream=None):
    """The INTRA Gather 0 layer with tiles fetched by geometry (see bsa.h);
    kv_idx / kv_cnt / quad_mask from gather0_layout."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o")):
        _dtype(t, n, torch.bfloat16)
    _dtype(lse, "lse", torch.float32)
    _dtype(quad_mask, "quad_mask", torch.uint8)
    B, H, N, D = q.shape
    H_kv = k.shape[1]
    if k.shape != (B, H_kv, N, D) or v.shape != k.shape or o.shape != q.shape:
        raise ValueError("q, o [B, H, N, D]; k, v [B, H_kv, N, D]")
    if N != n_text + img_h * img_w:
        raise ValueError("N must be n_text + img_h * img_w")
    _lists(B, H, N, kv_idx, kv_cnt, None, row_perm, lse)
    _rows(quad_mask, "quad_mask", B * H * (N // BLOCK), torch.uint8, cols=kv_idx.shape[1])
    _same_device(q, k, v, o, lse, kv_idx, kv_cnt, quad_mask, row_perm)
    code = load_library().bsa_forward_gather0(
        _ptr(q), _ptr(k), _ptr(v), B, H, H_kv, D, img_h, img_w, n_text, groups, _ptr(kv_idx),
        _ptr(kv_cnt), _ptr(quad_mask), kv_idx.shape[1], _ptr(row_perm), float(scale), _ptr(o),
        _ptr(lse), _stream(stream))
    _check("bsa_forward_gather0", code)


def forward_scatter(q, k, v, R: int, kv_idx, kv_cnt, o, lse, *, log_w=None, row_perm=None,
                    scale: float = 0.0, stream=None):
    """The Scatter layer with tiles fetched by geometry (see bsa.h): lists over
    gathered blocks, p = r*T + t holding token t*R + r."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o")):
        _dtype(t, n, torch.bfloat16)
    _dtype(lse, "lse", torch.float32)
    _dtype(log_w, "log_w", torch.float32)
    B, H, N, D = q.shape
    H_kv = k.shape[1]
    if k.shape != (B, H_kv, N, D) or v.shape != k.shape or o.shape != q.shape:
        raise ValueError("q, o [B, H, N, D]; k, v [B, H_kv, N, D]")
    _lists(B, H, N, kv_idx, kv_cnt, log_w, row_perm, lse)
    _same_device(q, k, v, o, lse, kv_idx, kv_cnt, log_w, row_perm)
    code = load_library().bsa_forward_scatter(
        _ptr(q), _ptr(k), _ptr(v), B, H, H_kv, N, D, int(R), _ptr(kv_idx), _ptr(kv_cnt),
        kv_idx.shape[1], _ptr(log_w), _ptr(row_perm), float(scale), _ptr(o), _ptr(lse), _stream(stream))
    _check("bsa_forward_scatter", code)


def device_status(stream=None) -> int:
    """Read and clear the device status word (synchronises the stream)."""
    out = ctypes.c_int32(0)
    _check("bsa_device_status", load_library().bsa_device_status(_stream(stream), ctypes.byref(out)))
    return out.value


def selftest_exp2(x, *, stream=None):
    """(y_fma, y_mufu, y_ref) = the three device 2^x of bsa_selftest.h for fp32 x."""
    import torch
    _dtype(x, "x", torch.float32)
    outs = [torch.empty_like(x) for _ in range(3)]
    _check("bsa_selftest_exp2", load_library().bsa_selftest_exp2(
        _ptr(x), *(_ptr(o) for o in outs), x.numel(), _stream(stream)))
    return tuple(outs)


def selftest_wait_timeout(limit_ns: int, *, stream=None):
    """Launch the bounded-wait self-test (records BSA_ERR_TIMEOUT on expiry)."""
    _check("bsa_selftest_wait_timeout",
           load_library().bsa_selftest_wait_timeout(int(limit_ns), _stream(stream)))


def resident_ctas(D: int) -> int:
    n = load_library().bsa_resident_ctas(int(D))
    if n <= 0:
        raise BsaError("bsa_resident_ctas", 4)
    return n


def effective_flops(kv_cnt, D: int) -> float:
    """FLOPs of the computed blocks: sum(cnt) * 4 * 128 * 128 * D (QK^T and PV)."""
    total = int(kv_cnt.sum().item()) if hasattr(kv_cnt, "sum") else int(sum(kv_cnt))
    return float(total) * 4.0 * BLOCK * BLOCK * D


def dense_attention_flops(N: int, H: int, D: int, causal: bool = False, B: int = 1) -> float:
    """4 N^2 D per head (two N x N x D products), halved for causal attention."""
    f = 4.0 * N * N * D * H * B
    return f / 2 if causal else f


__all__ = ["BLOCK", "BsaError", "IDX_MASK_U8", "IDX_THRESHOLD_F32", "IDX_TOPK_F32", "build_index",
           "reorder_rows", "sample_blocks", "forward", "device_status", "resident_ctas",
           "effective_flops", "dense_attention_flops", "load_library", "lib_path", "EXPORTS",
           "block_scores", "SCORE_MEAN_DOT", "SCORE_CENTROID_EXP", "build_crm", "forward_crm",
           "upscale_threshold", "gather_rows", "forward_masked", "forward_packed", "forward_gather0", "forward_scatter", "gather0_sizes",
           "gather0_layout",
           "spectral_order", "spectral_order_workspace_size", "spectral_order_noalloc",
           "NOALLOC_SCRATCH_BYTES", "reorder_guard", "set_forward_options",
           "selftest_exp2", "selftest_wait_timeout"]
