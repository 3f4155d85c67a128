"""The Python binding's argument checks (no GPU).

The C-ABI takes plain pointers and cannot see how large a buffer is, so the
binding rejects, before any launch, buffers smaller than what the kernels
touch, index arrays of another dtype, and tensors on different devices or
not on the current device.
With CPU tensors every accepted call stops at the binding's "expected a CUDA
tensor" step, so the tests tell an accepted call (that message) from a
rejected one (any other error).  The accepted shapes are the ones the GPU
tests and the benchmark pass: grouped heads with the first B*H_kv map rows,
larger-than-needed capacities, views of the count array.
"""
import pytest
import torch

import long_context_mask_gb300 as bsa
from long_context_mask_gb300 import build as bsa_build

CUDA_STEP = "expected a CUDA tensor"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    bsa_build.build()
    bsa.load_library()


def accepted(fn, *a, **kw):
    with pytest.raises(ValueError, match=CUDA_STEP):
        fn(*a, **kw)


def rejected(fn, *a, match=None, **kw):
    with pytest.raises((ValueError, TypeError)) as e:
        fn(*a, **kw)
    assert CUDA_STEP not in str(e.value)
    if match is not None:
        assert match in str(e.value), str(e.value)


def i32(*shape):
    return torch.zeros(shape, dtype=torch.int32)


def f32(*shape):
    return torch.zeros(shape, dtype=torch.float32)


def bf16(*shape):
    return torch.zeros(shape, dtype=torch.bfloat16)


B, H, N, D = 1, 4, 1024, 128
NQB = N // 128
ROWS = B * H * NQB


def fwd_args(max_kv=3):
    q = bf16(B, H, N, D)
    return dict(q=q, k=bf16(B, H, N, D), v=bf16(B, H, N, D), kv_idx=i32(ROWS, max_kv), kv_cnt=i32(ROWS),
                o=torch.empty_like(q), lse=f32(B, H, N))


def call_forward(a, **kw):
    bsa.forward(a["q"], a["k"], a["v"], a["kv_idx"], a["kv_cnt"], a["o"], a["lse"], **kw)


def test_forward_accepts_the_documented_shapes():
    a = fwd_args()
    accepted(call_forward, a)
    accepted(call_forward, a, log_w=f32(ROWS, 3), q_map=i32(B * H, N), kv_map=i32(B * H, N),
             row_perm=i32(B * H, NQB))
    accepted(call_forward, dict(a, kv_idx=i32(ROWS + 5, 3), kv_cnt=i32(ROWS + 5)))   # larger buffers
    accepted(call_forward, dict(a, kv_cnt=i32(B * H, NQB)))                          # any view of the counts


@pytest.mark.parametrize("change,match", [
    (dict(kv_idx=i32(ROWS - 1, 3)), "kv_idx"),
    (dict(kv_idx=i32(ROWS * 3)), "kv_idx"),                                  # not 2-D
    (dict(kv_idx=torch.zeros((ROWS, 3), dtype=torch.int64)), "kv_idx"),
    (dict(kv_cnt=i32(ROWS - 1)), "kv_cnt"),
    (dict(kv_cnt=torch.zeros(ROWS, dtype=torch.int64)), "kv_cnt"),
    (dict(lse=f32(B, H, N - 1)), "lse"),
])
def test_forward_rejects_short_or_mistyped_lists(change, match):
    rejected(call_forward, dict(fwd_args(), **change), match=match)


@pytest.mark.parametrize("kw,match", [
    (dict(log_w=f32(ROWS, 4)), "log_w"),           # another row stride than kv_idx
    (dict(log_w=f32(ROWS - 1, 3)), "log_w"),
    (dict(q_map=i32(B * H, N - 1)), "q_map"),
    (dict(kv_map=torch.zeros((B * H, N), dtype=torch.int64)), "kv_map"),
    (dict(row_perm=i32(B * H, NQB - 1)), "row_perm"),
    (dict(row_perm=torch.zeros((B * H, NQB), dtype=torch.int64)), "row_perm"),
])
def test_forward_rejects_short_or_mistyped_options(kw, match):
    rejected(call_forward, fwd_args(), match=match, **kw)


def test_forward_rejects_mixed_devices():
    a = fwd_args()
    rejected(call_forward, dict(a, kv_cnt=torch.zeros(ROWS, dtype=torch.int32, device="meta")),
             match="one device")


def test_forward_requires_lists():
    rejected(call_forward, dict(fwd_args(), kv_idx=None), match="required")


def test_masked_grouped_heads():
    H_kv = 2
    a = fwd_args()
    k, v = bf16(B, H_kv, N, D), bf16(B, H_kv, N, D)

    def call(**kw):
        bsa.forward_masked(a["q"], k, v, a["kv_idx"], a["kv_cnt"], a["o"], a["lse"], **kw)

    accepted(call, causal=True, window=256, sinks=4)
    accepted(call, q_map=i32(B * H, N), kv_map=i32(B * H_kv, N))      # kv_map over the K/V heads
    accepted(call, q_map=i32(B * H, N), kv_map=i32(B * H, N))         # a larger map is fine
    rejected(call, kv_map=i32(B * H_kv - 1, N), match="kv_map")
    rejected(call, q_map=i32(B * H_kv, N), match="q_map")


def test_packed_tiles_and_quadrant_masks():
    H_kv, N_kv, max_kv = 2, 3 * N, 5
    a = fwd_args(max_kv)
    k, v = bf16(B, H_kv, N, D), bf16(B, H_kv, N, D)

    def call(kv_map, **kw):
        bsa.forward_packed(a["q"], k, v, a["kv_idx"], a["kv_cnt"], kv_map, a["o"], a["lse"], **kw)

    qm = torch.zeros((ROWS, max_kv), dtype=torch.uint8)
    accepted(call, i32(B * H_kv, N_kv), quad_mask=qm, q_map=i32(B * H, N), row_perm=i32(B * H, NQB))
    rejected(call, i32(B * H_kv - 1, N_kv), match="kv_map")
    rejected(call, i32(B * H_kv, N_kv), quad_mask=qm[:, :4], match="quad_mask")
    rejected(call, None, match="kv_map")


def test_gather0_lists_and_quadrant_masks():
    img_h, img_w, n_text, groups = 32, 32, 128, 2
    Ng = n_text + img_h * img_w
    rows = B * H * (Ng // 128)
    q = bf16(B, H, Ng, D)
    k = bf16(B, 2, Ng, D)
    max_kv = 6

    def call(idx, cnt, qm, lse=None, **kw):
        bsa.forward_gather0(q, k, torch.empty_like(k), img_h, img_w, n_text, groups, idx, cnt,
                            torch.empty_like(q), f32(B, H, Ng) if lse is None else lse, quad_mask=qm, **kw)

    u8 = lambda *s: torch.zeros(s, dtype=torch.uint8)  # noqa: E731
    accepted(call, i32(rows, max_kv), i32(rows), u8(rows, max_kv))
    accepted(call, i32(rows, max_kv), i32(rows), None, row_perm=i32(B * H, Ng // 128))
    rejected(call, i32(rows, max_kv), i32(rows), u8(rows - 1, max_kv), match="quad_mask")
    rejected(call, i32(rows, max_kv), i32(rows), u8(rows, max_kv - 1), match="quad_mask")
    rejected(call, i32(rows, max_kv), i32(rows), i32(rows, max_kv), match="quad_mask")
    rejected(call, i32(rows - 1, max_kv), i32(rows), None, match="kv_idx")


def test_scatter_lists():
    a = fwd_args()

    def call(**kw):
        bsa.forward_scatter(a["q"], a["k"], a["v"], 8, a["kv_idx"], a["kv_cnt"], a["o"], a["lse"], **kw)

    accepted(call, log_w=f32(ROWS, 3), row_perm=i32(B * H, NQB))
    rejected(call, log_w=f32(ROWS, 2), match="log_w")
    rejected(call, row_perm=i32(B * H * NQB - 1), match="row_perm")


def test_crm_rows():
    a = fwd_args()
    words = i32(ROWS, 1)

    def call(w, **kw):
        bsa.forward_crm(a["q"], a["k"], a["v"], w, a["o"], a["lse"], **kw)

    accepted(call, words)
    accepted(call, i32(ROWS, 2), q_map=i32(B * H, N), kv_map=i32(B * H, N), row_perm=i32(B * H, NQB))
    rejected(call, i32(ROWS - 1, 1), match="crm")
    rejected(call, words, q_map=i32(N), match="q_map")
    rejected(lambda: bsa.forward_crm(a["q"], bf16(B, 2, N, D), a["v"], words, a["o"], a["lse"]),
             match="shape")
    src = torch.zeros((ROWS, NQB), dtype=torch.uint8)
    accepted(bsa.build_crm, bsa.IDX_MASK_U8, src, i32(ROWS, 1))
    rejected(bsa.build_crm, bsa.IDX_MASK_U8, src, i32(ROWS - 1, 1), match="words")


def test_build_index():
    rows, nkb = 40, 16
    T = f32(rows, nkb)
    accepted(bsa.build_index, bsa.IDX_THRESHOLD_F32, T, i32(rows, nkb), i32(rows), p=0.2)
    accepted(bsa.build_index, bsa.IDX_TOPK_F32, T, i32(rows, 4), i32(rows), k_per_row=i32(rows))
    rejected(bsa.build_index, bsa.IDX_THRESHOLD_F32, T, i32(rows - 1, nkb), i32(rows), match="kv_idx")
    rejected(bsa.build_index, bsa.IDX_THRESHOLD_F32, T, i32(rows, nkb), i32(rows - 1), match="kv_cnt")
    rejected(bsa.build_index, bsa.IDX_TOPK_F32, T, i32(rows, 4), i32(rows), k_per_row=i32(rows - 1),
             match="k_per_row")
    rejected(bsa.build_index, bsa.IDX_MASK_U8, T, i32(rows, nkb), i32(rows), match="src")


def test_sample_blocks():
    rows, nkb, m, cap = 30, 40, 6, 10
    s = f32(rows, nkb)
    u = torch.zeros(rows, dtype=torch.float64)

    def call(scores=s, ex=None, ec=None, uu=u, idx=None, cnt=None, lw=None, **kw):
        bsa.sample_blocks(scores, i32(rows, 3) if ex is None else ex, i32(rows) if ec is None else ec, m, uu,
                          i32(rows, cap) if idx is None else idx, i32(rows) if cnt is None else cnt,
                          f32(rows, cap) if lw is None else lw, **kw)

    accepted(call)
    accepted(call, scores=None, nkb=nkb)
    rejected(call, scores=None, match="nkb")
    rejected(call, uu=u[:-1], match="u")
    rejected(call, uu=u.float(), match="u")
    rejected(call, lw=f32(rows, cap - 1), match="log_w")
    rejected(call, ex=i32(rows - 1, 3), match="exact_idx")
    rejected(call, ec=i32(rows - 1), match="exact_cnt")
    rejected(call, cnt=i32(rows - 1), match="kv_cnt")


def test_reorder_and_spectral_order():
    heads, nqb = 3, 20
    cnt = i32(heads * nqb)
    accepted(bsa.reorder_rows, cnt.view(heads, nqb), 5, i32(heads, nqb), order_in=i32(heads, nqb))
    rejected(bsa.reorder_rows, cnt.view(heads, nqb), 5, i32(heads, nqb - 1), match="row_perm")
    rejected(bsa.reorder_rows, cnt.view(heads, nqb), 5, i32(heads, nqb), order_in=i32(heads * nqb - 1),
             match="order_in")
    idx = i32(heads * nqb, 7)
    x0 = f32(heads, nqb, 2)
    order = i32(heads, nqb)
    ws = torch.zeros(1 << 16, dtype=torch.uint8)
    accepted(bsa.spectral_order, idx, cnt, nqb, x0, order, workspace=ws, x_out=f32(heads, nqb, 2),
             angle=f32(heads, nqb))
    rejected(bsa.spectral_order, idx[:-1], cnt, nqb, x0, order, workspace=ws, match="kv_idx")
    rejected(bsa.spectral_order, idx, cnt, nqb, x0[:, :-1], order, workspace=ws, match="x0")
    rejected(bsa.spectral_order, idx, cnt, nqb, x0, order, workspace=ws, angle=f32(heads, nqb - 1),
             match="angle")
    accepted(bsa.spectral_order_noalloc, idx, cnt, nqb, x0, order)
    rejected(bsa.spectral_order_noalloc, idx, cnt[:-1], nqb, x0, order, match="kv_cnt")


def test_block_scores_and_upscale():
    q = bf16(B, H, N, D)
    ws = torch.zeros(1 << 20, dtype=torch.uint8)
    accepted(bsa.block_scores, q, bf16(B, H, N, D), f32(ROWS, NQB), workspace=ws, q_map=i32(B * H, N))
    rejected(bsa.block_scores, q, bf16(B, H, N, D), f32(ROWS, NQB - 1), workspace=ws, match="scores")
    rejected(bsa.block_scores, q, bf16(B, 2, N, D), f32(ROWS, NQB), workspace=ws, match="shape")
    accepted(bsa.upscale_threshold, f32(2, 3, 4), f32(2, 6, 8))
    rejected(bsa.upscale_threshold, f32(2, 3, 4), f32(3, 6, 8), match="heads")


def test_tensors_must_be_on_the_current_device(monkeypatch):
    """The kernels run on the current device: tensors of another device are
    refused (checked with device objects; no GPU needed)."""
    from long_context_mask_gb300 import binding
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 1)
    with pytest.raises(ValueError, match="current device"):
        binding._current_device(torch.device("cuda", 0))
    binding._current_device(torch.device("cuda", 1))
    binding._current_device(torch.device("cuda"))     # no index: allocated on the current device
    binding._current_device(torch.device("cpu"))      # stops later, at the CUDA pointer step
    with pytest.raises(ValueError, match="current device"):
        bsa.gather0_layout(32, 32, 128, 2, 1, device="cuda:0")
