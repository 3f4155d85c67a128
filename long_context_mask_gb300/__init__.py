"""GB300-native block-sparse attention: Python binding of ``libbsa.so``.

Every compute step runs in the CUDA library; this module only marshals
arguments (device pointers of torch tensors, sizes, the current CUDA stream)
into the C-ABI declared in ``include/bsa.h``.  There is no CPU fallback: if
the library is missing, every call raises.
"""
from __future__ import annotations

from .binding import (  # noqa: F401
    BLOCK,
    BsaError,
    IDX_MASK_U8,
    IDX_THRESHOLD_F32,
    IDX_TOPK_F32,
    SCORE_CENTROID_EXP,
    SCORE_MEAN_DOT,
    block_scores,
    NOALLOC_SCRATCH_BYTES,
    build_crm,
    build_index,
    dense_attention_flops,
    device_status,
    effective_flops,
    forward,
    forward_crm,
    forward_gather0,
    forward_masked,
    forward_packed,
    forward_scatter,
    gather0_layout,
    gather0_sizes,
    gather_rows,
    lib_path,
    load_library,
    reorder_guard,
    reorder_rows,
    resident_ctas,
    sample_blocks,
    set_forward_options,
    selftest_exp2,
    selftest_wait_timeout,
    spectral_order,
    spectral_order_noalloc,
    spectral_order_workspace_size,
    upscale_threshold,
)
