"""GB300 (sm_103a) 4-bit decode mat-vec on the integer route.

Thin Python binding over the C ABI in ``include/xq.h`` (``_build/libxq.so``):
argument marshalling only.  Every step of the path runs in the library's
CUDA kernels; PyTorch supplies device memory and streams.  There is no CPU
fallback: if the library is missing this package raises on import.

    xq  = quantize_q8(x)                       # x: f32 [batch, cols] on cuda
    y   = matvec_q4k(W, xq, rows, cols)        # W: uint8 Q4_K rows on cuda
    y   = matvec_cb4(W, table, xq, rows, cols) # W: uint8 codebook rows
    y   = linear_q4k(x, W, rows, cols)         # fused: quantise + mat-vec, one launch
    y   = linear_ws("q4k", x, W, rows, cols, ws)  # the same, quantising once (workspace)
    xq  = rmsnorm_q8(x)                        # RMSNorm + q8 pack of the next input
    y   = norm_linear_q4k(x, W, rows, cols)    # fused: RMSNorm + quantise + mat-vec
    Wr  = repack_cb4(W, rows, cols)            # codebook rows -> resident rows
    y   = matvec_cb4r(Wr, table, xq, rows, cols)
"""
from __future__ import annotations

from . import _native
from ._native import (  # noqa: F401
    COUNT_LINEAR_CB4,
    COUNT_LINEAR_Q4K,
    COUNT_MATVEC_CB4,
    COUNT_MATVEC_ID_CB4,
    COUNT_MATVEC_ID_Q4K,
    COUNT_MATVEC_Q4K,
    COUNT_N,
    COUNT_NORM_LINEAR_CB4,
    COUNT_NORM_LINEAR_Q4K,
    COUNT_QUANTIZE,
    COUNT_REPACK_CB4,
    COUNT_MATVEC_CB4R,
    COUNT_SUBDOTS_CB4R,
    COUNT_LINEAR_CB4R,
    COUNT_NORM_LINEAR_CB4R,
    COUNT_MATVEC_ID_CB4R,
    COUNT_QUANTISE_ONCE,
    COUNT_RMSNORM_Q8,
    COUNT_SUBDOTS_CB4,
    COUNT_SUBDOTS_Q4K,
    XQError,
    cb4_bytes,
    cb4r_bytes,
    repack_cb4,
    matvec_cb4r,
    linear_cb4r,
    norm_linear_cb4r,
    subdots_cb4r,
    device_status,
    last_plan,
    launch_count,
    lib_path,
    linear_cb4,
    linear_q4k,
    linear_q4k_static,
    linear_workspace_bytes,
    linear_ws,
    matvec_cb4,
    matvec_id,
    matvec_q4k,
    norm_linear_cb4,
    norm_linear_q4k,
    plan_matvec,
    q4k_bytes,
    q8_bytes,
    quantize_q8,
    rmsnorm_q8,
    set_plan_override,
    set_row_block_override,
    set_vector_pairs_override,
    set_tensor_override,
    set_overlap_launches,
    overlap_launches,
    set_quantise_once_override,
    subdots_cb4,
    subdots_q4k,
)

__all__ = [n for n in dir(_native) if not n.startswith("_") and n not in ("ctypes", "os",
                                                                         "np", "torch")]
