"""ctypes marshalling for libxq.so (the C ABI declared in include/xq.h)."""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libxq.so")

if not os.path.exists(_LIB_PATH):
    raise ImportError(
        f"the CUDA library {_LIB_PATH} is missing; build it first "
        "(python -m quantized_decode_mat_gb300.build, or __graft_entry__.build())")

_lib = ctypes.CDLL(_LIB_PATH)

_P, _I32, _I64, _SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t


class _Plan(ctypes.Structure):
    _fields_ = [("warps", ctypes.c_int32), ("stages", ctypes.c_int32), ("grid", ctypes.c_int32),
                ("rows_per_group", ctypes.c_int32), ("segments", ctypes.c_int32),
                ("chunks_per_row", ctypes.c_int32), ("groups", ctypes.c_int64),
                ("batch_per_launch", ctypes.c_int32), ("launches", ctypes.c_int32),
                ("smem_bytes", ctypes.c_int64), ("row_block", ctypes.c_int32),
                ("quantise_once", ctypes.c_int32), ("vector_pairs", ctypes.c_int32),
                ("tensor", ctypes.c_int32)]


def _sig(name, restype, argtypes):
    fn = getattr(_lib, name)
    fn.restype = restype
    fn.argtypes = argtypes
    return fn


_q8_bytes = _sig("xq_q8_bytes", _SZ, [_I64, _I64])
_q4k_bytes = _sig("xq_q4k_bytes", _SZ, [_I64, _I64])
_cb4_bytes = _sig("xq_cb4_bytes", _SZ, [_I64, _I64])
_quantize = _sig("xq_quantize_q8", ctypes.c_int, [_P, _P, _I64, _I64, _P])
_matvec_q4k = _sig("xq_matvec_q4k", ctypes.c_int, [_P, _P, _P, _I64, _I64, _I64, _P])
_matvec_cb4 = _sig("xq_matvec_cb4", ctypes.c_int, [_P, _P, _P, _P, _I64, _I64, _I64, _P])
_linear_q4k = _sig("xq_linear_q4k", ctypes.c_int, [_P, _P, _P, _I64, _I64, _I64, _P])
_linear_cb4 = _sig("xq_linear_cb4", ctypes.c_int, [_P, _P, _P, _P, _I64, _I64, _I64, _P])
_rmsnorm_q8 = _sig("xq_rmsnorm_q8", ctypes.c_int, [_P, _P, _P, _I64, _I64, _P])
_norm_linear_q4k = _sig("xq_norm_linear_q4k", ctypes.c_int, [_P, _P, _P, _I64, _I64, _I64, _P])
_norm_linear_cb4 = _sig("xq_norm_linear_cb4", ctypes.c_int,
                        [_P, _P, _P, _P, _I64, _I64, _I64, _P])
_matvec_q4k_id = _sig("xq_matvec_q4k_id", ctypes.c_int,
                      [_P, _P, _P, _P, _I64, _I64, _I64, _I64, _I32, _P])
_matvec_cb4_id = _sig("xq_matvec_cb4_id", ctypes.c_int,
                      [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I32, _P])
_cb4r_bytes = _sig("xq_cb4r_bytes", _SZ, [_I64, _I64])
_repack_cb4 = _sig("xq_repack_cb4", ctypes.c_int, [_P, _P, _I64, _I64, _I64, _I64, _P])
_matvec_cb4r = _sig("xq_matvec_cb4r", ctypes.c_int, [_P, _P, _P, _P, _I64, _I64, _I64, _P])
_linear_cb4r = _sig("xq_linear_cb4r", ctypes.c_int, [_P, _P, _P, _P, _I64, _I64, _I64, _P])
_norm_linear_cb4r = _sig("xq_norm_linear_cb4r", ctypes.c_int,
                         [_P, _P, _P, _P, _I64, _I64, _I64, _P])
_matvec_cb4r_id = _sig("xq_matvec_cb4r_id", ctypes.c_int,
                       [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I32, _P])
_subdots_cb4r = _sig("xq_subdots_cb4r", ctypes.c_int, [_P, _P, _P, _P, _I64, _I64, _I64, _P])
_linear_ws_bytes = _sig("xq_linear_workspace_bytes", _SZ, [_I64, _I64])
_linear_q4k_ws = _sig("xq_linear_q4k_ws", ctypes.c_int,
                      [_P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P])
_linear_cb4_ws = _sig("xq_linear_cb4_ws", ctypes.c_int,
                      [_P, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P])
_linear_cb4r_ws = _sig("xq_linear_cb4r_ws", ctypes.c_int,
                       [_P, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P])
_set_qonce = _sig("xq_set_quantise_once_override", None, [_I32])
_set_overlap = _sig("xq_set_overlap_launches", None, [_I32])
_get_overlap = _sig("xq_overlap_launches", _I32, [])
_linear_q4k_static = _sig("xq_linear_q4k_static", ctypes.c_int,
                          [_P, _P, _P, _I64, _I64, _I64, _P])
_subdots_q4k = _sig("xq_subdots_q4k", ctypes.c_int, [_P, _P, _P, _I64, _I64, _I64, _P])
_subdots_cb4 = _sig("xq_subdots_cb4", ctypes.c_int, [_P, _P, _P, _P, _I64, _I64, _I64, _P])
_plan = _sig("xq_plan_matvec", ctypes.c_int, [_I32, _I64, _I64, _I64, _I32, _I64,
                                             ctypes.POINTER(_Plan)])
_set_override = _sig("xq_set_plan_override", None, [_I32, _I32])
_set_row_block = _sig("xq_set_row_block_override", None, [_I32])
_set_vector_pairs = _sig("xq_set_vector_pairs_override", None, [_I32])
_set_tensor = _sig("xq_set_tensor_override", None, [_I32])
_last_plan = _sig("xq_last_plan", ctypes.c_int, [ctypes.POINTER(_Plan)])
_launch_count = _sig("xq_launch_count", ctypes.c_uint64, [_I32])
_device_status = _sig("xq_device_status", ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32),
                                                        _I32, _P])
_status_string = _sig("xq_status_string", ctypes.c_char_p, [ctypes.c_int])
_last_error = _sig("xq_last_error", ctypes.c_char_p, [])
_version = _sig("xq_version", _I32, [])

(COUNT_QUANTIZE, COUNT_MATVEC_Q4K, COUNT_MATVEC_CB4, COUNT_SUBDOTS_Q4K, COUNT_SUBDOTS_CB4,
 COUNT_LINEAR_Q4K, COUNT_LINEAR_CB4, COUNT_MATVEC_ID_Q4K, COUNT_MATVEC_ID_CB4,
 COUNT_RMSNORM_Q8, COUNT_NORM_LINEAR_Q4K, COUNT_NORM_LINEAR_CB4, COUNT_REPACK_CB4,
 COUNT_MATVEC_CB4R, COUNT_SUBDOTS_CB4R, COUNT_LINEAR_CB4R, COUNT_NORM_LINEAR_CB4R,
 COUNT_MATVEC_ID_CB4R, COUNT_QUANTISE_ONCE) = range(19)
COUNT_N = 19


class XQError(RuntimeError):
    def __init__(self, status: int, detail: str):
        self.status = status
        self.detail = detail
        super().__init__(f"{_status_string(status).decode()}: {detail}")


def lib_path() -> str:
    return _LIB_PATH


def _check(status: int) -> None:
    if status != 0:
        raise XQError(status, (_last_error() or b"").decode())


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dev(t: torch.Tensor, name: str, dtype=None, nbytes: int | None = None) -> int:
    """Device address of t after checking it: CUDA, dtype, contiguous, and at
    least nbytes long (the C ABI takes raw pointers and cannot check sizes, so
    a short buffer would be read or written past its end)."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if nbytes is not None and t.numel() * t.element_size() < nbytes:
        raise ValueError(f"{name} holds {t.numel() * t.element_size()} bytes, {nbytes} needed")
    return t.data_ptr()


def _w_bytes(rows: int, cols: int) -> int:
    """Bytes of a weight matrix: 144 per 256 weights in every format."""
    return rows * max(cols // 256, 0) * 144


def _wp(W: torch.Tensor, rows: int, cols: int, name: str = "W") -> int:
    return _dev(W, name, torch.uint8, _w_bytes(rows, cols))


def _yp(y: torch.Tensor, batch: int, rows: int) -> int:
    return _dev(y, "y", torch.float32, 4 * batch * rows)


def _dotsp(d: torch.Tensor, batch: int, rows: int, cols: int) -> int:
    return _dev(d, "dots", torch.int32, 4 * batch * rows * (cols // 32))


def _table(table) -> ctypes.Array:
    kv = np.asarray(table.cpu() if isinstance(table, torch.Tensor) else table)
    if kv.size != 16:
        raise ValueError("the codebook table must have 16 entries")
    kv = kv.astype(np.int8).reshape(16)
    return (ctypes.c_int8 * 16)(*[int(v) for v in kv])


def q8_bytes(cols: int, batch: int = 1) -> int:
    return int(_q8_bytes(cols, batch))


def q4k_bytes(rows: int, cols: int) -> int:
    return int(_q4k_bytes(rows, cols))


def cb4_bytes(rows: int, cols: int) -> int:
    return int(_cb4_bytes(rows, cols))


def quantize_q8(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """x: f32 [batch, cols] (or [cols]) on CUDA -> uint8 [batch, cols/256, 320]."""
    if x.dim() == 1:
        x = x.unsqueeze(0)
    batch, cols = x.shape
    if out is None:
        out = torch.empty((batch, max(cols // 256, 0), 320), dtype=torch.uint8, device=x.device)
    _check(_quantize(_dev(x, "x", torch.float32),
                     _dev(out, "xq", torch.uint8, q8_bytes(cols, batch)), cols, batch,
                     _stream(stream)))
    return out


def _batch_of(xq: torch.Tensor, cols: int) -> int:
    per = q8_bytes(cols, 1)
    if per == 0 or xq.numel() % per:
        raise ValueError("xq size does not match cols")
    return xq.numel() // per


def matvec_q4k(W: torch.Tensor, xq: torch.Tensor, rows: int, cols: int,
               out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y[b, r] for Q4_K rows W (uint8, CUDA) and q8 blocks xq -> f32 [batch, rows]."""
    batch = _batch_of(xq, cols)
    if out is None:
        out = torch.empty((batch, rows), dtype=torch.float32, device=xq.device)
    _check(_matvec_q4k(_wp(W, rows, cols), _dev(xq, "xq", torch.uint8),
                       _yp(out, batch, rows), rows, cols, batch, _stream(stream)))
    return out


def matvec_cb4(W: torch.Tensor, table, xq: torch.Tensor, rows: int, cols: int,
               out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y[b, r] for codebook rows W with a host 16-entry int8 table."""
    batch = _batch_of(xq, cols)
    if out is None:
        out = torch.empty((batch, rows), dtype=torch.float32, device=xq.device)
    _check(_matvec_cb4(_wp(W, rows, cols), ctypes.cast(_table(table), _P),
                       _dev(xq, "xq", torch.uint8), _yp(out, batch, rows), rows, cols,
                       batch, _stream(stream)))
    return out


def _x2d(x: torch.Tensor) -> torch.Tensor:
    return x.unsqueeze(0) if x.dim() == 1 else x


def linear_q4k(x: torch.Tensor, W: torch.Tensor, rows: int, cols: int,
               out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Fused decode step: quantise x (f32 [batch, cols], CUDA) and multiply by
    the Q4_K rows W in one launch -> f32 [batch, rows]."""
    x = _x2d(x)
    batch = x.shape[0]
    if x.shape[1] != cols:
        raise ValueError("x has the wrong number of columns")
    if out is None:
        out = torch.empty((batch, rows), dtype=torch.float32, device=x.device)
    _check(_linear_q4k(_dev(x, "x", torch.float32), _wp(W, rows, cols),
                       _yp(out, batch, rows), rows, cols, batch, _stream(stream)))
    return out


def linear_cb4(x: torch.Tensor, W: torch.Tensor, table, rows: int, cols: int,
               out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Fused decode step for codebook rows W with a host 16-entry int8 table."""
    x = _x2d(x)
    batch = x.shape[0]
    if x.shape[1] != cols:
        raise ValueError("x has the wrong number of columns")
    if out is None:
        out = torch.empty((batch, rows), dtype=torch.float32, device=x.device)
    _check(_linear_cb4(_dev(x, "x", torch.float32), _wp(W, rows, cols),
                       ctypes.cast(_table(table), _P), _yp(out, batch, rows), rows,
                       cols, batch, _stream(stream)))
    return out


def linear_workspace_bytes(cols: int, batch: int = 1) -> int:
    return int(_linear_ws_bytes(cols, batch))


def linear_ws(fmt: str, x: torch.Tensor, W: torch.Tensor, rows: int, cols: int,
              ws: torch.Tensor, table=None, out: torch.Tensor | None = None,
              stream=None) -> torch.Tensor:
    """The fused decode step with a caller workspace ``ws`` (uint8, CUDA, at
    least linear_workspace_bytes(cols, batch) bytes): the same y as
    linear_q4k / linear_cb4 / linear_cb4r, with the activation quantised once
    across the grid when the plan says so.  fmt: "q4k", "cb4" or "cb4r"."""
    x = _x2d(x)
    batch = x.shape[0]
    if x.shape[1] != cols:
        raise ValueError("x has the wrong number of columns")
    if out is None:
        out = torch.empty((batch, rows), dtype=torch.float32, device=x.device)
    xp, Wp, yp = _dev(x, "x", torch.float32), _wp(W, rows, cols), _yp(out, batch, rows)
    wp, nbytes = _dev(ws, "ws", torch.uint8), ws.numel()
    if fmt == "q4k":
        st = _linear_q4k_ws(xp, Wp, yp, rows, cols, batch, wp, nbytes, _stream(stream))
    elif fmt in ("cb4", "cb4r"):
        fn = _linear_cb4_ws if fmt == "cb4" else _linear_cb4r_ws
        st = fn(xp, Wp, ctypes.cast(_table(table), _P), yp, rows, cols, batch, wp, nbytes,
                _stream(stream))
    else:
        raise ValueError(f"unknown format {fmt!r}")
    _check(st)
    return out


def linear_q4k_static(x: torch.Tensor, W: torch.Tensor, rows: int, cols: int,
                      out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """linear_ws("q4k", ...) with the library's fixed scratch instead of a
    caller workspace (for callers that may not allocate; batch * cols <=
    209664).  ``out`` must be given by a caller that may not allocate."""
    x = _x2d(x)
    batch = x.shape[0]
    if x.shape[1] != cols:
        raise ValueError("x has the wrong number of columns")
    if out is None:
        out = torch.empty((batch, rows), dtype=torch.float32, device=x.device)
    _check(_linear_q4k_static(_dev(x, "x", torch.float32), _wp(W, rows, cols),
                              _yp(out, batch, rows), rows, cols, batch, _stream(stream)))
    return out


def set_overlap_launches(enable: bool) -> None:
    """Overlapped launches (see xq_set_overlap_launches in include/xq.h): a
    launch may start streaming W while the kernel before it on the stream
    finishes.  Only when that kernel does not write the W being read."""
    _set_overlap(1 if enable else 0)


def overlap_launches() -> bool:
    return bool(_get_overlap())


def set_quantise_once_override(mode: int = 0) -> None:
    """The decode step's choice (xq_plan.quantise_once): 1 every CTA of the one
    fused launch quantises x; 2 x is quantised once, by a launch of its own,
    into the workspace; 0 automatic (once from 33 q8 blocks a launch)."""
    _set_qonce(mode)


def rmsnorm_q8(x: torch.Tensor, out: torch.Tensor | None = None, y: torch.Tensor | None = None,
               stream=None) -> torch.Tensor:
    """RMSNorm + q8 pack: x f32 [batch, cols] (CUDA) -> the q8 blocks of
    x * scale (uint8 [batch, cols/256, 320]); writes the f32 x * scale into
    ``y`` too when it is given."""
    x = _x2d(x)
    batch, cols = x.shape
    if out is None:
        out = torch.empty((batch, max(cols // 256, 0), 320), dtype=torch.uint8, device=x.device)
    yp = None if y is None else _dev(y, "y", torch.float32, 4 * batch * cols)
    _check(_rmsnorm_q8(_dev(x, "x", torch.float32), _dev(out, "xq", torch.uint8,
                                                         q8_bytes(cols, batch)), yp, cols,
                       batch, _stream(stream)))
    return out


def _norm_linear(fn, x, W, table, rows, cols, out, stream):
    x = _x2d(x)
    batch = x.shape[0]
    if x.shape[1] != cols:
        raise ValueError("x has the wrong number of columns")
    if out is None:
        out = torch.empty((batch, rows), dtype=torch.float32, device=x.device)
    args = [_dev(x, "x", torch.float32), _wp(W, rows, cols)]
    if table is not None:
        args.append(ctypes.cast(_table(table), _P))
    _check(fn(*args, _yp(out, batch, rows), rows, cols, batch, _stream(stream)))
    return out


def norm_linear_q4k(x: torch.Tensor, W: torch.Tensor, rows: int, cols: int,
                    out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """RMSNorm, quantise and multiply by the Q4_K rows W in one launch."""
    return _norm_linear(_norm_linear_q4k, x, W, None, rows, cols, out, stream)


def norm_linear_cb4(x: torch.Tensor, W: torch.Tensor, table, rows: int, cols: int,
                    out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """RMSNorm, quantise and multiply by the codebook rows W in one launch."""
    return _norm_linear(_norm_linear_cb4, x, W, table, rows, cols, out, stream)


def matvec_id(fmt: str, W: torch.Tensor, sel: torch.Tensor, xq: torch.Tensor,
              rows_per_expert: int, cols: int, n_experts: int, table=None,
              x_per_slot: bool = False, out: torch.Tensor | None = None,
              stream=None) -> torch.Tensor:
    """Grouped experts: y[kk] = W[expert sel[kk]] . x (x = xq vector 0, or
    vector kk with x_per_slot) -> f32 [used, rows_per_expert].  fmt: "q4k",
    "cb4" (raw codebook rows) or "cb4r" (resident codebook rows)."""
    used = int(sel.numel())
    if out is None:
        out = torch.empty((used, rows_per_expert), dtype=torch.float32, device=xq.device)
    s = _dev(sel, "sel", torch.int32)
    Wp = _dev(W, "W", torch.uint8, n_experts * _w_bytes(rows_per_expert, cols))
    xp = _dev(xq, "xq", torch.uint8, (used if x_per_slot else 1) * q8_bytes(cols, 1))
    yp = _dev(out, "y", torch.float32, 4 * used * rows_per_expert)
    if fmt == "q4k":
        _check(_matvec_q4k_id(Wp, s, xp, yp, rows_per_expert, cols, n_experts, used,
                              int(x_per_slot), _stream(stream)))
    elif fmt in ("cb4", "cb4r"):
        fn = _matvec_cb4_id if fmt == "cb4" else _matvec_cb4r_id
        _check(fn(Wp, ctypes.cast(_table(table), _P), s, xp, yp, rows_per_expert, cols, n_experts,
                  used, int(x_per_slot), _stream(stream)))
    else:
        raise ValueError(f"unknown format {fmt!r}")
    return out


def subdots_q4k(W: torch.Tensor, xq: torch.Tensor, rows: int, cols: int,
                out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Exact per-sub-block int32 dots, [batch, rows, cols/32]."""
    batch = _batch_of(xq, cols)
    if out is None:
        out = torch.empty((batch, rows, cols // 32), dtype=torch.int32, device=xq.device)
    _check(_subdots_q4k(_wp(W, rows, cols), _dev(xq, "xq", torch.uint8),
                        _dotsp(out, batch, rows, cols), rows, cols, batch, _stream(stream)))
    return out


def subdots_cb4(W: torch.Tensor, table, xq: torch.Tensor, rows: int, cols: int,
                out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    batch = _batch_of(xq, cols)
    if out is None:
        out = torch.empty((batch, rows, cols // 32), dtype=torch.int32, device=xq.device)
    _check(_subdots_cb4(_wp(W, rows, cols), ctypes.cast(_table(table), _P),
                        _dev(xq, "xq", torch.uint8), _dotsp(out, batch, rows, cols), rows, cols,
                        batch, _stream(stream)))
    return out


# ---------------------------------------------------------------- resident codebook rows
def cb4r_bytes(rows: int, cols: int) -> int:
    return int(_cb4r_bytes(rows, cols))


def repack_cb4(src: torch.Tensor, rows: int, cols: int, out: torch.Tensor | None = None,
               block_base: int = 0, n_blocks: int | None = None, src_offset: int = 0,
               stream=None) -> torch.Tensor:
    """Repack raw codebook blocks (uint8, CUDA; the n_blocks blocks starting at
    byte src_offset of src, which are blocks block_base.. of the matrix) into
    the resident rows ``out`` (uint8 [cb4r_bytes(rows, cols)], CUDA)."""
    if n_blocks is None:
        n_blocks = rows * (cols // 32) - block_base
    if out is None:
        out = torch.zeros(cb4r_bytes(rows, cols), dtype=torch.uint8, device=src.device)
    base = _dev(src, "src", torch.uint8)
    if src_offset < 0 or src_offset + 18 * n_blocks > src.numel():
        raise ValueError("src is too small for the chunk")
    _check(_repack_cb4(base + src_offset, _dev(out, "Wr", torch.uint8, cb4r_bytes(rows, cols)),
                       block_base, n_blocks,
                       rows, cols, _stream(stream)))
    return out


def matvec_cb4r(Wr: torch.Tensor, table, xq: torch.Tensor, rows: int, cols: int,
                out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y[b, r] for resident codebook rows Wr with a host 16-entry int8 table."""
    batch = _batch_of(xq, cols)
    if out is None:
        out = torch.empty((batch, rows), dtype=torch.float32, device=xq.device)
    _check(_matvec_cb4r(_wp(Wr, rows, cols, "Wr"), ctypes.cast(_table(table), _P),
                        _dev(xq, "xq", torch.uint8), _yp(out, batch, rows), rows, cols,
                        batch, _stream(stream)))
    return out


def linear_cb4r(x: torch.Tensor, Wr: torch.Tensor, table, rows: int, cols: int,
                out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Fused decode step (quantise + mat-vec, one launch) on resident codebook rows."""
    x = _x2d(x)
    batch = x.shape[0]
    if x.shape[1] != cols:
        raise ValueError("x has the wrong number of columns")
    if out is None:
        out = torch.empty((batch, rows), dtype=torch.float32, device=x.device)
    _check(_linear_cb4r(_dev(x, "x", torch.float32), _wp(Wr, rows, cols, "Wr"),
                        ctypes.cast(_table(table), _P), _yp(out, batch, rows), rows,
                        cols, batch, _stream(stream)))
    return out


def norm_linear_cb4r(x: torch.Tensor, Wr: torch.Tensor, table, rows: int, cols: int,
                     out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """RMSNorm, quantise and multiply by resident codebook rows in one launch."""
    return _norm_linear(_norm_linear_cb4r, x, Wr, table, rows, cols, out, stream)


def subdots_cb4r(Wr: torch.Tensor, table, xq: torch.Tensor, rows: int, cols: int,
                 out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    batch = _batch_of(xq, cols)
    if out is None:
        out = torch.empty((batch, rows, cols // 32), dtype=torch.int32, device=xq.device)
    _check(_subdots_cb4r(_wp(Wr, rows, cols, "Wr"), ctypes.cast(_table(table), _P),
                         _dev(xq, "xq", torch.uint8), _dotsp(out, batch, rows, cols), rows,
                         cols, batch, _stream(stream)))
    return out


def _plan_dict(p: _Plan) -> dict:
    return {f: getattr(p, f) for f, _ in _Plan._fields_}


FORMATS = {"q4k": 0, "cb4": 1, "cb4r": 2}


def plan_matvec(rows: int, cols: int, batch: int = 1, fmt: str = "q4k", sm_count: int = 152,
                smem_optin: int = 232448) -> dict:
    """Host-only launch plan (no GPU needed)."""
    p = _Plan()
    _check(_plan(FORMATS[fmt], rows, cols, batch, sm_count, smem_optin, ctypes.byref(p)))
    return _plan_dict(p)


def last_plan() -> dict:
    p = _Plan()
    _check(_last_plan(ctypes.byref(p)))
    return _plan_dict(p)


def set_plan_override(warps: int = 0, stages: int = 0) -> None:
    """Force the warps a CTA (clamped to the kernel's limit: 20 at batch 1,
    16 for the fused RMSNorm form there; Q4_K 12 at batch 2, 8 above;
    codebook 16 up to batch 4, 8 above) and the stages a warp (1..8, lowered
    until shared memory fits); 0 restores the automatic plan.  For sweeps
    and tests: process-wide, not for use beside concurrent launches."""
    _set_override(warps, stages)


def set_row_block_override(row_block: int = 0) -> None:
    """1 forces one row group per warp unit; 0 restores the automatic plan."""
    _set_row_block(row_block)


def set_vector_pairs_override(mode: int = 0) -> None:
    """Warp pairs sharing each unit (xq_plan.vector_pairs): 1 never, 2 wherever
    they apply (then set_plan_override's warps and stages, if set, size the
    pairs), 0 automatic.  The results are bit-identical either way."""
    _set_vector_pairs(mode)


def set_tensor_override(mode: int = 0) -> None:
    """Dots on the tensor cores (xq_plan.tensor): 1 never, 2 wherever they
    apply (then set_plan_override's stages, if set, size the plan), 0
    automatic.  The results are bit-identical either way."""
    _set_tensor(mode)


def launch_count(which: int) -> int:
    return int(_launch_count(which))


def device_status(clear: bool = False, stream=None) -> int:
    """Device status word (0 = fine); synchronises the stream."""
    v = ctypes.c_uint32(0)
    st = _device_status(ctypes.byref(v), int(clear), _stream(stream))
    if st not in (0, 5):
        _check(st)
    return int(v.value)


def version() -> int:
    return int(_version())
