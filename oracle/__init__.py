"""CPU oracle for the 4-bit decode mat-vec on the integer route.

TEST INFRASTRUCTURE ONLY: tests/, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the product package
``quantized_decode_mat_gb300`` never does, and this package never imports it.

The arithmetic lives in ``xq_oracle.c`` (plain C11, ``-ffp-contract=off``,
no fast-math); this module only compiles it with gcc and marshals numpy
arrays through ctypes.  Every function names the passage it follows in the C
source.  Pins that tie the oracle to the pages and to mathematics (not to
itself) are in ``tests/test_oracle_*.py``.

Parity status of each function (all pinned, none "parity unpinned"):
  quantize_q8      hand cases, tie cases, invariants, the guide's fixture
  q4k_unpack       hand-packed golden block, pack/unpack round trip
  matvec_q4k       hand-worked golden blocks, brute-force dequantised dot,
                   integer-GEMV special case (numpy int64 matmul)
  cb4_unpack/matvec hand-worked golden blocks, half-order pin, brute force,
                   integer-GEMV special case
  f16_to_f64       all 65536 bit patterns against numpy's binary16
  repack_cb4 /     literal hand-written resident bytes (whole and chunked),
  dequant_cb4r     chunking invariance, same weights as the raw matrix
  rmsnorm_q8       hand-derived f32 sums that fix the summation order, the
                   guide's three-four case, a constant-vector closed form,
                   the f32 error bound against binary64
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "xq_oracle.c")
_BUILD = os.path.join(_HERE, "_build")

Q8_BYTES = 320       # activation block bytes (guide 25.2)
Q4K_BYTES = 144      # super-block bytes (substrate spec 2.3)
CB4_BYTES = 18       # codebook block bytes (guide 25.2.1)

_lock = threading.Lock()
_libs: dict[int, ctypes.CDLL] = {}


def lib_path(fault: int = 0) -> str:
    name = "liboracle.so" if fault == 0 else f"liboracle_fault{fault}.so"
    return os.path.join(_BUILD, name)


def build(fault: int = 0, force: bool = False) -> str:
    """Compile the oracle (gcc) into ``oracle/_build``; returns the .so path.

    ``fault`` > 0 compiles a planted-mistake variant used only by the tests
    that prove the pins catch mistakes.
    """
    os.makedirs(_BUILD, exist_ok=True)
    out = lib_path(fault)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", f"-DORACLE_FAULT={fault}", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _load(fault: int = 0) -> ctypes.CDLL:
    with _lock:
        if fault in _libs:
            return _libs[fault]
        lib = ctypes.CDLL(build(fault))
        P, I64 = ctypes.c_void_p, ctypes.c_int64
        lib.oracle_fault.restype = ctypes.c_int
        lib.oracle_f16_to_f64.restype = ctypes.c_double
        lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_quantize_q8.argtypes = [P, P, I64, I64]
        lib.oracle_dequant_q8.argtypes = [P, P, I64, I64]
        lib.oracle_q4k_unpack.argtypes = [P, P, P, P, P, P]
        lib.oracle_dequant_q4k.argtypes = [P, P, I64, I64]
        lib.oracle_subdots_q4k.argtypes = [P, P, P, I64, I64, I64]
        lib.oracle_matvec_q4k.argtypes = [P, P, P, P, I64, I64, I64]
        lib.oracle_cb4_unpack.argtypes = [P, P, P, P]
        lib.oracle_dequant_cb4.argtypes = [P, P, P, I64, I64]
        lib.oracle_subdots_cb4.argtypes = [P, P, P, P, I64, I64, I64]
        lib.oracle_matvec_cb4.argtypes = [P, P, P, P, P, I64, I64, I64]
        lib.oracle_rmsnorm_sumsq.restype = ctypes.c_float
        lib.oracle_rmsnorm_sumsq.argtypes = [P, I64]
        lib.oracle_rmsnorm_scale.restype = ctypes.c_float
        lib.oracle_rmsnorm_scale.argtypes = [P, I64]
        lib.oracle_rmsnorm_q8.argtypes = [P, P, P, I64, I64]
        lib.oracle_cb4r_prefix.restype = I64
        lib.oracle_cb4r_prefix.argtypes = [I64]
        lib.oracle_cb4r_row_bytes.restype = I64
        lib.oracle_cb4r_row_bytes.argtypes = [I64]
        lib.oracle_repack_cb4.argtypes = [P, P, I64, I64, I64]
        lib.oracle_dequant_cb4r.argtypes = [P, P, P, I64, I64]
        for fn in ("oracle_quantize_q8", "oracle_dequant_q8", "oracle_q4k_unpack",
                   "oracle_dequant_q4k", "oracle_subdots_q4k", "oracle_matvec_q4k",
                   "oracle_cb4_unpack", "oracle_dequant_cb4", "oracle_subdots_cb4",
                   "oracle_matvec_cb4", "oracle_rmsnorm_q8", "oracle_repack_cb4",
                   "oracle_dequant_cb4r"):
            getattr(lib, fn).restype = None
        _libs[fault] = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _u8(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint8
    return a


class Oracle:
    """Bound view of one oracle build (``fault=0`` is the real oracle)."""

    def __init__(self, fault: int = 0):
        self.fault = fault
        self.lib = _load(fault)
        assert self.lib.oracle_fault() == fault

    # -- scalars ----------------------------------------------------------
    def f16_to_f64(self, h: int) -> float:
        return self.lib.oracle_f16_to_f64(int(h) & 0xFFFF)

    # -- q8 activation blocks ----------------------------------------------
    def quantize_q8(self, x: np.ndarray) -> np.ndarray:
        """x: float32 [batch, cols] -> uint8 [batch, cols/256, 320]."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        if x.ndim == 1:
            x = x[None, :]
        batch, cols = x.shape
        assert cols % 256 == 0
        out = np.empty((batch, cols // 256, Q8_BYTES), np.uint8)
        self.lib.oracle_quantize_q8(_ptr(x), _ptr(out), cols, batch)
        return out

    def dequant_q8(self, xq: np.ndarray, cols: int) -> np.ndarray:
        xq = _u8(xq)
        batch = xq.size // ((cols // 256) * Q8_BYTES)
        out = np.empty((batch, cols), np.float64)
        self.lib.oracle_dequant_q8(_ptr(xq), _ptr(out), cols, batch)
        return out

    # -- Q4_K super-blocks ----------------------------------------------------
    def q4k_unpack(self, blk: np.ndarray):
        blk = _u8(blk).reshape(-1)[:Q4K_BYTES].copy()
        d = np.zeros(1, np.float64)
        dmin = np.zeros(1, np.float64)
        sc = np.zeros(8, np.uint8)
        m = np.zeros(8, np.uint8)
        q = np.zeros(256, np.uint8)
        self.lib.oracle_q4k_unpack(_ptr(blk), _ptr(d), _ptr(dmin), _ptr(sc), _ptr(m), _ptr(q))
        return float(d[0]), float(dmin[0]), sc, m, q

    def dequant_q4k(self, W: np.ndarray, rows: int, cols: int) -> np.ndarray:
        W = _u8(W)
        out = np.empty((rows, cols), np.float64)
        self.lib.oracle_dequant_q4k(_ptr(W), _ptr(out), rows, cols)
        return out

    def subdots_q4k(self, W, xq, rows: int, cols: int, batch: int) -> np.ndarray:
        W, xq = _u8(W), _u8(xq)
        out = np.empty((batch, rows, (cols // 256) * 8), np.int32)
        self.lib.oracle_subdots_q4k(_ptr(W), _ptr(xq), _ptr(out), rows, cols, batch)
        return out

    def matvec_q4k(self, W, xq, rows: int, cols: int, batch: int, with_abs: bool = False):
        """Returns y (float64 [batch, rows]) and, if asked, y_abs."""
        W, xq = _u8(W), _u8(xq)
        y = np.empty((batch, rows), np.float64)
        ya = np.empty((batch, rows), np.float64) if with_abs else None
        self.lib.oracle_matvec_q4k(_ptr(W), _ptr(xq), _ptr(y), _ptr(ya) if with_abs else None,
                                   rows, cols, batch)
        return (y, ya) if with_abs else y

    # -- nonlinear codebook blocks ------------------------------------------
    def cb4_unpack(self, blk: np.ndarray, kv: np.ndarray):
        blk = _u8(blk).reshape(-1)[:CB4_BYTES].copy()
        kv = np.ascontiguousarray(kv, dtype=np.int8)
        d = np.zeros(1, np.float64)
        c = np.zeros(32, np.int8)
        self.lib.oracle_cb4_unpack(_ptr(blk), _ptr(kv), _ptr(d), _ptr(c))
        return float(d[0]), c

    def dequant_cb4(self, W, kv, rows: int, cols: int) -> np.ndarray:
        W = _u8(W)
        kv = np.ascontiguousarray(kv, dtype=np.int8)
        out = np.empty((rows, cols), np.float64)
        self.lib.oracle_dequant_cb4(_ptr(W), _ptr(kv), _ptr(out), rows, cols)
        return out

    def subdots_cb4(self, W, kv, xq, rows: int, cols: int, batch: int) -> np.ndarray:
        W, xq = _u8(W), _u8(xq)
        kv = np.ascontiguousarray(kv, dtype=np.int8)
        out = np.empty((batch, rows, cols // 32), np.int32)
        self.lib.oracle_subdots_cb4(_ptr(W), _ptr(kv), _ptr(xq), _ptr(out), rows, cols, batch)
        return out

    def matvec_cb4(self, W, kv, xq, rows: int, cols: int, batch: int, with_abs: bool = False):
        W, xq = _u8(W), _u8(xq)
        kv = np.ascontiguousarray(kv, dtype=np.int8)
        y = np.empty((batch, rows), np.float64)
        ya = np.empty((batch, rows), np.float64) if with_abs else None
        self.lib.oracle_matvec_cb4(_ptr(W), _ptr(kv), _ptr(xq), _ptr(y),
                                   _ptr(ya) if with_abs else None, rows, cols, batch)
        return (y, ya) if with_abs else y


    # -- RMSNorm + q8 pack ---------------------------------------------------
    def rmsnorm_sumsq(self, x: np.ndarray) -> float:
        x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
        return float(self.lib.oracle_rmsnorm_sumsq(_ptr(x), x.size))

    def rmsnorm_scale(self, x: np.ndarray) -> float:
        x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
        return float(self.lib.oracle_rmsnorm_scale(_ptr(x), x.size))

    def rmsnorm_q8(self, x: np.ndarray):
        """x: f32 [batch, cols] -> (q8 blocks of y, y = x * scale as f32)."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        if x.ndim == 1:
            x = x[None, :]
        batch, cols = x.shape
        assert cols % 256 == 0
        xq = np.empty((batch, cols // 256, Q8_BYTES), np.uint8)
        y = np.empty((batch, cols), np.float32)
        self.lib.oracle_rmsnorm_q8(_ptr(x), _ptr(xq), _ptr(y), cols, batch)
        return xq, y

    # -- resident codebook rows ---------------------------------------------------
    def cb4r_row_bytes(self, cols: int) -> int:
        return int(self.lib.oracle_cb4r_row_bytes(cols // 32))

    def cb4r_prefix(self, cols: int) -> int:
        return int(self.lib.oracle_cb4r_prefix(cols // 32))

    def repack_cb4(self, src_blocks: np.ndarray, dst: np.ndarray, block_base: int,
                   n_blocks: int, cols: int) -> np.ndarray:
        """Moves raw blocks block_base.. (src holds exactly n_blocks of 18
        bytes) into the resident matrix dst (uint8, modified in place)."""
        src = _u8(src_blocks).reshape(-1)
        assert src.size >= 18 * n_blocks and dst.flags["C_CONTIGUOUS"] and dst.dtype == np.uint8
        self.lib.oracle_repack_cb4(_ptr(src), _ptr(dst), block_base, n_blocks, cols)
        return dst

    def repack_cb4_whole(self, W: np.ndarray, rows: int, cols: int) -> np.ndarray:
        dst = np.zeros(rows * self.cb4r_row_bytes(cols), np.uint8)
        return self.repack_cb4(W, dst, 0, rows * (cols // 32), cols)

    def dequant_cb4r(self, Wr, kv, rows: int, cols: int) -> np.ndarray:
        Wr = _u8(Wr)
        kv = np.ascontiguousarray(kv, dtype=np.int8)
        out = np.empty((rows, cols), np.float64)
        self.lib.oracle_dequant_cb4r(_ptr(Wr), _ptr(kv), _ptr(out), rows, cols)
        return out


_default: Oracle | None = None


def get() -> Oracle:
    """The real oracle (no planted fault)."""
    global _default
    if _default is None:
        _default = Oracle(0)
    return _default
