"""The oracle over every row of a large matrix, the rows split into contiguous
slices across host threads.

The oracle's C functions release the GIL while they run (ctypes foreign
calls), so the slices run in parallel; each slice is the oracle's own
computation on those rows, and the slices are put back together in row order.
Test infrastructure only, like the oracle itself."""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np


def _slices(rows: int, threads: int) -> list[tuple[int, int]]:
    per = -(-rows // threads)
    return [(r0, min(rows, r0 + per)) for r0 in range(0, rows, per)]


def _threads(rows: int) -> int:
    return max(1, min(os.cpu_count() or 1, 32, rows // 256 or 1))


def matvec(orc, fmt: str, W: np.ndarray, kv, xq_ref: np.ndarray, rows: int, cols: int,
           batch: int) -> np.ndarray:
    """y_ref [batch, rows] (binary64) of a Q4_K ("q4k") or codebook ("cb4",
    raw blocks) matrix."""
    def part(s):
        r0, r1 = s
        Ws = W[r0:r1]
        if fmt == "q4k":
            return orc.matvec_q4k(Ws, xq_ref, r1 - r0, cols, batch)
        return orc.matvec_cb4(Ws, kv, xq_ref, r1 - r0, cols, batch)
    with ThreadPoolExecutor(_threads(rows)) as ex:
        parts = list(ex.map(part, _slices(rows, _threads(rows))))
    return np.concatenate(parts, axis=1)


def subdots(orc, fmt: str, W: np.ndarray, kv, xq_ref: np.ndarray, rows: int, cols: int,
            batch: int) -> np.ndarray:
    """The exact int32 dots [batch, rows, cols/32] of every row."""
    def part(s):
        r0, r1 = s
        Ws = W[r0:r1]
        if fmt == "q4k":
            return orc.subdots_q4k(Ws, xq_ref, r1 - r0, cols, batch)
        return orc.subdots_cb4(Ws, kv, xq_ref, r1 - r0, cols, batch)
    with ThreadPoolExecutor(_threads(rows)) as ex:
        parts = list(ex.map(part, _slices(rows, _threads(rows))))
    return np.concatenate(parts, axis=1)
