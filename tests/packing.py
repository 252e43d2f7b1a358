"""Test-side block packers, written from the block layouts (the inverse
direction of the oracle's and the kernels' unpackers), used to build
hand-controlled blocks for the pins.

Q4_K super-block (144 bytes; stride and the nibble group offset 16+32g from
"cajeta.xpu - one kernel, any device" section 2.3; field layout as read for the
workload): f16 d @0, f16 dmin @2, twelve 6-bit scale/min bytes @4, nibbles @16.
Codebook block (18 bytes; "25 - Writing XPU Kernels" 25.2.1): f16 d @0, then
16 payload bytes whose low nibbles are elements 0..15 and high nibbles 16..31.
q8 activation block (320 bytes; 25.2): int8[256] @0, int32 sums[8] @256,
f32 scale @288, zero padding to 320.
"""
from __future__ import annotations

import numpy as np


def pack_scales(sc, m) -> np.ndarray:
    """Eight 6-bit scales and eight 6-bit mins -> twelve bytes.

    Bytes 0..3: low 6 bits = sc[0..3], top 2 bits = top 2 bits of sc[4..7].
    Bytes 4..7: low 6 bits = m[0..3],  top 2 bits = top 2 bits of m[4..7].
    Bytes 8..11: low nibble = low 4 bits of sc[4..7], high nibble = low 4 bits
    of m[4..7].
    """
    sc = [int(v) for v in sc]
    m = [int(v) for v in m]
    assert all(0 <= v < 64 for v in sc + m)
    out = np.zeros(12, np.uint8)
    for j in range(4):
        out[j] = sc[j] | ((sc[j + 4] >> 4) << 6)
        out[j + 4] = m[j] | ((m[j + 4] >> 4) << 6)
        out[j + 8] = (sc[j + 4] & 15) | ((m[j + 4] & 15) << 4)
    return out


def pack_q4k_block(d_bits: int, dmin_bits: int, sc, m, q) -> np.ndarray:
    """One 144-byte super-block from f16 bit patterns, scales/mins and the
    256 nibble values q[0..255] (weight order)."""
    q = np.asarray(q, dtype=np.int64)
    assert q.shape == (256,) and q.min() >= 0 and q.max() < 16
    blk = np.zeros(144, np.uint8)
    blk[0], blk[1] = d_bits & 0xFF, (d_bits >> 8) & 0xFF
    blk[2], blk[3] = dmin_bits & 0xFF, (dmin_bits >> 8) & 0xFF
    blk[4:16] = pack_scales(sc, m)
    for g in range(4):
        for i in range(32):
            blk[16 + 32 * g + i] = q[64 * g + i] | (q[64 * g + 32 + i] << 4)
    return blk


def pack_cb4_block(d_bits: int, idx) -> np.ndarray:
    """One 18-byte codebook block from an f16 bit pattern and 32 nibble
    indices (element order)."""
    idx = np.asarray(idx, dtype=np.int64)
    assert idx.shape == (32,) and idx.min() >= 0 and idx.max() < 16
    blk = np.zeros(18, np.uint8)
    blk[0], blk[1] = d_bits & 0xFF, (d_bits >> 8) & 0xFF
    for j in range(16):
        blk[2 + j] = idx[j] | (idx[j + 16] << 4)
    return blk


def make_q8_block(q, xs: float | None = None, xs_bits: int | None = None) -> np.ndarray:
    """A 320-byte activation block straight from int8 values and a scale
    (consistent sums, zero padding) -- for feeding hand cases to the mat-vec."""
    q = np.asarray(q, dtype=np.int64)
    assert q.shape == (256,) and q.min() >= -128 and q.max() <= 127
    blk = np.zeros(320, np.uint8)
    blk[:256] = q.astype(np.int8).view(np.uint8)
    blk[256:288] = q.reshape(8, 32).sum(axis=1).astype("<i4").view(np.uint8)
    if xs_bits is None:
        xs_bits = int(np.array([xs], dtype="<f4").view("<u4")[0])
    blk[288:292] = np.array([xs_bits], dtype="<u4").view(np.uint8)
    return blk


def f16_bits(v: float) -> int:
    return int(np.array([v], dtype=np.float16).view(np.uint16)[0])
