"""Seeded synthetic inputs shared by the oracle tests, the GPU parity tests and
the bench.

This module holds none of the mat-vec's arithmetic: it draws random bytes,
random f32 activations and random f16 scale fields, and knows the byte size
of each block format only to size its arrays.  Uniform random bytes in the
packed fields are uniform, independent 6-bit scales/mins and uniform nibbles,
because every bit of the twelve packed scale bytes and of every nibble byte
belongs to exactly one field.

Workloads (sizes, distributions) follow the five decode configurations:
  1. Q4_K 256x1024, batch 1 (tiny)
  2. Q4_K 4096x4096, batch 1, x with 0.1% outliers scaled x20
  3. Q4_K FFN pair 14336x4096 (up) and 4096x14336 (down), batch 1/2/4/8
  4. codebook 4096x4096 and 11008x4096, batch 1
  5. Q4_K 128256x4096 (L2-exceeding vocabulary projection), batch 1 and 8
and one measurement case beside them: the codebook format at the vocabulary
projection's shape, 128256x4096 batch 1 (raw and resident rows), so that the
codebook kernel also has a matrix larger than the L2 cache.
PRNG: numpy PCG64 (``np.random.Generator``); normals are numpy's standard
normal in float64, cast to float32.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

Q4K_BLOCK_BYTES = 144   # bytes per 256-weight super-block (sizing only)
CB4_BLOCK_BYTES = 18    # bytes per 32-weight codebook block (sizing only)
SEED_BASE = 0x51A7


def seed_for(cfg: int, stream: str) -> int:
    """Per-config seed streams: weights, activations, codebook table."""
    if stream == "W":
        return SEED_BASE + 16 * cfg
    if stream == "x":
        return SEED_BASE + 16 * cfg + 1
    if stream == "table":
        return SEED_BASE + 99
    raise ValueError(stream)


def _f16_bits(values: np.ndarray) -> np.ndarray:
    """float -> IEEE binary16 bit patterns, round to nearest even (numpy)."""
    return values.astype(np.float32).astype(np.float16).view(np.uint16)


def q4k_weights(rows: int, cols: int, seed: int, scale: float = 1e-3) -> np.ndarray:
    """Q4_K rows: uint8 [rows, cols/256*144].

    Per super-block: f16 d and f16 dmin drawn as |N(0,1)|*scale, then 140
    uniform random bytes (packed 6-bit scales/mins and nibbles).
    """
    assert cols % 256 == 0 and rows >= 0
    nb = cols // 256
    rng = np.random.Generator(np.random.PCG64(seed))
    W = rng.integers(0, 256, size=(rows, nb, Q4K_BLOCK_BYTES), dtype=np.uint8)
    dd = np.abs(rng.standard_normal((rows, nb, 2))) * scale
    W[:, :, 0:4] = _f16_bits(dd).reshape(rows, nb, 2).view(np.uint8).reshape(rows, nb, 4)
    return W.reshape(rows, nb * Q4K_BLOCK_BYTES)


def cb4_weights(rows: int, cols: int, seed: int, scale: float = 1e-2) -> np.ndarray:
    """Codebook rows: uint8 [rows, cols/32*18]; f16 d = |N(0,1)|*scale, then
    16 uniform random payload bytes per block."""
    assert cols % 32 == 0
    bpr = cols // 32
    rng = np.random.Generator(np.random.PCG64(seed))
    W = rng.integers(0, 256, size=(rows, bpr, CB4_BLOCK_BYTES), dtype=np.uint8)
    d = np.abs(rng.standard_normal((rows, bpr, 1))) * scale
    W[:, :, 0:2] = _f16_bits(d).reshape(rows, bpr, 1).view(np.uint8).reshape(rows, bpr, 2)
    return W.reshape(rows, bpr * CB4_BLOCK_BYTES)


def cb4_table(seed: int = SEED_BASE + 99) -> np.ndarray:
    """Seeded monotone 16-entry int8 codebook: kv[0] = -127, kv[15] = 113 and
    14 distinct interior integers drawn without replacement from (-127, 113),
    sorted ascending."""
    rng = np.random.Generator(np.random.PCG64(seed))
    interior = rng.choice(np.arange(-126, 113), size=14, replace=False)
    kv = np.concatenate([[-127], np.sort(interior), [113]]).astype(np.int8)
    return kv


def activations(batch: int, cols: int, seed: int, outlier_frac: float = 0.0,
                outlier_gain: float = 20.0) -> np.ndarray:
    """float32 [batch, cols] ~ N(0,1); optionally round(outlier_frac*cols)
    distinct positions per vector multiplied by ``outlier_gain``."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal((batch, cols)).astype(np.float32)
    k = int(round(outlier_frac * cols))
    for b in range(batch):
        if k:
            pos = rng.choice(cols, size=k, replace=False)
            x[b, pos] *= np.float32(outlier_gain)
    return x


def guide_fixture_x(cols: int) -> np.ndarray:
    """The guide's deterministic activation fixture x[j] = ((j % 25) - 12)/64
    ("Writing XPU Kernels", 25.7.1)."""
    j = np.arange(cols)
    return (((j % 25) - 12).astype(np.float32) / np.float32(64.0)).astype(np.float32)


@dataclass(frozen=True)
class MatvecCase:
    name: str
    fmt: str            # "q4k", "cb4", or "cb4r" (the codebook matrix, held in resident rows)
    rows: int
    cols: int
    batch: int
    cfg: int
    outliers: float = 0.0
    sub: int = 0        # second matrix of a config (the FFN down projection)

    @property
    def w_bytes(self) -> int:
        if self.fmt == "q4k":
            return self.rows * (self.cols // 256) * Q4K_BLOCK_BYTES
        return self.rows * (self.cols // 32) * CB4_BLOCK_BYTES

    def weights(self) -> np.ndarray:
        s = seed_for(self.cfg, "W") + 2 * self.sub
        if self.fmt == "q4k":
            return q4k_weights(self.rows, self.cols, s)
        return cb4_weights(self.rows, self.cols, s)

    def x(self) -> np.ndarray:
        return activations(self.batch, self.cols, seed_for(self.cfg, "x") + 2 * self.sub,
                           self.outliers)


# The five configurations as individual mat-vec cases.
CASES = {
    "c1_q4k_256x1024_b1": MatvecCase("c1_q4k_256x1024_b1", "q4k", 256, 1024, 1, 1),
    "c2_q4k_4096x4096_b1": MatvecCase("c2_q4k_4096x4096_b1", "q4k", 4096, 4096, 1, 2, 0.001),
    **{f"c3_q4k_up_14336x4096_b{b}": MatvecCase(f"c3_q4k_up_14336x4096_b{b}", "q4k", 14336,
                                                4096, b, 3) for b in (1, 2, 4, 8)},
    **{f"c3_q4k_down_4096x14336_b{b}": MatvecCase(f"c3_q4k_down_4096x14336_b{b}", "q4k", 4096,
                                                  14336, b, 3, sub=1) for b in (1, 2, 4, 8)},
    "c4_cb4_4096x4096_b1": MatvecCase("c4_cb4_4096x4096_b1", "cb4", 4096, 4096, 1, 4),
    "c4_cb4_11008x4096_b1": MatvecCase("c4_cb4_11008x4096_b1", "cb4", 11008, 4096, 1, 4,
                                         sub=1),
    # the same codebook matrices, repacked into resident rows by the library
    "c4_cb4r_4096x4096_b1": MatvecCase("c4_cb4r_4096x4096_b1", "cb4r", 4096, 4096, 1, 4),
    "c4_cb4r_11008x4096_b1": MatvecCase("c4_cb4r_11008x4096_b1", "cb4r", 11008, 4096, 1, 4,
                                          sub=1),
    "c5_q4k_128256x4096_b1": MatvecCase("c5_q4k_128256x4096_b1", "q4k", 128256, 4096, 1, 5),
    "c5_q4k_128256x4096_b8": MatvecCase("c5_q4k_128256x4096_b8", "q4k", 128256, 4096, 8, 5),
    # the codebook format with W larger than the L2 cache (295.5 MB), raw blocks
    # and the same matrix in resident rows
    "hbm_cb4_128256x4096_b1": MatvecCase("hbm_cb4_128256x4096_b1", "cb4", 128256, 4096, 1, 6),
    "hbm_cb4r_128256x4096_b1": MatvecCase("hbm_cb4r_128256x4096_b1", "cb4r", 128256, 4096, 1,
                                          6),
}
