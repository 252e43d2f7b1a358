"""Pins that tie the CPU oracle to the pages and to mathematics.

Each pin takes an ``oracle.Oracle`` and raises ``AssertionError`` when the
oracle disagrees with something fixed outside the oracle: a hand-derived
golden value (tests/golden), a closed form, an invariant the format states, a
special case that reduces to a library routine (numpy's binary16 conversion,
numpy integer matmul), or a brute-force dequantised dot.  The same pins run
against planted-fault builds of the oracle (tests/test_oracle_faults.py) to
show that each kind of plausible mistake is caught.
"""
from __future__ import annotations

import json
import os

import numpy as np

import synthetic
from packing import f16_bits, make_q8_block, pack_cb4_block, pack_q4k_block

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _i32(b: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(b).view("<i4")


def _f32(b: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(b).view("<f4")


# ---------------------------------------------------------------- binary16
def pin_f16_all_patterns(o):
    """Every one of the 65536 binary16 patterns decodes as numpy's float16."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([o.f16_to_f64(int(h)) for h in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


# ---------------------------------------------------------------- q8 blocks
def pin_q8_hand_cases(o):
    g = _golden("q8_hand.json")
    for case in g["cases"]:
        x = np.zeros(256, np.float32)
        if case["name"] == "ramp j-128":
            x = (np.arange(256) - 128).astype(np.float32)
        for k, v in case.get("x_sparse", {}).items():
            x[int(k)] = v
        blk = o.quantize_q8(x[None, :])[0, 0]
        q = blk[:256].view(np.int8).astype(np.int64)
        if case["name"] == "ramp j-128":
            for k, v in case["q_at_k"].items():
                assert q[int(k) + 128] == v, (case["name"], k, q[int(k) + 128], v)
        else:
            want = np.zeros(256, np.int64)
            for k, v in case["q_sparse"].items():
                want[int(k)] = v
            assert np.array_equal(q, want), case["name"]
        assert list(_i32(blk[256:288])) == case["bsum"], (case["name"], list(_i32(blk[256:288])))
        assert int(blk[288:292].view("<u4")[0]) == case["d_bits"], case["name"]
        assert not blk[292:].any(), case["name"]


def _q8_invariants(x: np.ndarray, xq: np.ndarray):
    batch, cols = x.shape
    nb = cols // 256
    blocks = xq.reshape(batch, nb, 320)
    q = blocks[:, :, :256].view(np.int8).astype(np.int64)
    bsum = blocks[:, :, 256:288].copy().view("<i4").astype(np.int64)
    d = blocks[:, :, 288:292].copy().view("<f4")[..., 0].astype(np.float64)
    xb = x.reshape(batch, nb, 256).astype(np.float64)
    # (i) stored sub-block sums equal the sums of their int8 values
    assert np.array_equal(bsum, q.reshape(batch, nb, 8, 32).sum(axis=3))
    # (ii) round trip within half a scale step (f32 rounding slack 1e-4 step)
    err = np.abs(xb - d[..., None] * q)
    assert np.all(err <= d[..., None] * (0.5 + 1e-4)), float((err / np.maximum(d[..., None], 1e-300)).max())
    # (iii) the largest magnitude maps to 127 in every non-zero block
    amax = np.abs(xb).max(axis=2)
    nz = amax > 0
    assert np.all(np.abs(q).max(axis=2)[nz] == 127)
    assert np.all(q[~nz] == 0) and np.all(d[~nz] == 0)
    # (iv) the scale is one step of the grid that reaches amax: d*127 ~ amax
    assert np.allclose(d[nz] * 127.0, amax[nz], rtol=2e-7, atol=0)
    # (v) values stay in the symmetric range; padding bytes are zero
    assert q.min() >= -127 and q.max() <= 127
    assert not blocks[:, :, 292:].any()


def pin_q8_invariants(o):
    cases = [synthetic.activations(3, 1024, 11),
             synthetic.activations(2, 4096, 12, outlier_frac=0.001),
             synthetic.guide_fixture_x(2048)[None, :],
             np.zeros((1, 512), np.float32),
             (synthetic.activations(1, 768, 13) * np.float32(1e-30)).astype(np.float32)]
    for x in cases:
        _q8_invariants(x, o.quantize_q8(x))


def pin_q8_nonfinite_and_tiny(o):
    """The rule's edge cases, in closed form: a NaN value does not count
    towards amax and quantises to 0, so the block's bytes are those of the
    same block with 0 there; an inf makes amax inf, so iscale = 127/inf = 0,
    every finite value quantises to 0 and the inf to 0*inf = NaN -> 0, and
    d = inf; an all-NaN block is an all-zero block; and an amax so small that
    127/amax overflows to inf sends every nonzero value to +-127 (0 stays 0:
    0*inf = NaN -> 0) while d = amax/127 rounds to 0."""
    rng = np.random.Generator(np.random.PCG64(77))
    base = rng.standard_normal(256).astype(np.float32)
    # NaN at a few places == 0 at those places, byte for byte
    xn, xz = base.copy(), base.copy()
    xn[[3, 100, 255]] = np.nan
    xz[[3, 100, 255]] = 0.0
    assert np.array_equal(o.quantize_q8(xn[None, :]), o.quantize_q8(xz[None, :]))
    # an inf: all zeros, d = +inf
    xi = base.copy()
    xi[17] = -np.inf
    blk = o.quantize_q8(xi[None, :])[0, 0]
    assert not blk[:288].any()
    assert int(blk[288:292].view("<u4")[0]) == 0x7F800000
    # all NaN: the zero block
    blk = o.quantize_q8(np.full((1, 256), np.nan, np.float32))[0, 0]
    assert not blk.any()
    # amax of two smallest subnormals: 127/amax = inf
    xt = np.zeros(256, np.float32)
    tiny = np.float32(np.ldexp(1.0, -149))  # the smallest positive subnormal
    xt[0], xt[1], xt[40] = tiny, -2 * tiny, tiny
    with np.errstate(over="ignore"):
        assert np.isinf(np.float32(127.0) / np.float32(2 * tiny))
    blk = o.quantize_q8(xt[None, :])[0, 0]
    q = blk[:256].view(np.int8).astype(np.int64)
    want = np.zeros(256, np.int64)
    want[0], want[1], want[40] = 127, -127, 127
    assert np.array_equal(q, want)
    assert list(_i32(blk[256:288])) == [0, 127, 0, 0, 0, 0, 0, 0]
    assert int(blk[288:292].view("<u4")[0]) == 0  # 2^-148 / 127 rounds to +0


# ---------------------------------------------------------------- Q4_K
def pin_q4k_scale_pack(o):
    g = _golden("q4k_scale_pack.json")
    blk = np.zeros(144, np.uint8)
    blk[4:16] = g["scale_bytes"]
    _, _, sc, m, _ = o.q4k_unpack(blk)
    assert list(sc) == g["sc"] and list(m) == g["m"], (list(sc), list(m))


def pin_q4k_roundtrip(o):
    rng = np.random.Generator(np.random.PCG64(7))
    for _ in range(64):
        sc = rng.integers(0, 64, 8)
        m = rng.integers(0, 64, 8)
        q = rng.integers(0, 16, 256)
        dv, dmv = rng.random() * 0.01, rng.random() * 0.01
        blk = pack_q4k_block(f16_bits(dv), f16_bits(dmv), sc, m, q)
        d, dmin, sc2, m2, q2 = o.q4k_unpack(blk)
        assert np.array_equal(sc2, sc) and np.array_equal(m2, m) and np.array_equal(q2, q)
        assert d == float(np.float16(dv)) and dmin == float(np.float16(dmv))


def _q4k_golden_case(case):
    blk = np.zeros(144, np.uint8)
    blk[0:2] = np.array([case["d_bits"]], "<u2").view(np.uint8)
    blk[2:4] = np.array([case["dmin_bits"]], "<u2").view(np.uint8)
    blk[4:16] = case["scale_bytes"]
    for g, byte in enumerate(case["group_bytes"]):
        blk[16 + 32 * g:16 + 32 * g + 32] = byte
    q8 = np.repeat(np.array(case["q8_per_subblock"]), 32)
    xq = make_q8_block(q8, xs_bits=case["xs_bits"])
    return blk, xq


def pin_q4k_block_y(o):
    for case in _golden("q4k_block_y.json")["cases"]:
        blk, xq = _q4k_golden_case(case)
        y = o.matvec_q4k(blk[None, :], xq[None, None, :], 1, 256, 1)
        assert y[0, 0] == case["y"], (case["name"], y[0, 0], case["y"])


def pin_q4k_bruteforce(o):
    """Integer route == dequantise-then-dot in binary64 (exact arithmetic
    identity; the only differences are binary64 roundings)."""
    for rows, cols, batch, seed in ((5, 512, 2, 21), (3, 1024, 1, 22), (7, 256, 3, 23)):
        W = synthetic.q4k_weights(rows, cols, seed)
        x = synthetic.activations(batch, cols, seed + 100)
        xq = o.quantize_q8(x)
        y, yabs = o.matvec_q4k(W, xq, rows, cols, batch, with_abs=True)
        ref = o.dequant_q8(xq, cols) @ o.dequant_q4k(W, rows, cols).T
        assert np.all(np.abs(y - ref) <= 1e-12 * yabs + 1e-300), np.abs(y - ref).max()
        # the guide's bound: within 1e-4 relative of the brute force
        assert np.all(np.abs(y - ref) <= 1e-4 * np.abs(ref) + 1e-12)


def _special_q8(rng, batch, cols):
    """Integer-valued activations with amax 127 in every block, so that the
    q8 quantiser yields q = x and scale 1 exactly."""
    x = rng.integers(-127, 128, size=(batch, cols)).astype(np.float32)
    x.reshape(batch, cols // 256, 256)[:, :, 5] = 127.0
    return x


def pin_q4k_gemv_special(o):
    """All sc = 1, m = 0, d = 1 and xs = 1: y is the plain integer GEMV of the
    nibble matrix with the activation (numpy int64 matmul)."""
    rng = np.random.Generator(np.random.PCG64(31))
    rows, cols, batch = 6, 768, 2
    Q = rng.integers(0, 16, size=(rows, cols))
    W = np.concatenate([np.concatenate([pack_q4k_block(0x3C00, 0x3C00, [1] * 8, [0] * 8,
                                                       Q[r, 256 * k:256 * k + 256])
                                        for k in range(cols // 256)]) for r in range(rows)])
    x = _special_q8(rng, batch, cols)
    xq = o.quantize_q8(x)
    assert np.all(xq.reshape(batch, -1, 320)[:, :, 288:292].copy().view("<f4") == 1.0)
    y = o.matvec_q4k(W, xq, rows, cols, batch)
    ref = x.astype(np.int64) @ Q.T.astype(np.int64)
    assert np.array_equal(y, ref.astype(np.float64))
    dots = o.subdots_q4k(W, xq, rows, cols, batch)
    ref_d = np.einsum("bks,rks->brk", x.astype(np.int64).reshape(batch, -1, 32),
                      Q.reshape(rows, -1, 32).astype(np.int64))
    assert np.array_equal(dots, ref_d)


def pin_q4k_min_term(o):
    """Closed form of the min term: nibbles all 0 leave only -dmin*m*xs*bsum."""
    rng = np.random.Generator(np.random.PCG64(41))
    m = rng.integers(0, 64, 8)
    blk = pack_q4k_block(0x3C00, f16_bits(0.5), [7] * 8, m, [0] * 256)
    qv = rng.integers(-127, 128, 256)
    xq = make_q8_block(qv, xs=2.0)
    y = o.matvec_q4k(blk[None, :], xq[None, None, :], 1, 256, 1)
    want = -0.5 * 2.0 * float((m * qv.reshape(8, 32).sum(axis=1)).sum())
    assert y[0, 0] == want, (y[0, 0], want)


# ---------------------------------------------------------------- codebook
def pin_cb4_block_y(o):
    g = _golden("cb4_block_y.json")
    kv = np.array(g["kv"], np.int8)
    ones = make_q8_block(np.ones(256, np.int64), xs=1.0)
    c0, c1, c2 = g["cases"]
    for k in range(16):
        blk = pack_cb4_block(0x3C00, [k] * 32)
        row = np.concatenate([blk] + [pack_cb4_block(0, [0] * 32)] * 7)
        y = o.matvec_cb4(row[None, :], kv, ones[None, None, :], 1, 256, 1)
        assert y[0, 0] == c0["y_by_k"][k], (k, y[0, 0])
    pm = np.concatenate([np.ones(16), -np.ones(16), np.zeros(224)]).astype(np.int64)
    row = np.concatenate([pack_cb4_block(0x3C00, [0] * 16 + [15] * 16)]
                         + [pack_cb4_block(0, [0] * 32)] * 7)
    y = o.matvec_cb4(row[None, :], kv, make_q8_block(pm, xs=1.0)[None, None, :], 1, 256, 1)
    assert y[0, 0] == c1["y"], y[0, 0]
    row = np.concatenate([pack_cb4_block(0x3C00, [k] * 32) for k in range(16)])
    xq = np.stack([make_q8_block(np.ones(256, np.int64), xs=1.0),
                   make_q8_block(np.ones(256, np.int64), xs=2.0)])
    y = o.matvec_cb4(row[None, :], kv, xq[None, :, :], 1, 512, 1)
    assert y[0, 0] == c2["y"], y[0, 0]
    dots = o.subdots_cb4(row[None, :], kv, xq[None, :, :], 1, 512, 1)
    assert list(dots[0, 0]) == [32 * int(v) for v in kv]


def pin_cb4_bruteforce(o):
    kv = synthetic.cb4_table()
    for rows, cols, batch, seed in ((5, 512, 2, 51), (3, 1024, 1, 52)):
        W = synthetic.cb4_weights(rows, cols, seed)
        x = synthetic.activations(batch, cols, seed + 100)
        xq = o.quantize_q8(x)
        y, yabs = o.matvec_cb4(W, kv, xq, rows, cols, batch, with_abs=True)
        ref = o.dequant_q8(xq, cols) @ o.dequant_cb4(W, kv, rows, cols).T
        assert np.all(np.abs(y - ref) <= 1e-12 * yabs + 1e-300), np.abs(y - ref).max()


def pin_cb4_gemv_special(o):
    """d = 1 and xs = 1: y is the integer GEMV of the decoded table values with
    the activation (numpy int64 matmul)."""
    rng = np.random.Generator(np.random.PCG64(61))
    kv = synthetic.cb4_table()
    rows, cols, batch = 4, 512, 2
    idx = rng.integers(0, 16, size=(rows, cols))
    W = np.concatenate([np.concatenate([pack_cb4_block(0x3C00, idx[r, 32 * k:32 * k + 32])
                                        for k in range(cols // 32)]) for r in range(rows)])
    x = _special_q8(rng, batch, cols)
    xq = o.quantize_q8(x)
    y = o.matvec_cb4(W, kv, xq, rows, cols, batch)
    C = kv.astype(np.int64)[idx]
    assert np.array_equal(y, (x.astype(np.int64) @ C.T).astype(np.float64))
    dots = o.subdots_cb4(W, kv, xq, rows, cols, batch)
    ref_d = np.einsum("bks,rks->brk", x.astype(np.int64).reshape(batch, -1, 32),
                      C.reshape(rows, -1, 32))
    assert np.array_equal(dots, ref_d)


# ---------------------------------------------------------------- RMSNorm + q8
_EPS32 = float(np.float32(1e-5))
_U32 = 2.0 ** -24          # unit roundoff of binary32


def _sparse_vector(case) -> np.ndarray:
    x = np.full(case["n"], case.get("x_rest", 0.0), np.float32)
    for k, v in case["x_sparse"].items():
        x[int(k)] = v
    return x


def pin_rmsnorm_order(o):
    """Hand-derived f32 sums of squares whose value depends on the summation
    order: the strided per-item loop, the butterfly inside a wave and the
    wave-0-upward order across waves."""
    for case in _golden("rmsnorm_hand.json")["sums"]:
        got = o.rmsnorm_sumsq(_sparse_vector(case))
        assert got == case["total"], (case["name"], got, case["total"])


def _scale_bound(n: int) -> float:
    """Relative error bound of the f32 scale against binary64: each square
    passes through one product, at most ceil(n/256) loop additions, five
    butterfly and eight cross-wave additions (positive terms, so the sum's
    relative error is at most that count times u); then the mean, the eps
    addition, sqrt (halves the relative error) and the reciprocal."""
    k = 1 + -(-n // 256) + 5 + 8
    return ((k + 2) / 2 + 2) * _U32 * 1.01


def _scale64(x: np.ndarray) -> float:
    import math
    s = math.fsum(float(v) * float(v) for v in x.astype(np.float64))
    return 1.0 / math.sqrt(s / x.size + _EPS32)


def pin_rmsnorm_hand(o):
    """The three-four case: q codes 95 and 127 whatever the scale's last bits,
    and the scale within the f32 error bound of the binary64 value."""
    case = _golden("rmsnorm_hand.json")["cases"][0]
    x = _sparse_vector(case)
    xq, y = o.rmsnorm_q8(x[None, :])
    q = xq[0, 0, :256].view(np.int8).astype(np.int64)
    want = np.zeros(256, np.int64)
    for k, v in case["q_sparse"].items():
        want[int(k)] = v
    assert np.array_equal(q, want)
    assert int(_i32(xq[0, 0, 256:260])[0]) == case["bsum0"]
    ref = _scale64(x)
    assert abs(o.rmsnorm_scale(x) - ref) <= _scale_bound(x.size) * ref
    assert abs(float(y[0, 1]) - 4.0 * ref) <= (_scale_bound(x.size) + _U32) * 4.0 * ref


def pin_rmsnorm_constant(o):
    """A constant vector c: the sum of squares n*c^2 is exact in every order
    (small multiples of a power of two), so the scale is 1/sqrt(c^2 + eps)
    within four roundings, and every q8 code of y is 127 with sub-block sums
    32*127."""
    for c, n in ((0.5, 1024), (2.0, 4096), (1.0, 256)):
        x = np.full(n, c, np.float32)
        assert o.rmsnorm_sumsq(x) == n * c * c
        ref = 1.0 / np.sqrt(c * c + _EPS32)
        assert abs(o.rmsnorm_scale(x) - ref) <= 4 * _U32 * ref
        xq, _ = o.rmsnorm_q8(x[None, :])
        q = xq[0, :, :256].view(np.int8)
        assert np.all(q == 127)
        assert np.all(xq[0, :, 256:288].copy().view("<i4") == 32 * 127)


def pin_rmsnorm_bound(o):
    """Seeded vectors of the decode widths (and one with outliers): the f32
    scale lies within its error bound of the binary64 value, y = x*scale
    within one more rounding, and the q8 blocks of y meet the block
    invariants."""
    cases = [synthetic.activations(2, 4096, 71),
             synthetic.activations(1, 14336, 72, outlier_frac=0.001),
             synthetic.activations(3, 768, 73),
             (synthetic.activations(1, 1024, 74) * np.float32(1e-3)).astype(np.float32)]
    for x in cases:
        xq, y = o.rmsnorm_q8(x)
        for b in range(x.shape[0]):
            ref = _scale64(x[b])
            bound = _scale_bound(x.shape[1])
            assert abs(o.rmsnorm_scale(x[b]) - ref) <= bound * ref
            err = np.abs(y[b].astype(np.float64) - x[b].astype(np.float64) * ref)
            assert np.all(err <= (bound + _U32) * 1.01 * np.abs(x[b].astype(np.float64)) * ref)
        _q8_invariants(y, xq)


# ---------------------------------------------------------------- resident codebook rows
def _raw_from_rule(scale_lo) -> np.ndarray:
    blocks = []
    for j, lo in enumerate(scale_lo):
        blocks.append(np.array([lo, 60] + [(16 * j + m) % 256 for m in range(16)], np.uint8))
    return np.concatenate(blocks)


def pin_cb4r_literal(o):
    """Hand-written resident bytes for three small matrices, one of them
    repacked in two chunks that cross a row boundary and one with a padded
    prefix."""
    for case in _golden("cb4_resident.json")["cases"]:
        rows, cols = case["rows"], case["cols"]
        raw = _raw_from_rule(case["scale_lo"])
        rb = sum(len(r["prefix"]) + r["payload_count"] for r in case["expect_rows"]) // rows
        assert o.cb4r_row_bytes(cols) == rb, (case["name"], o.cb4r_row_bytes(cols), rb)
        dst = np.full(rows * rb, case["fill"], np.uint8)
        for base, n in case["chunks"]:
            o.repack_cb4(raw[18 * base:18 * (base + n)], dst, base, n, cols)
        for r, want in enumerate(case["expect_rows"]):
            row = dst[r * rb:(r + 1) * rb]
            npf = len(want["prefix"])
            assert list(row[:npf]) == want["prefix"], (case["name"], r, list(row[:npf]))
            pay = np.arange(want["payload_from"], want["payload_from"] + want["payload_count"])
            assert np.array_equal(row[npf:], (pay % 256).astype(np.uint8)), (case["name"], r)


def pin_cb4r_chunks_and_weights(o):
    """Any chunking gives the same resident bytes, and the resident matrix
    holds the same weights as the raw one (the raw dequantisation is pinned
    separately)."""
    rng = np.random.Generator(np.random.PCG64(81))
    kv = synthetic.cb4_table()
    for rows, cols in ((3, 256), (5, 96), (4, 1024), (2, 4096)):
        W = synthetic.cb4_weights(rows, cols, seed=rows + cols).reshape(-1)
        whole = o.repack_cb4_whole(W, rows, cols)
        nblk = rows * (cols // 32)
        cuts = np.sort(rng.choice(np.arange(1, nblk), size=min(4, nblk - 1), replace=False))
        bounds = [0, *cuts.tolist(), nblk]
        dst = np.zeros_like(whole)
        for a, b in zip(bounds[:-1], bounds[1:]):
            o.repack_cb4(W[18 * a:18 * b], dst, a, b - a, cols)
        assert np.array_equal(dst, whole), (rows, cols)
        assert np.array_equal(o.dequant_cb4r(whole, kv, rows, cols),
                              o.dequant_cb4(W, kv, rows, cols)), (rows, cols)


ALL_PINS = [pin_f16_all_patterns, pin_q8_hand_cases, pin_q8_invariants, pin_q8_nonfinite_and_tiny,
            pin_q4k_scale_pack,
            pin_q4k_roundtrip, pin_q4k_block_y, pin_q4k_bruteforce, pin_q4k_gemv_special,
            pin_q4k_min_term, pin_cb4_block_y, pin_cb4_bruteforce, pin_cb4_gemv_special,
            pin_rmsnorm_order, pin_rmsnorm_hand, pin_rmsnorm_constant, pin_rmsnorm_bound,
            pin_cb4r_literal, pin_cb4r_chunks_and_weights]
