"""Why the kernels carry each super-block's term as an unevaluated pair of
f32 values to the end of the row sum.

y = sum over super-blocks b of xs_b * (d_b * S1_b - dmin_b * S2_b), with S1
and S2 exact integers.  Rounding each term once to f32, even if the rounded
terms are then added exactly, already leaves outputs of configuration 2
(Q4_K 4096 x 4096, x with outliers) outside the parity gate
|y - y_ref| <= 1e-5 |y_ref| + 1e-6, while the exact terms reproduce the
oracle's y.  Everything here comes from the oracle (its exact sub-block dots,
its q8 blocks, its y) and the block format's field layout."""
import numpy as np

import synthetic

REL, ABS = 1e-5, 1e-6


def _terms(orc, name):
    c = synthetic.CASES[name]
    W, x = c.weights(), c.x()
    nb = c.cols // 256
    xq = orc.quantize_q8(x)
    y_ref = orc.matvec_q4k(W, xq, c.rows, c.cols, c.batch)
    dots = orc.subdots_q4k(W, xq, c.rows, c.cols, c.batch).astype(np.int64)
    dots = dots.reshape(c.batch, c.rows, nb, 8)
    blk = W.reshape(c.rows, nb, 144)
    d = blk[:, :, 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    dmin = blk[:, :, 2:4].copy().view(np.float16)[..., 0].astype(np.float64)
    s = blk[:, :, 4:16].astype(np.int64)
    sc = np.empty((c.rows, nb, 8), np.int64)
    m = np.empty_like(sc)
    for j in range(4):  # the k-quant packing of the twelve scale bytes
        sc[..., j] = s[..., j] & 63
        m[..., j] = s[..., j + 4] & 63
        sc[..., j + 4] = (s[..., j + 8] & 15) | ((s[..., j] >> 6) << 4)
        m[..., j + 4] = (s[..., j + 8] >> 4) | ((s[..., j + 4] >> 6) << 4)
    q = xq.reshape(c.batch, nb, 320)
    bsum = q[:, :, 256:288].copy().view(np.int32).astype(np.int64)
    xs = q[:, :, 288:292].copy().view(np.float32)[..., 0].astype(np.float64)
    S1 = (dots * sc[None]).sum(-1)
    S2 = (bsum[:, None] * m[None]).sum(-1)
    return xs[:, None, :] * (d[None] * S1 - dmin[None] * S2), y_ref


def _outside(y, y_ref):
    return int((np.abs(y - y_ref) > REL * np.abs(y_ref) + ABS).sum())


def test_one_rounding_per_term_is_not_enough(orc):
    terms, y_ref = _terms(orc, "c2_q4k_4096x4096_b1")
    # the exact terms give the oracle's y (to binary64 rounding)
    assert _outside(terms.sum(-1), y_ref) == 0
    assert np.allclose(terms.sum(-1), y_ref, rtol=1e-12, atol=1e-12)
    # each term rounded once to f32, the rounded terms added exactly
    rounded = terms.astype(np.float32).astype(np.float64).sum(-1)
    y = rounded.astype(np.float32).astype(np.float64)
    assert _outside(y, y_ref) >= 1
