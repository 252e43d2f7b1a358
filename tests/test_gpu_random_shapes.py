"""Seeded random shapes across every format and entry-point family: rows
1..700, cols 256..17920 (every row-group shape: whole rows in a box, row
segments with a ragged last segment), batch 1..8, both plans of the
workspace step, overlap on and off.  Exact dots and y within the parity gate
against the oracle; the fused, workspace and two-call forms bit-identical."""
import numpy as np
import pytest
import torch

import oracle_rows
import synthetic
from test_gpu_parity import check_y, dev

pytestmark = pytest.mark.gpu

N_CASES = 36


@pytest.fixture(scope="module")
def xq():
    import quantized_decode_mat_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    return m


def _draw(i):
    rng = np.random.Generator(np.random.PCG64(1000 + i))
    fmt = ("q4k", "cb4", "cb4r")[i % 3]
    nb = int(rng.choice([1, 2, 3, 4, 5, 8, 9, 16, 17, 31, 32, 33, 40, 56, 64, 70]))
    rows = int(rng.integers(1, 701))
    batch = int(rng.integers(1, 9))
    return fmt, rows, 256 * nb, batch, bool(i % 2)


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_shape(xq, orc, i):
    fmt, rows, cols, batch, overlap = _draw(i)
    seed = 77 * i + rows
    kv = synthetic.cb4_table()
    x = synthetic.activations(batch, cols, seed + 1, outlier_frac=0.001)
    W = (synthetic.q4k_weights(rows, cols, seed) if fmt == "q4k"
         else synthetic.cb4_weights(rows, cols, seed))
    Wd = dev(W)
    if fmt == "cb4r":
        Wd = xq.repack_cb4(Wd, rows, cols)
    xd = dev(x)
    xq_ref = orc.quantize_q8(x)
    ws = torch.full((xq.linear_workspace_bytes(cols, batch),), 0xFF, dtype=torch.uint8,
                    device="cuda")
    try:
        xq.set_overlap_launches(overlap)
        q8 = xq.quantize_q8(xd)
        if fmt == "q4k":
            dots = xq.subdots_q4k(Wd, q8, rows, cols)
            y_mv = xq.matvec_q4k(Wd, q8, rows, cols)
            y_lin = xq.linear_q4k(xd, Wd, rows, cols)
        elif fmt == "cb4":
            dots = xq.subdots_cb4(Wd, kv, q8, rows, cols)
            y_mv = xq.matvec_cb4(Wd, kv, q8, rows, cols)
            y_lin = xq.linear_cb4(xd, Wd, kv, rows, cols)
        else:
            dots = xq.subdots_cb4r(Wd, kv, q8, rows, cols)
            y_mv = xq.matvec_cb4r(Wd, kv, q8, rows, cols)
            y_lin = xq.linear_cb4r(xd, Wd, kv, rows, cols)
        ys = []
        for mode in (1, 2):
            xq.set_quantise_once_override(mode)
            ys.append(xq.linear_ws(fmt, xd, Wd, rows, cols, ws, table=kv))
        torch.cuda.synchronize()
    finally:
        xq.set_overlap_launches(False)
        xq.set_quantise_once_override(0)
    assert np.array_equal(q8.cpu().numpy(), xq_ref)
    ref_dots = (orc.subdots_q4k(W, xq_ref, rows, cols, batch) if fmt == "q4k"
                else orc.subdots_cb4(W, kv, xq_ref, rows, cols, batch))
    assert np.array_equal(dots.cpu().numpy(), ref_dots)
    y = y_mv.cpu().numpy()
    for other in (y_lin, *ys):
        assert np.array_equal(other.cpu().numpy(), y)
    y_ref = (orc.matvec_q4k(W, xq_ref, rows, cols, batch) if fmt == "q4k"
             else orc.matvec_cb4(W, kv, xq_ref, rows, cols, batch))
    check_y(y, y_ref, f"random {i}: {fmt} {rows}x{cols} b{batch} overlap {overlap}")
    assert xq.device_status() == 0


N_LARGE = 12


def _draw_large(i):
    rng = np.random.Generator(np.random.PCG64(5000 + i))
    fmt = ("q4k", "cb4", "cb4r")[i % 3]
    nb = int(rng.choice([4, 8, 16, 24, 31, 32, 40, 56, 64, 80]))
    rows = int(rng.integers(2000, 20000))
    batch = int(rng.integers(1, 9))
    return fmt, rows, 256 * nb, batch, bool(i % 2), rng


@pytest.mark.parametrize("i", range(N_LARGE))
def test_random_large_shape(xq, orc, i):
    """Seeded large shapes (2000..20000 rows), so the plans with many warps a
    CTA, both q8 staging paths and the row blocking are drawn at random too:
    the workspace step agrees bit for bit with the mat-vec on q8 blocks, and
    with the oracle on every row."""
    fmt, rows, cols, batch, overlap, _ = _draw_large(i)
    seed = 31 * i + rows
    kv = synthetic.cb4_table()
    x = synthetic.activations(batch, cols, seed + 1, outlier_frac=0.001)
    W = (synthetic.q4k_weights(rows, cols, seed) if fmt == "q4k"
         else synthetic.cb4_weights(rows, cols, seed))
    Wd = dev(W)
    if fmt == "cb4r":
        Wd = xq.repack_cb4(Wd, rows, cols)
    xd = dev(x)
    ws = torch.full((xq.linear_workspace_bytes(cols, batch),), 0xFF, dtype=torch.uint8,
                    device="cuda")
    try:
        xq.set_overlap_launches(overlap)
        y = xq.linear_ws(fmt, xd, Wd, rows, cols, ws, table=kv)
        q8 = xq.quantize_q8(xd)
        y_mv = (xq.matvec_q4k(Wd, q8, rows, cols) if fmt == "q4k"
                else xq.matvec_cb4(Wd, kv, q8, rows, cols) if fmt == "cb4"
                else xq.matvec_cb4r(Wd, kv, q8, rows, cols))
        torch.cuda.synchronize()
    finally:
        xq.set_overlap_launches(False)
    y = y.cpu().numpy()
    assert np.array_equal(y, y_mv.cpu().numpy())
    xq_ref = orc.quantize_q8(x)
    y_ref = oracle_rows.matvec(orc, "q4k" if fmt == "q4k" else "cb4", W, kv, xq_ref, rows, cols,
                               batch)
    check_y(y, y_ref, f"{fmt} {rows}x{cols} b{batch}")
    assert xq.device_status() == 0
