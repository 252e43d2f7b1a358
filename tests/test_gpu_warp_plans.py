"""The wide plans: 20 warps a CTA at batch 1 (codebook blocks, and the
Q4_K mat-vec behind a quantise launch), 16 for the codebook at batch 2..4,
12 for Q4_K at batch 2 and where 16 warps of two stages do not fit, and 16
for the fused RMSNorm form.  Each shape is large enough that the planner
takes that count; y is bit-identical to the same call at 8 warps (the warps
only split the work units) and within the parity gate of the oracle."""
import numpy as np
import pytest
import torch

import synthetic
from test_gpu_parity import check_y, dev

pytestmark = pytest.mark.gpu

# (format, rows, cols, batch, warps the step's plan takes)
STEPS = [
    ("cb4", 6000, 4096, 1, 20),
    ("cb4r", 6000, 4096, 1, 20),
    ("q4k", 4096, 14336, 1, 20),
    ("cb4", 5000, 4096, 2, 16),
    ("cb4", 5000, 4096, 3, 16),
    ("cb4r", 5000, 4096, 4, 16),
    ("q4k", 7500, 4096, 2, 12),
    ("cb4", 3000, 16384, 4, 12),
]


@pytest.fixture(scope="module")
def xq():
    import quantized_decode_mat_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    return m


def _case(orc, fmt, rows, cols, batch):
    seed = 31 * rows + cols + batch
    kv = synthetic.cb4_table()
    x = synthetic.activations(batch, cols, seed + 1, outlier_frac=0.001)
    if fmt == "q4k":
        W = synthetic.q4k_weights(rows, cols, seed)
        Wd = dev(W)
    else:
        W = synthetic.cb4_weights(rows, cols, seed)
        Wd = dev(W if fmt == "cb4" else orc.repack_cb4_whole(W.reshape(-1), rows, cols))
    y_ref = (orc.matvec_q4k(W, orc.quantize_q8(x), rows, cols, batch) if fmt == "q4k"
             else orc.matvec_cb4(W, kv, orc.quantize_q8(x), rows, cols, batch))
    return Wd, kv, x, y_ref


@pytest.mark.parametrize("fmt,rows,cols,batch,warps", STEPS)
def test_wide_step_plan(xq, orc, fmt, rows, cols, batch, warps):
    Wd, kv, x, y_ref = _case(orc, fmt, rows, cols, batch)
    xd = dev(x)
    ws = torch.empty(xq.linear_workspace_bytes(cols, batch), dtype=torch.uint8, device="cuda")
    y = xq.linear_ws(fmt, xd, Wd, rows, cols, ws, table=kv)
    torch.cuda.synchronize()
    p = xq.last_plan()
    assert p["warps"] == warps, p
    assert p["smem_bytes"] <= torch.cuda.get_device_properties(0).shared_memory_per_block_optin
    try:
        xq.set_plan_override(8, 0)
        y8 = xq.linear_ws(fmt, xd, Wd, rows, cols, ws, table=kv)
        torch.cuda.synchronize()
        assert xq.last_plan()["warps"] == 8
    finally:
        xq.set_plan_override(0, 0)
    y = y.cpu().numpy()
    assert np.array_equal(y, y8.cpu().numpy())
    check_y(y, y_ref, f"{fmt} {rows}x{cols} b{batch} at {warps} warps")
    assert xq.device_status() == 0


@pytest.mark.parametrize("fmt,rows,cols", [("q4k", 4096, 14336), ("cb4", 6000, 4096)])
def test_fused_rmsnorm_keeps_16_warps(xq, orc, fmt, rows, cols):
    """The fused RMSNorm form is built for at most 16 warps at batch 1 and is
    planned so, also where the plain step takes 20."""
    Wd, kv, x, _ = _case(orc, fmt, rows, cols, 1)
    xd = dev(x)
    if fmt == "q4k":
        y = xq.norm_linear_q4k(xd, Wd, rows, cols)
    else:
        y = xq.norm_linear_cb4(xd, Wd, kv, rows, cols)
    torch.cuda.synchronize()
    assert xq.last_plan()["warps"] == 16
    q8 = xq.rmsnorm_q8(xd)
    y2 = (xq.matvec_q4k(Wd, q8, rows, cols) if fmt == "q4k"
          else xq.matvec_cb4(Wd, kv, q8, rows, cols))
    assert np.array_equal(y.cpu().numpy(), y2.cpu().numpy())
