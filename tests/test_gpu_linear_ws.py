"""GPU parity of the decode step with a workspace (xq_linear_*_ws): the same
y bits as the fused step and as quantise-then-mat-vec, in both of its forms
(every CTA quantises; quantise once into the workspace, then the mat-vec),
within tolerance of the oracle, and replayable from a CUDA graph."""
import numpy as np
import pytest
import torch

import oracle_rows
import synthetic
from test_gpu_parity import Guarded, check_y, dev, run_quantize

pytestmark = pytest.mark.gpu

SHAPES = [(1, 256, 1), (101, 1024, 2), (300, 4096, 1), (77, 4096, 8), (64, 14336, 3),
          (37, 14336, 8), (5, 65536, 8), (1000, 2304, 4)]


@pytest.fixture(scope="module")
def xq():
    import quantized_decode_mat_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    return m


def _case(orc, fmt, rows, cols, batch):
    seed = 13 * rows + cols + batch
    kv = synthetic.cb4_table()
    x = synthetic.activations(batch, cols, seed + 1, outlier_frac=0.001)
    if fmt == "q4k":
        W = synthetic.q4k_weights(rows, cols, seed)
        Wdev = W
    else:
        W = synthetic.cb4_weights(rows, cols, seed)
        Wdev = W if fmt == "cb4" else orc.repack_cb4_whole(W.reshape(-1), rows, cols)
    return W, dev(Wdev), kv, x


def _reference_y(xq, fmt, Wd, kv, xd, rows, cols):
    if fmt == "q4k":
        return xq.linear_q4k(xd, Wd, rows, cols)
    if fmt == "cb4":
        return xq.linear_cb4(xd, Wd, kv, rows, cols)
    return xq.linear_cb4r(xd, Wd, kv, rows, cols)


@pytest.mark.parametrize("fmt", ["q4k", "cb4", "cb4r"])
@pytest.mark.parametrize("rows,cols,batch", SHAPES)
@pytest.mark.parametrize("mode", [1, 2, 0])
def test_linear_ws_is_the_fused_step(xq, orc, fmt, rows, cols, batch, mode):
    W, Wd, kv, x = _case(orc, fmt, rows, cols, batch)
    xd = dev(x)
    y_ref_gpu = _reference_y(xq, fmt, Wd, kv, xd, rows, cols)
    ws = torch.full((xq.linear_workspace_bytes(cols, batch),), 0xFF, dtype=torch.uint8,
                    device="cuda")
    out = Guarded((batch, rows), torch.float32)
    try:
        xq.set_quantise_once_override(mode)
        before = xq.launch_count(xq.COUNT_QUANTISE_ONCE)
        xq.linear_ws(fmt, xd, Wd, rows, cols, ws, table=kv, out=out.t)
        torch.cuda.synchronize()
        p = xq.last_plan()
        after = xq.launch_count(xq.COUNT_QUANTISE_ONCE)
    finally:
        xq.set_quantise_once_override(0)
    out.check_guard()
    if mode == 1:
        assert p["quantise_once"] == 0
    if mode == 2:
        assert p["quantise_once"] == 1
    assert after - before == (p["launches"] if p["quantise_once"] else 0)
    y = out.t.cpu().numpy()
    assert np.array_equal(y, y_ref_gpu.cpu().numpy())
    xq_ref = orc.quantize_q8(x)
    y_ref = (orc.matvec_q4k(W, xq_ref, rows, cols, batch) if fmt == "q4k"
             else orc.matvec_cb4(W, kv, xq_ref, rows, cols, batch))
    check_y(y, y_ref, f"linear ws {fmt} {rows}x{cols} b{batch} mode {mode}")
    assert xq.device_status() == 0


def test_quantise_once_writes_the_q8_blocks(xq, orc):
    """The workspace holds, after a quantise-once call, exactly the q8 blocks
    xq_quantize_q8 writes (all 320 bytes of each)."""
    rows, cols, batch = 200, 14336, 4
    W, Wd, kv, x = _case(orc, "q4k", rows, cols, batch)
    ws = torch.zeros(xq.linear_workspace_bytes(cols, batch), dtype=torch.uint8, device="cuda")
    try:
        xq.set_quantise_once_override(2)
        xq.linear_ws("q4k", dev(x), Wd, rows, cols, ws)
        torch.cuda.synchronize()
    finally:
        xq.set_quantise_once_override(0)
    n = xq.q8_bytes(cols, batch)
    assert np.array_equal(ws[:n].cpu().numpy().reshape(batch, cols // 256, 320),
                          orc.quantize_q8(x))


def test_linear_ws_graph_replay(xq, orc):
    """The two launches of the quantise-once form replay from a CUDA graph
    with the same bits, call after call."""
    rows, cols, batch = 4096, 14336, 2
    W, Wd, kv, x = _case(orc, "q4k", rows, cols, batch)
    xd = dev(x)
    ws = torch.empty(xq.linear_workspace_bytes(cols, batch), dtype=torch.uint8, device="cuda")
    y = torch.empty((batch, rows), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        xq.linear_ws("q4k", xd, Wd, rows, cols, ws, out=y)
    s.synchronize()
    assert xq.last_plan()["quantise_once"] == 1
    eager = y.cpu().numpy().copy()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):
            xq.linear_ws("q4k", xd, Wd, rows, cols, ws, out=y)
    for _ in range(4):
        y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(y.cpu().numpy(), eager)
    check_y(eager, orc.matvec_q4k(W, orc.quantize_q8(x), rows, cols, batch), "graph ws")
    assert xq.device_status() == 0


def test_linear_ws_rejects_a_small_workspace(xq):
    rows, cols, batch = 64, 4096, 2
    x = dev(synthetic.activations(batch, cols, 3))
    Wd = dev(synthetic.q4k_weights(rows, cols, 4))
    need = xq.linear_workspace_bytes(cols, batch)
    ws = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(xq.XQError) as e:
        xq.linear_ws("q4k", x, Wd, rows, cols, ws)
    assert e.value.status == 1 and "too small" in e.value.detail


@pytest.mark.parametrize("name", sorted(synthetic.CASES))
def test_step_at_full_size(xq, orc, name):
    """Every configuration at full size through the step the bench times
    (xq_linear_*_ws, planned as the bench plans it): every output of every
    row against the oracle."""
    c = synthetic.CASES[name]
    W, x = c.weights(), c.x()
    kv = synthetic.cb4_table()
    Wd = dev(W)
    if c.fmt == "cb4r":
        Wd = xq.repack_cb4(Wd, c.rows, c.cols)
    ws = torch.full((xq.linear_workspace_bytes(c.cols, c.batch),), 0xFF, dtype=torch.uint8,
                    device="cuda")
    out = Guarded((c.batch, c.rows), torch.float32)
    xq.linear_ws(c.fmt, dev(x), Wd, c.rows, c.cols, ws, table=kv, out=out.t)
    torch.cuda.synchronize()
    out.check_guard()
    y = out.t.cpu().numpy()
    xq_ref = orc.quantize_q8(x)
    y_ref = oracle_rows.matvec(orc, "q4k" if c.fmt == "q4k" else "cb4", W, kv, xq_ref, c.rows,
                               c.cols, c.batch)
    check_y(y, y_ref, f"step {name}")
