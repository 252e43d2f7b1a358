"""Overlapped launches (xq_set_overlap_launches): a launch may start while the
kernel before it on the stream finishes, touching only the weights before it
waits for that kernel.  A chain in which every kernel reads what the one
before it wrote must give the same bits as with overlap off, eagerly and
replayed from a CUDA graph."""
import numpy as np
import pytest
import torch

import synthetic

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def xq():
    import quantized_decode_mat_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    return m


def _chain(xq, W1, W2, Wc, kv, sel_src, slab, x, ws, Ww, wsw):
    """Each step's input is the previous step's output (square 4096 x 4096
    layers, and a wide-activation step that takes the quantise-once path)."""
    n = 4096
    y1 = xq.matvec_q4k(W1, xq.rmsnorm_q8(x), n, n)              # rmsnorm -> mat-vec
    y2 = xq.matvec_q4k(W2, xq.quantize_q8(y1), n, n)            # quantise reads y1
    y3 = xq.linear_ws("q4k", y2, W1, n, n, ws)                  # fused step on y2
    y4 = xq.norm_linear_cb4(y3, Wc, kv, n, n)                   # codebook on y3
    y5 = xq.linear_ws("q4k", torch.cat([y4, y3, y2, y1]), W2, n, n, ws)  # 64 blocks: once
    sel = (sel_src + y5[:1, :3].abs().argmin(dim=1, keepdim=True).int() * 0).reshape(-1)
    y6 = xq.matvec_id("q4k", slab, sel, xq.quantize_q8(y5[:1].contiguous()), 512, n, 3)
    # 8 vectors of 65536: the batch is split over launches, each a quantise
    # launch into the shared workspace and a mat-vec
    xw = y5.reshape(-1).repeat(32).reshape(8, 65536)
    y7 = xq.linear_ws("q4k", xw, Ww, 64, 65536, wsw)
    return [y1, y2, y3, y4, y5, y6, y7]


def test_overlapped_chain_is_bit_identical(xq):
    n = 4096
    W1 = torch.from_numpy(synthetic.q4k_weights(n, n, 1)).cuda()
    W2 = torch.from_numpy(synthetic.q4k_weights(n, n, 2)).cuda()
    Wc = torch.from_numpy(synthetic.cb4_weights(n, n, 3)).cuda()
    slab = torch.from_numpy(synthetic.q4k_weights(3 * 512, n, 4)).cuda()
    kv = synthetic.cb4_table()
    x = torch.from_numpy(synthetic.activations(1, n, 5)).cuda()
    sel_src = torch.tensor([[2], [0], [1]], dtype=torch.int32, device="cuda")
    ws = torch.empty(xq.linear_workspace_bytes(n, 4), dtype=torch.uint8, device="cuda")
    Ww = torch.from_numpy(synthetic.q4k_weights(64, 65536, 6)).cuda()
    wsw = torch.empty(xq.linear_workspace_bytes(65536, 8), dtype=torch.uint8, device="cuda")
    runs = {}
    try:
        for ov in (False, True):
            xq.set_overlap_launches(ov)
            assert xq.overlap_launches() == ov
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                eager = [t.clone() for t in _chain(xq, W1, W2, Wc, kv, sel_src, slab, x, ws, Ww,
                                                   wsw)]
                p = xq.last_plan()
                assert p["launches"] > 1 and p["quantise_once"] == 1
            s.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                outs = _chain(xq, W1, W2, Wc, kv, sel_src, slab, x, ws, Ww, wsw)
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize()
            runs[ov] = ([t.cpu().numpy() for t in eager], [t.cpu().numpy() for t in outs])
    finally:
        xq.set_overlap_launches(False)
    for k, (a, b) in enumerate(zip(runs[False][0], runs[True][0])):
        assert np.array_equal(a, b), f"eager step {k + 1}"
    for k, (a, b) in enumerate(zip(runs[False][0], runs[True][1])):
        assert np.array_equal(a, b), f"graph step {k + 1}"
    assert all(np.isfinite(a).all() for a in runs[False][0])
    assert xq.device_status() == 0


def test_two_streams_with_own_buffers(xq):
    """The end-to-end pattern: steps alternate between two streams, each with
    its own x, y and workspace, copies to and from pinned host memory in line,
    overlap on.  Every step's y equals the same step run alone."""
    rows, cols, batch = 4096, 14336, 2   # 112 q8 blocks: the quantise-once plan
    W = torch.from_numpy(synthetic.q4k_weights(rows, cols, 21)).cuda()
    xs_host = [torch.from_numpy(synthetic.activations(batch, cols, 30 + i)).pin_memory()
               for i in range(6)]
    ref = []
    ws0 = torch.empty(xq.linear_workspace_bytes(cols, batch), dtype=torch.uint8, device="cuda")
    for xh in xs_host:
        ref.append(xq.linear_ws("q4k", xh.cuda(), W, rows, cols, ws0).cpu().numpy())
    lanes = [{"s": torch.cuda.Stream(), "x": torch.empty((batch, cols), device="cuda"),
              "y": torch.empty((batch, rows), device="cuda"),
              "ws": torch.empty_like(ws0)} for _ in range(2)]
    outs = [torch.empty((batch, rows), dtype=torch.float32).pin_memory() for _ in xs_host]
    try:
        xq.set_overlap_launches(True)
        torch.cuda.synchronize()
        for i, xh in enumerate(xs_host):
            ln = lanes[i % 2]
            with torch.cuda.stream(ln["s"]):
                ln["x"].copy_(xh, non_blocking=True)
                xq.linear_ws("q4k", ln["x"], W, rows, cols, ln["ws"], out=ln["y"])
                outs[i].copy_(ln["y"], non_blocking=True)
        torch.cuda.synchronize()
    finally:
        xq.set_overlap_launches(False)
    for i in range(len(xs_host)):
        assert np.array_equal(outs[i].numpy(), ref[i]), f"step {i}"
