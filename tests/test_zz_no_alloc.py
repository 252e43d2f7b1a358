"""The allocation-free decode step, xq_linear_q4k_static, called through the C
ABI: it is for callers that cannot allocate device memory where they run the
step (a framework that owns all device memory, a serving loop that may not
call cudaMalloc), so it takes its scratch from the library's fixed device
array.  Its y must match the workspace step's (xq_linear_q4k_ws) within the
parity tolerance, on two calls in a row, in both plan forms (the fused launch,
which needs no scratch, and the quantise-once form, which uses it).

This file is collected last, so a run that stops at the first failure has run
every other test before it."""
import ctypes

import numpy as np
import pytest
import torch

import synthetic

pytestmark = pytest.mark.gpu

REL, ABS = 1e-5, 1e-6
SCRATCH_BYTES = 256 * 1024


@pytest.fixture(scope="module")
def lib():
    import quantized_decode_mat_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    raw = ctypes.CDLL(m.lib_path())
    fn = raw.xq_linear_q4k_static
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                   ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]
    err = raw.xq_last_error
    err.restype = ctypes.c_char_p
    return m, fn, err


def call_static(fn, x, W, y, rows, cols, batch):
    stream = torch.cuda.current_stream().cuda_stream
    return fn(x.data_ptr(), W.data_ptr(), y.data_ptr(), rows, cols, batch, stream)


def within(y, ref):
    y, ref = y.astype(np.float64), ref.astype(np.float64)
    return np.all(np.abs(y - ref) <= REL * np.abs(ref) + ABS)


@pytest.mark.parametrize("rows,cols,batch", [(4096, 14336, 4), (300, 4096, 2), (77, 4096, 1),
                                             (1000, 25600, 8)])
def test_static_step_matches_the_workspace_step(lib, rows, cols, batch):
    m, fn, err = lib
    W = torch.from_numpy(synthetic.q4k_weights(rows, cols, rows + cols)).cuda()
    ws = torch.empty(m.linear_workspace_bytes(cols, batch), dtype=torch.uint8, device="cuda")
    for call in range(2):  # two calls in a row, different activations
        x = torch.from_numpy(synthetic.activations(batch, cols, 7 * call + batch,
                                                   outlier_frac=0.001)).cuda()
        y_ref = m.linear_ws("q4k", x, W, rows, cols, ws)
        y = torch.full((batch, rows), float("nan"), dtype=torch.float32, device="cuda")
        st = call_static(fn, x, W, y, rows, cols, batch)
        torch.cuda.synchronize()
        assert st == 0, err().decode()
        assert within(y.cpu().numpy(), y_ref.cpu().numpy()), f"call {call}"
    assert m.device_status() == 0


def test_static_step_rejects_shapes_beyond_its_scratch(lib):
    m, fn, err = lib
    rows, cols, batch = 16, 65536, 4  # 1024 q8 blocks, more than the 819 that fit
    assert m.linear_workspace_bytes(cols, batch) > SCRATCH_BYTES
    W = torch.zeros(m.q4k_bytes(rows, cols), dtype=torch.uint8, device="cuda")
    x = torch.zeros((batch, cols), dtype=torch.float32, device="cuda")
    y = torch.zeros((batch, rows), dtype=torch.float32, device="cuda")
    before = m.launch_count(m.COUNT_LINEAR_Q4K)
    assert call_static(fn, x, W, y, rows, cols, batch) == 3  # XQ_ESHAPE
    assert b"fixed scratch" in err()
    assert m.launch_count(m.COUNT_LINEAR_Q4K) == before
