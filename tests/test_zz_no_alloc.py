"""The allocation-free decode step, xq_linear_q4k_static, called through the C
ABI.  It is for callers that cannot allocate device memory where they run the
step (a framework that owns all device memory through its own pool, a serving
loop that may not call cudaMalloc because it can synchronise the device), so
it takes its scratch from the library's fixed device array.

On two calls in a row, with different activations, its y must be the
workspace step's (xq_linear_q4k_ws) bit for bit -- the two run the same
kernels -- and within the parity tolerance of the oracle.  The cases cover
both plan forms: the fused launch, which needs no scratch, and the
quantise-once form, which writes the q8 blocks into the fixed array (the
plan says which), up to the array's limit of 819 q8 blocks; one block more
is refused.  Around the two calls neither the device's free memory nor
torch's allocator changes.

This file is collected last, so a run that stops at the first failure has run
every other test before it."""
import ctypes

import numpy as np
import pytest
import torch

import oracle_rows
import synthetic
from test_gpu_parity import check_y

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 256 * 1024
MAX_BLOCKS = SCRATCH_BYTES // 320  # 819 q8 blocks
XQ_EINVAL, XQ_ESHAPE = 1, 3


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


# (rows, cols, batch, whether the plan quantises once into the scratch)
CASES = [(4096, 14336, 4, 1), (300, 4096, 3, 1), (300, 4096, 2, 0), (77, 4096, 1, 0),
         (1000, 25600, 8, 1),
         (64, 69888, 3, 1)]  # the last: 3 * 273 = 819 q8 blocks, the whole array


@pytest.mark.parametrize("rows,cols,batch,once", CASES)
def test_static_step_matches_the_workspace_step(lib, orc, rows, cols, batch, once):
    m, fn, err = lib
    assert batch * cols // 256 <= MAX_BLOCKS
    W_np = synthetic.q4k_weights(rows, cols, rows + cols)
    W = torch.from_numpy(W_np).cuda()
    ws = torch.empty(m.linear_workspace_bytes(cols, batch), dtype=torch.uint8, device="cuda")
    xs = [synthetic.activations(batch, cols, 7 * call + batch, outlier_frac=0.001)
          for call in range(2)]
    xd = [torch.from_numpy(x).cuda() for x in xs]
    ys = [torch.full((batch, rows), float("nan"), dtype=torch.float32, device="cuda")
          for _ in range(2)]
    # one call first, so that the address lookup and the kernels' lazy loading
    # are behind the measured calls
    assert call_static(fn, xd[1], W, ys[1], rows, cols, batch) == 0, err().decode()
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    alloc0, reserved0 = torch.cuda.memory_allocated(), torch.cuda.memory_reserved()
    plans = []
    for call in range(2):  # two calls in a row, different activations
        ys[call].fill_(float("nan"))
        st = call_static(fn, xd[call], W, ys[call], rows, cols, batch)
        assert st == 0, err().decode()
        plans.append(m.last_plan())
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0, "device memory changed across the calls"
    assert torch.cuda.memory_allocated() == alloc0 and torch.cuda.memory_reserved() == reserved0
    for call in range(2):
        assert plans[call]["quantise_once"] == once, plans[call]
        y = ys[call].cpu().numpy()
        y_ws = m.linear_ws("q4k", xd[call], W, rows, cols, ws).cpu().numpy()
        assert m.last_plan()["quantise_once"] == once
        assert np.array_equal(y, y_ws), f"call {call}: not bit-identical to the workspace step"
        xq_ref = orc.quantize_q8(xs[call])
        y_ref = oracle_rows.matvec(orc, "q4k", W_np, None, xq_ref, rows, cols, batch)
        check_y(y, y_ref, f"static step {rows}x{cols} b{batch}, call {call}")
    assert m.device_status() == 0


def test_static_step_rejects_shapes_beyond_its_scratch(lib):
    m, fn, err = lib
    rows = 16
    for cols, batch in ((52480, 4), (65536, 4)):  # 820 and 1024 q8 blocks
        assert batch * cols // 256 > MAX_BLOCKS
        assert m.linear_workspace_bytes(cols, batch) > SCRATCH_BYTES
        W = torch.zeros(m.q4k_bytes(rows, cols), dtype=torch.uint8, device="cuda")
        x = torch.zeros((batch, cols), dtype=torch.float32, device="cuda")
        y = torch.zeros((batch, rows), dtype=torch.float32, device="cuda")
        before = m.launch_count(m.COUNT_LINEAR_Q4K)
        assert call_static(fn, x, W, y, rows, cols, batch) == XQ_ESHAPE
        assert b"fixed scratch" in err()
        assert m.launch_count(m.COUNT_LINEAR_Q4K) == before


def test_static_step_refuses_bad_arguments_before_any_launch(lib):
    m, fn, err = lib
    rows, cols, batch = 16, 4096, 1
    W = torch.zeros(m.q4k_bytes(rows, cols), dtype=torch.uint8, device="cuda")
    x = torch.zeros((batch, cols), dtype=torch.float32, device="cuda")
    y = torch.zeros((batch, rows), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    before = m.launch_count(m.COUNT_LINEAR_Q4K)
    assert fn(None, W.data_ptr(), y.data_ptr(), rows, cols, batch, stream) == XQ_EINVAL
    assert b"null" in err()
    assert fn(x.data_ptr(), W.data_ptr(), y.data_ptr(), rows, cols + 1, batch, stream) == XQ_ESHAPE
    assert fn(x.data_ptr(), W.data_ptr(), y.data_ptr(), rows, cols, 9, stream) == XQ_ESHAPE
    assert m.launch_count(m.COUNT_LINEAR_Q4K) == before
