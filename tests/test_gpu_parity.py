"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the
same seeded inputs.

Bars (the decode workload's parity rules):
  * q8 blocks: all 320 bytes bit-exact (the quantiser decides integers in f32
    on both sides, one rounding per operation).
  * per-sub-block / per-block int32 dots: bit-exact.
  * y (f32): |y_gpu - y_ref| <= 1e-5 * |y_ref| + 1e-6 per element, y_ref the
    oracle's exact-integer / binary64 value.
Outputs are poisoned with 0xFF (NaN) before each launch and guarded by a
poisoned tail that must come back unchanged.
"""
import numpy as np
import pytest
import torch

import oracle_rows
import synthetic

pytestmark = pytest.mark.gpu

REL, ABS = 1e-5, 1e-6
GUARD = 256  # poisoned bytes after every output


@pytest.fixture(scope="module")
def xq():
    import quantized_decode_mat_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    return m


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda")


class Guarded:
    """An output tensor followed by a poisoned guard band in one allocation."""

    def __init__(self, shape, dtype):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.raw = torch.full((n + GUARD,), 0xFF, dtype=torch.uint8, device="cuda")
        self.t = self.raw[:n].view(dtype).view(shape)

    def check_guard(self):
        tail = self.raw[-GUARD:].cpu().numpy()
        assert np.all(tail == 0xFF), "write past the end of an output"


def check_y(y: np.ndarray, y_ref: np.ndarray, what: str):
    y = y.astype(np.float64)
    assert not np.isnan(y).any(), f"{what}: NaN in output (unwritten rows?)"
    err = np.abs(y - y_ref)
    tol = REL * np.abs(y_ref) + ABS
    bad = err > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {y.size} outside 1e-5 rel + 1e-6 abs; "
                           f"worst err {err.max():.3e} at |y| {np.abs(y_ref).flat[err.argmax()]:.3e}")
    assert np.any(y != 0), f"{what}: all-zero output"


def run_quantize(xq, x):
    batch, cols = x.shape
    out = Guarded((batch, cols // 256, 320), torch.uint8)
    xq.quantize_q8(dev(x), out=out.t)
    torch.cuda.synchronize()
    out.check_guard()
    return out.t


def run_matvec(xq, fmt, W, kv, xq_dev, rows, cols, batch, dots=False):
    if dots:
        out = Guarded((batch, rows, cols // 32), torch.int32)
    else:
        out = Guarded((batch, rows), torch.float32)
    Wd = dev(W)
    if fmt == "q4k":
        (xq.subdots_q4k if dots else xq.matvec_q4k)(Wd, xq_dev, rows, cols, out=out.t)
    elif dots:
        xq.subdots_cb4(Wd, kv, xq_dev, rows, cols, out=out.t)
    else:
        xq.matvec_cb4(Wd, kv, xq_dev, rows, cols, out=out.t)
    torch.cuda.synchronize()
    out.check_guard()
    return out.t.cpu().numpy()


# ---------------------------------------------------------------- q8 blocks
def _x_kind(kind, batch, cols, seed):
    if kind == "normal":
        return synthetic.activations(batch, cols, seed)
    if kind == "outliers":
        return synthetic.activations(batch, cols, seed, outlier_frac=0.001)
    if kind == "fixture":
        return np.tile(synthetic.guide_fixture_x(cols), (batch, 1))
    if kind == "zeros":
        return np.zeros((batch, cols), np.float32)
    if kind == "tiny":
        return (synthetic.activations(batch, cols, seed) * np.float32(1e-33)).astype(np.float32)
    if kind == "huge":
        return (synthetic.activations(batch, cols, seed) * np.float32(1e30)).astype(np.float32)
    if kind == "ties":
        rng = np.random.Generator(np.random.PCG64(seed))
        x = (rng.integers(-254, 255, size=(batch, cols)) / 2.0).astype(np.float32)
        x.reshape(batch, -1, 256)[:, :, 0] = 127.0
        return x
    if kind == "subnormal":
        # blocks scaled into and around the subnormal range: where amax is
        # below 127 / FLT_MAX, iscale = 127/amax overflows to inf and every
        # nonzero value must still land on +-127 (zeros on 0)
        x = synthetic.activations(batch, cols, seed).reshape(batch, -1, 256)
        scales = np.array([1e-45, 1e-41, 1e-39, 3e-38, 1e-37, 1e-36], np.float32)
        for k in range(x.shape[1]):
            x[:, k] *= scales[k % len(scales)]
        x[:, ::7, 3] = 0.0
        return x.reshape(batch, cols)
    if kind == "nonfinite":
        # NaN values do not count towards amax and quantise to 0; an inf
        # makes amax inf, iscale 0, the finite values 0 and the inf itself
        # 0 * inf = NaN -> 0
        x = synthetic.activations(batch, cols, seed).reshape(batch, -1, 256)
        nb = x.shape[1]
        x[:, 0, 5] = np.nan
        if nb > 1:
            x[:, 1, 17] = np.inf
        if nb > 2:
            x[:, 2, 200] = -np.inf
            x[:, 2, 201] = np.nan
        if nb > 3:
            x[:, 3, :] = np.nan
        if nb > 4:
            x[:, 4, :] = 0.0
            x[:, 4, 9] = np.nan
        return x.reshape(batch, cols)
    raise ValueError(kind)


@pytest.mark.parametrize("kind", ["normal", "outliers", "fixture", "zeros", "tiny", "huge",
                                  "ties", "subnormal", "nonfinite"])
@pytest.mark.parametrize("cols,batch", [(256, 1), (1024, 3), (4096, 8), (14336, 2)])
def test_quantize_bit_exact(xq, orc, kind, cols, batch):
    x = _x_kind(kind, batch, cols, 1000 + cols + batch)
    before = xq.launch_count(xq.COUNT_QUANTIZE)
    got = run_quantize(xq, x).cpu().numpy()
    assert xq.launch_count(xq.COUNT_QUANTIZE) == before + 1
    ref = orc.quantize_q8(x)
    diff = np.argwhere(got != ref)
    assert diff.size == 0, f"{len(diff)} bytes differ, first at {diff[:4].tolist()}"


# ---------------------------------------------------------------- exact dots
SHAPES = [(1, 256, 1), (31, 512, 2), (32, 1024, 1), (33, 1024, 4), (101, 2304, 3),
          (300, 4096, 1), (77, 4096, 8), (64, 14336, 2), (3, 169984, 2)]


def _weights(fmt, rows, cols, seed):
    return (synthetic.q4k_weights(rows, cols, seed) if fmt == "q4k"
            else synthetic.cb4_weights(rows, cols, seed))


@pytest.mark.parametrize("fmt", ["q4k", "cb4"])
@pytest.mark.parametrize("rows,cols,batch", SHAPES)
def test_subdots_bit_exact(xq, orc, fmt, rows, cols, batch):
    seed = rows * 7 + cols + batch
    W = _weights(fmt, rows, cols, seed)
    kv = synthetic.cb4_table()
    x = synthetic.activations(batch, cols, seed + 1)
    xq_dev = run_quantize(xq, x)
    which = xq.COUNT_SUBDOTS_Q4K if fmt == "q4k" else xq.COUNT_SUBDOTS_CB4
    before = xq.launch_count(which)
    got = run_matvec(xq, fmt, W, kv, xq_dev, rows, cols, batch, dots=True)
    assert xq.launch_count(which) == before + xq.last_plan()["launches"]
    xq_ref = orc.quantize_q8(x)
    ref = (orc.subdots_q4k(W, xq_ref, rows, cols, batch) if fmt == "q4k"
           else orc.subdots_cb4(W, kv, xq_ref, rows, cols, batch))
    diff = np.argwhere(got != ref)
    assert diff.size == 0, f"{len(diff)} dots differ, first at {diff[:4].tolist()}"


@pytest.mark.parametrize("fmt", ["q4k", "cb4"])
@pytest.mark.parametrize("rows,cols,batch", SHAPES)
def test_matvec_within_tolerance(xq, orc, fmt, rows, cols, batch):
    seed = rows * 11 + cols + batch
    W = _weights(fmt, rows, cols, seed)
    kv = synthetic.cb4_table()
    x = synthetic.activations(batch, cols, seed + 1, outlier_frac=0.001)
    xq_dev = run_quantize(xq, x)
    which = xq.COUNT_MATVEC_Q4K if fmt == "q4k" else xq.COUNT_MATVEC_CB4
    before = xq.launch_count(which)
    y = run_matvec(xq, fmt, W, kv, xq_dev, rows, cols, batch)
    assert xq.launch_count(which) == before + xq.last_plan()["launches"]
    xq_ref = orc.quantize_q8(x)
    y_ref = (orc.matvec_q4k(W, xq_ref, rows, cols, batch) if fmt == "q4k"
             else orc.matvec_cb4(W, kv, xq_ref, rows, cols, batch))
    check_y(y, y_ref, f"{fmt} {rows}x{cols} b{batch}")


# ---------------------------------------------------------------- the configurations
L2_BYTES = 129 * 1024 * 1024
SMALL_CASES = [k for k, c in synthetic.CASES.items()
               if c.w_bytes < L2_BYTES and c.fmt != "cb4r"]  # resident: test_gpu_resident
LARGE_CASES = [k for k, c in synthetic.CASES.items()
               if c.w_bytes >= L2_BYTES and c.fmt != "cb4r"]


@pytest.mark.parametrize("name", SMALL_CASES)
def test_config_full(xq, orc, name):
    """Configurations 1-4 at full size, every output against the oracle."""
    c = synthetic.CASES[name]
    W, x = c.weights(), c.x()
    kv = synthetic.cb4_table()
    xq_dev = run_quantize(xq, x)
    assert np.array_equal(xq_dev.cpu().numpy(), orc.quantize_q8(x))
    y = run_matvec(xq, c.fmt, W, kv, xq_dev, c.rows, c.cols, c.batch)
    xq_ref = orc.quantize_q8(x)
    y_ref = (orc.matvec_q4k(W, xq_ref, c.rows, c.cols, c.batch) if c.fmt == "q4k"
             else orc.matvec_cb4(W, kv, xq_ref, c.rows, c.cols, c.batch))
    check_y(y, y_ref, name)


@pytest.mark.parametrize("name", LARGE_CASES)
def test_large_config_every_row(xq, orc, name):
    """The L2-exceeding vocabulary projection at full size (configuration 5,
    and the codebook format at the same shape), in the launch configuration
    the bench times: every output of every row against the oracle (so an
    unwritten row anywhere shows as NaN poison), and every exact sub-block
    dot of every row bit for bit."""
    c = synthetic.CASES[name]
    W, x = c.weights(), c.x()
    kv = synthetic.cb4_table()
    xq_dev = run_quantize(xq, x)
    xq_ref = orc.quantize_q8(x)
    assert np.array_equal(xq_dev.cpu().numpy(), xq_ref)
    y = run_matvec(xq, c.fmt, W, kv, xq_dev, c.rows, c.cols, c.batch)
    plan = xq.last_plan()
    units = -(-plan["groups"] // plan["row_block"])
    assert plan["grid"] == min(units, torch.cuda.get_device_properties(0).multi_processor_count)
    assert plan["row_block"] == (2 if c.batch >= 2 and c.fmt == "q4k" else 1)
    assert y.shape == (c.batch, c.rows)
    y_ref = oracle_rows.matvec(orc, c.fmt, W, kv, xq_ref, c.rows, c.cols, c.batch)
    check_y(y, y_ref, name)
    dots = run_matvec(xq, c.fmt, W, kv, xq_dev, c.rows, c.cols, c.batch, dots=True)
    ref_d = oracle_rows.subdots(orc, c.fmt, W, kv, xq_ref, c.rows, c.cols, c.batch)
    diff = np.argwhere(dots != ref_d)
    assert diff.size == 0, f"{len(diff)} dots differ, first at {diff[:4].tolist()}"


# ---------------------------------------------------------------- degenerate cases
@pytest.mark.parametrize("fmt", ["q4k", "cb4"])
def test_zero_weights_and_zero_activations(xq, orc, fmt):
    rows, cols, batch = 45, 1024, 2
    kv = synthetic.cb4_table()
    W0 = np.zeros_like(_weights(fmt, rows, cols, 1))
    x = synthetic.activations(batch, cols, 2)
    y = run_matvec(xq, fmt, W0, kv, run_quantize(xq, x), rows, cols, batch)
    assert np.all(y == 0.0)
    W = _weights(fmt, rows, cols, 3)
    y = run_matvec(xq, fmt, W, kv, run_quantize(xq, np.zeros((batch, cols), np.float32)), rows,
                   cols, batch)
    assert np.all(y == 0.0)


def test_extreme_codes(xq, orc):
    """All nibbles 15, all six-bit scales/mins 63 and all activations at +-127:
    the largest integer sums the route can form stay exact."""
    rows, cols, batch = 40, 2048, 1
    W = synthetic.q4k_weights(rows, cols, 9)
    W.reshape(rows, -1, 144)[:, :, 4:] = 0xFF
    x = np.full((batch, cols), 127.0, np.float32)
    xq_dev = run_quantize(xq, x)
    xq_ref = orc.quantize_q8(x)
    check_y(run_matvec(xq, "q4k", W, None, xq_dev, rows, cols, batch),
            orc.matvec_q4k(W, xq_ref, rows, cols, batch), "extreme q4k")
    assert np.array_equal(run_matvec(xq, "q4k", W, None, xq_dev, rows, cols, batch, dots=True),
                          orc.subdots_q4k(W, xq_ref, rows, cols, batch))


# ---------------------------------------------------------------- launch plans
@pytest.mark.parametrize("cols", [256, 512, 1024, 2048, 4096, 4352, 14336])
def test_plan_fires(xq, orc, cols):
    """Each shape takes the work-unit shape meant for it: whole rows in one
    box when cols/256 is a power of two below 32, else 32-chunk row segments."""
    rows = 70
    W = synthetic.q4k_weights(rows, cols, 4)
    x = synthetic.activations(1, cols, 5)
    xq_dev = run_quantize(xq, x)
    before = xq.launch_count(xq.COUNT_MATVEC_Q4K)
    y = run_matvec(xq, "q4k", W, None, xq_dev, rows, cols, 1)
    assert xq.launch_count(xq.COUNT_MATVEC_Q4K) == before + 1
    p = xq.last_plan()
    nb = cols // 256
    R = 32 // nb if nb < 32 and 32 % nb == 0 else 1
    assert p["rows_per_group"] == R and p["segments"] == (1 if R > 1 else -(-nb // 32))
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert p["groups"] == -(-rows // R) and p["grid"] == min(p["groups"], sms)
    check_y(y, orc.matvec_q4k(W, orc.quantize_q8(x), rows, cols, 1), f"plan {cols}")


def test_batch_split_when_activations_exceed_shared_memory(xq, orc):
    """cols = 65536 with 8 vectors: the q8 blocks (8 x 256 x 304 bytes) do not
    fit in shared memory, so the call makes several launches of fewer vectors."""
    rows, cols, batch = 37, 65536, 8
    W = synthetic.q4k_weights(rows, cols, 14)
    x = synthetic.activations(batch, cols, 15)
    xq_dev = run_quantize(xq, x)
    before = xq.launch_count(xq.COUNT_MATVEC_Q4K)
    y = run_matvec(xq, "q4k", W, None, xq_dev, rows, cols, batch)
    p = xq.last_plan()
    assert p["launches"] > 1 and xq.launch_count(xq.COUNT_MATVEC_Q4K) == before + p["launches"]
    xq_ref = orc.quantize_q8(x)
    check_y(y, orc.matvec_q4k(W, xq_ref, rows, cols, batch), "batch split")
    dots = run_matvec(xq, "q4k", W, None, xq_dev, rows, cols, batch, dots=True)
    assert np.array_equal(dots, orc.subdots_q4k(W, xq_ref, rows, cols, batch))


@pytest.mark.parametrize("warps,stages", [(1, 2), (2, 3), (3, 5), (8, 2), (8, 6), (4, 8)])
def test_plan_overrides_agree(xq, orc, warps, stages):
    """Every warps/stages split reads the same bytes and forms the same dots;
    y stays within tolerance of the oracle."""
    rows, cols, batch = 200, 4096, 2
    W = synthetic.q4k_weights(rows, cols, 6)
    x = synthetic.activations(batch, cols, 7)
    xq_dev = run_quantize(xq, x)
    xq_ref = orc.quantize_q8(x)
    try:
        xq.set_plan_override(warps, stages)
        xq.set_row_block_override(1)  # one row group per unit: every split fits
        dots = run_matvec(xq, "q4k", W, None, xq_dev, rows, cols, batch, dots=True)
        y = run_matvec(xq, "q4k", W, None, xq_dev, rows, cols, batch)
        p = xq.last_plan()
        assert p["warps"] == warps and p["stages"] == stages
    finally:
        xq.set_plan_override(0, 0)
        xq.set_row_block_override(0)
    assert np.array_equal(dots, orc.subdots_q4k(W, xq_ref, rows, cols, batch))
    check_y(y, orc.matvec_q4k(W, xq_ref, rows, cols, batch), f"override {warps}x{stages}")


def test_plan_override_clamped_to_shared_memory(xq, orc):
    """8 warps x 8 stages do not fit in shared memory: the planner lowers the
    stage count until they do, and the result is still exact."""
    rows, cols, batch = 64, 4096, 2
    W = synthetic.q4k_weights(rows, cols, 8)
    x = synthetic.activations(batch, cols, 9)
    xq_dev = run_quantize(xq, x)
    try:
        xq.set_plan_override(8, 8)
        dots = run_matvec(xq, "q4k", W, None, xq_dev, rows, cols, batch, dots=True)
        p = xq.last_plan()
    finally:
        xq.set_plan_override(0, 0)
    assert p["warps"] == 8 and p["stages"] < 8
    assert p["smem_bytes"] <= torch.cuda.get_device_properties(0).shared_memory_per_block_optin
    assert np.array_equal(dots, orc.subdots_q4k(W, orc.quantize_q8(x), rows, cols, batch))


# ---------------------------------------------------------------- fused quantise + mat-vec
@pytest.mark.parametrize("fmt", ["q4k", "cb4"])
@pytest.mark.parametrize("rows,cols,batch", [(1, 256, 1), (101, 1024, 2), (77, 4096, 8),
                                             (300, 4096, 1), (64, 14336, 3), (37, 65536, 8)])
def test_linear_is_the_two_call_path(xq, orc, fmt, rows, cols, batch):
    """The fused launch quantises x with the quantiser's own arithmetic, so y
    is bit-identical to xq_quantize_q8 followed by the mat-vec, and within
    the tolerance of the oracle."""
    seed = rows + cols + 3 * batch
    W = _weights(fmt, rows, cols, seed)
    kv = synthetic.cb4_table()
    x = synthetic.activations(batch, cols, seed + 1, outlier_frac=0.001)
    y2 = run_matvec(xq, fmt, W, kv, run_quantize(xq, x), rows, cols, batch)
    out = Guarded((batch, rows), torch.float32)
    which = xq.COUNT_LINEAR_Q4K if fmt == "q4k" else xq.COUNT_LINEAR_CB4
    before = xq.launch_count(which)
    if fmt == "q4k":
        xq.linear_q4k(dev(x), dev(W), rows, cols, out=out.t)
    else:
        xq.linear_cb4(dev(x), dev(W), kv, rows, cols, out=out.t)
    torch.cuda.synchronize()
    out.check_guard()
    assert xq.launch_count(which) == before + xq.last_plan()["launches"]
    y1 = out.t.cpu().numpy()
    assert np.array_equal(y1, y2)
    xq_ref = orc.quantize_q8(x)
    y_ref = (orc.matvec_q4k(W, xq_ref, rows, cols, batch) if fmt == "q4k"
             else orc.matvec_cb4(W, kv, xq_ref, rows, cols, batch))
    check_y(y1, y_ref, f"linear {fmt} {rows}x{cols} b{batch}")


@pytest.mark.parametrize("kind", ["zeros", "tiny", "huge", "ties", "subnormal", "nonfinite"])
@pytest.mark.parametrize("fmt", ["q4k", "cb4"])
@pytest.mark.parametrize("rows,cols,batch", [(5, 1024, 2), (37, 4096, 8), (65, 14336, 3),
                                             (16, 65536, 1)])
def test_linear_quantises_edge_inputs_like_the_quantiser(xq, orc, kind, fmt, rows, cols, batch):
    """The fused launch quantises several blocks a warp at once; on inputs
    that reach every branch of the rule (all-zero blocks, an iscale that
    overflows, NaN and inf values) y has the bits of xq_quantize_q8 followed
    by the mat-vec (NaN where both have NaN)."""
    seed = 3 * rows + cols + batch
    W = _weights(fmt, rows, cols, seed)
    kv = synthetic.cb4_table()
    x = _x_kind(kind, batch, cols, seed + 1)
    xq_dev = run_quantize(xq, x)
    assert np.array_equal(xq_dev.cpu().numpy(), orc.quantize_q8(x))
    y2 = run_matvec(xq, fmt, W, kv, xq_dev, rows, cols, batch)
    out = Guarded((batch, rows), torch.float32)
    if fmt == "q4k":
        xq.linear_q4k(dev(x), dev(W), rows, cols, out=out.t)
    else:
        xq.linear_cb4(dev(x), dev(W), kv, rows, cols, out=out.t)
    torch.cuda.synchronize()
    out.check_guard()
    y1 = out.t.cpu().numpy()
    assert np.array_equal(y1, y2, equal_nan=True)


# ---------------------------------------------------------------- RMSNorm + q8 pack
def _norm_x(kind, batch, cols, seed):
    if kind == "order":
        # the hand-derived order cases: one large square among ones (the
        # butterfly and the wave order decide the f32 sum), and a large
        # square last in an item's strided loop
        x = np.ones((batch, cols), np.float32)
        x[:, 0] = 4096.0
        if batch > 1:
            x[1] = 0.0
            x[1, 0] = x[1, 256 % cols] = 1.0
            x[1, 512 % cols] = 4096.0
        return x
    return _x_kind(kind, batch, cols, seed)


@pytest.mark.parametrize("kind", ["normal", "outliers", "fixture", "zeros", "tiny", "huge",
                                  "ties", "order"])
@pytest.mark.parametrize("cols,batch", [(256, 1), (768, 2), (4096, 8), (14336, 2), (65536, 1)])
def test_rmsnorm_q8_bit_exact(xq, orc, kind, cols, batch):
    """The scale is summed in the same fixed order on both sides, so y and
    every byte of the q8 blocks agree bit for bit."""
    x = _norm_x(kind, batch, cols, cols + batch)
    xq_ref, y_ref = orc.rmsnorm_q8(x)
    out = Guarded((batch, cols // 256, 320), torch.uint8)
    y = Guarded((batch, cols), torch.float32)
    before = xq.launch_count(xq.COUNT_RMSNORM_Q8)
    xq.rmsnorm_q8(dev(x), out=out.t, y=y.t)
    torch.cuda.synchronize()
    out.check_guard()
    y.check_guard()
    assert xq.launch_count(xq.COUNT_RMSNORM_Q8) == before + 1
    got_y = y.t.cpu().numpy()
    assert np.array_equal(got_y.view(np.uint32), y_ref.view(np.uint32)), \
        f"y differs at {np.argwhere(got_y.view(np.uint32) != y_ref.view(np.uint32))[:4]}"
    got = out.t.cpu().numpy()
    bad = np.argwhere(got != xq_ref)
    assert bad.size == 0, f"q8 bytes differ at {bad[:4]}"
    # without y: the same q8 bytes
    out2 = Guarded((batch, cols // 256, 320), torch.uint8)
    xq.rmsnorm_q8(dev(x), out=out2.t)
    torch.cuda.synchronize()
    out2.check_guard()
    assert np.array_equal(out2.t.cpu().numpy(), xq_ref)


@pytest.mark.parametrize("fmt", ["q4k", "cb4"])
@pytest.mark.parametrize("rows,cols,batch", [(1, 256, 1), (101, 1024, 2), (77, 4096, 8),
                                             (300, 4096, 1), (64, 14336, 3), (37, 65536, 8),
                                             (4096, 4096, 1)])
def test_norm_linear_is_rmsnorm_then_matvec(xq, orc, fmt, rows, cols, batch):
    """Every CTA of the fused launch computes the RMSNorm scale in the same
    order (whatever its warp count), so y is bit-identical to xq_rmsnorm_q8
    followed by the mat-vec, and within tolerance of the oracle."""
    seed = 7 * rows + cols + batch
    W = _weights(fmt, rows, cols, seed)
    kv = synthetic.cb4_table()
    x = synthetic.activations(batch, cols, seed + 1, outlier_frac=0.001)
    xq2 = Guarded((batch, cols // 256, 320), torch.uint8)
    xq.rmsnorm_q8(dev(x), out=xq2.t)
    y2 = run_matvec(xq, fmt, W, kv, xq2.t, rows, cols, batch)
    out = Guarded((batch, rows), torch.float32)
    which = xq.COUNT_NORM_LINEAR_Q4K if fmt == "q4k" else xq.COUNT_NORM_LINEAR_CB4
    before = xq.launch_count(which)
    if fmt == "q4k":
        xq.norm_linear_q4k(dev(x), dev(W), rows, cols, out=out.t)
    else:
        xq.norm_linear_cb4(dev(x), dev(W), kv, rows, cols, out=out.t)
    torch.cuda.synchronize()
    out.check_guard()
    assert xq.launch_count(which) == before + xq.last_plan()["launches"]
    y1 = out.t.cpu().numpy()
    assert np.array_equal(y1, y2)
    xq_ref, _ = orc.rmsnorm_q8(x)
    y_ref = (orc.matvec_q4k(W, xq_ref, rows, cols, batch) if fmt == "q4k"
             else orc.matvec_cb4(W, kv, xq_ref, rows, cols, batch))
    check_y(y1, y_ref, f"norm linear {fmt} {rows}x{cols} b{batch}")


def test_norm_linear_with_few_and_many_warps(xq, orc):
    """Plans of 1, 3, 7, 8 and 16 warps and 1 to 3 stages: below eight warps
    one warp walks each vector for its scale; from eight up warps 0..7 are
    the workgroup, their partials meeting in warp 0's last stage.  The same
    bits every way."""
    rows, cols = 2048, 4096
    W = _weights("q4k", rows, cols, 91)
    x = synthetic.activations(1, cols, 92)
    xq_ref, _ = orc.rmsnorm_q8(x)
    y_ref = orc.matvec_q4k(W, xq_ref, rows, cols, 1)
    ys = []
    try:
        for w, st in ((1, 0), (3, 0), (7, 0), (8, 0), (8, 1), (16, 0), (16, 1), (16, 3)):
            xq.set_plan_override(w, st)
            y = xq.norm_linear_q4k(dev(x), dev(W), rows, cols)
            torch.cuda.synchronize()
            assert xq.last_plan()["warps"] == w
            assert st == 0 or xq.last_plan()["stages"] == st
            ys.append(y.cpu().numpy())
    finally:
        xq.set_plan_override(0, 0)
    for y in ys:
        assert np.array_equal(y, ys[0])
    check_y(ys[0], y_ref, "norm linear warps")


# ---------------------------------------------------------------- grouped experts
def _slab(fmt, E, rpe, cols, seed):
    return np.concatenate([_weights(fmt, rpe, cols, seed + 17 * e) for e in range(E)])


@pytest.mark.parametrize("fmt", ["q4k", "cb4"])
@pytest.mark.parametrize("rpe,cols", [(64, 2048), (45, 4096), (33, 1024), (20, 14336), (64, 256)])
@pytest.mark.parametrize("x_per_slot", [False, True])
def test_matvec_id_is_per_expert_launches(xq, orc, fmt, rpe, cols, x_per_slot):
    """One grouped launch over a six-expert slab equals, bit for bit, one dense
    launch per selected expert ("25 - Writing XPU Kernels" 25.7.1's gate: ==,
    never a tolerance); and it is within tolerance of the oracle."""
    E, ids = 6, [4, 0, 3]
    used = len(ids)
    slab = _slab(fmt, E, rpe, cols, rpe + cols)
    kv = synthetic.cb4_table()
    nvec = used if x_per_slot else 1
    x = synthetic.activations(nvec, cols, cols + 1)
    xq_dev = run_quantize(xq, x)
    sel = torch.tensor(ids, dtype=torch.int32, device="cuda")
    out = Guarded((used, rpe), torch.float32)
    which = xq.COUNT_MATVEC_ID_Q4K if fmt == "q4k" else xq.COUNT_MATVEC_ID_CB4
    before = xq.launch_count(which)
    xq.matvec_id(fmt, dev(slab), sel, xq_dev, rpe, cols, E, table=kv, x_per_slot=x_per_slot,
                 out=out.t)
    torch.cuda.synchronize()
    out.check_guard()
    assert xq.launch_count(which) == before + 1
    y_id = out.t.cpu().numpy()
    xq_ref = orc.quantize_q8(x)
    for kk, e in enumerate(ids):
        W_e = np.ascontiguousarray(slab[e * rpe:(e + 1) * rpe])
        v = kk if x_per_slot else 0
        y_dense = run_matvec(xq, fmt, W_e, kv, xq_dev[v:v + 1].contiguous(), rpe, cols, 1)
        assert np.array_equal(y_id[kk], y_dense[0]), f"slot {kk}"
        y_ref = (orc.matvec_q4k(W_e, xq_ref[v:v + 1], rpe, cols, 1) if fmt == "q4k"
                 else orc.matvec_cb4(W_e, kv, xq_ref[v:v + 1], rpe, cols, 1))
        check_y(y_id[kk:kk + 1], y_ref, f"id slot {kk}")
    assert not np.isnan(y_id).any()


def test_matvec_id_bad_expert_id_reports_without_trapping(xq, orc):
    """An id outside [0, n_experts) reads nothing: its slot's rows are NaN, the
    other slots are exact, and the device status word says so."""
    E, rpe, cols = 4, 40, 2048
    slab = _slab("q4k", E, rpe, cols, 5)
    x = synthetic.activations(1, cols, 6)
    xq_dev = run_quantize(xq, x)
    xq.device_status(clear=True)
    sel = torch.tensor([1, 99, 2, -3], dtype=torch.int32, device="cuda")
    y = xq.matvec_id("q4k", dev(slab), sel, xq_dev, rpe, cols, E)
    torch.cuda.synchronize()
    y = y.cpu().numpy()
    assert np.isnan(y[1]).all() and np.isnan(y[3]).all()
    for kk, e in ((0, 1), (2, 2)):
        y_dense = run_matvec(xq, "q4k", np.ascontiguousarray(slab[e * rpe:(e + 1) * rpe]), None,
                             xq_dev, rpe, cols, 1)
        assert np.array_equal(y[kk], y_dense[0])
    assert xq.device_status(clear=True) == 2
    assert xq.device_status() == 0


# ---------------------------------------------------------------- streams and graphs
def test_side_stream_and_graph_replay(xq, orc):
    rows, cols, batch = 500, 4096, 1
    W = dev(synthetic.q4k_weights(rows, cols, 12))
    x = synthetic.activations(batch, cols, 13)
    xd = dev(x)
    xq_buf = torch.empty((batch, cols // 256, 320), dtype=torch.uint8, device="cuda")
    y = torch.empty((batch, rows), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        xq.quantize_q8(xd, out=xq_buf)
        xq.matvec_q4k(W, xq_buf, rows, cols, out=y)
    s.synchronize()
    eager = y.cpu().numpy().copy()
    g = torch.cuda.CUDAGraph()
    y.fill_(float("nan"))
    with torch.cuda.graph(g):
        xq.quantize_q8(xd, out=xq_buf)
        xq.matvec_q4k(W, xq_buf, rows, cols, out=y)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy(), eager)
    y_ref = orc.matvec_q4k(W.cpu().numpy(), orc.quantize_q8(x), rows, cols, batch)
    check_y(eager, y_ref, "stream/graph")


def test_device_status_clean(xq):
    assert xq.device_status(clear=False) == 0


# ---------------------------------------------------------------- row blocking
@pytest.mark.parametrize("rows,cols,batch", [(33, 256, 2), (31, 1024, 3), (77, 4096, 8),
                                             (101, 4096, 2), (9, 14336, 4), (64, 14336, 8),
                                             (64, 14336, 4),
                                             (5, 2304, 5), (3, 32768, 2)])
def test_row_block_is_bit_identical(xq, orc, rows, cols, batch):
    """Two row groups per warp unit (the automatic plan for Q4_K at batch >= 2)
    and one give the same dots and the same y bits, fused or not: only which
    warp handles a chunk differs.  Odd group counts leave a half unit."""
    W = synthetic.q4k_weights(rows, cols, 3 * rows + cols)
    x = synthetic.activations(batch, cols, rows + 5, outlier_frac=0.001)
    xq_dev = run_quantize(xq, x)
    Wd, xd = dev(W), dev(x)
    out = {}
    try:
        for rb in (1, 0):
            xq.set_row_block_override(rb)
            dots = run_matvec(xq, "q4k", W, None, xq_dev, rows, cols, batch, dots=True)
            y = run_matvec(xq, "q4k", W, None, xq_dev, rows, cols, batch)
            p = xq.last_plan()
            y_lin = xq.linear_q4k(xd, Wd, rows, cols).cpu().numpy()
            y_nl = xq.norm_linear_q4k(xd, Wd, rows, cols).cpu().numpy()
            out[rb] = (p["row_block"], dots, y, y_lin, y_nl)
    finally:
        xq.set_row_block_override(0)
    props = torch.cuda.get_device_properties(0)
    auto = xq.plan_matvec(rows, cols, batch, sm_count=props.multi_processor_count,
                          smem_optin=props.shared_memory_per_block_optin)["row_block"]
    assert out[1][0] == 1 and out[0][0] == auto
    assert auto == 2
    for a, b in zip(out[1][1:], out[0][1:]):
        assert np.array_equal(a, b)
    xq_ref = orc.quantize_q8(x)
    assert np.array_equal(out[0][1], orc.subdots_q4k(W, xq_ref, rows, cols, batch))
    check_y(out[0][2], orc.matvec_q4k(W, xq_ref, rows, cols, batch), "row block")


# ---------------------------------------------------------------- warp pairs
@pytest.mark.parametrize("rows,batch", [(1, 8), (3, 8), (5, 8), (77, 8), (1000, 8), (4099, 8),
                                        (14338, 8)])
def test_vector_pairs_are_bit_identical(xq, orc, rows, batch):
    """Warp pairs (two warps share each unit and its stages, each computing
    half of the vectors) give the y bits of the one-warp unit, with any pair
    count and stage depth, on the mat-vec and on the decode step; pairs with
    no unit, half units and ragged tails included."""
    cols = 4096
    W = synthetic.q4k_weights(rows, cols, 7 * rows + batch)
    x = synthetic.activations(batch, cols, rows + 11, outlier_frac=0.001)
    xq_dev = run_quantize(xq, x)
    Wd, xd = dev(W), dev(x)
    ws = torch.empty(xq.linear_workspace_bytes(cols, batch), dtype=torch.uint8, device="cuda")
    out = []
    try:
        for vp, warps, stages in ((1, 0, 0), (2, 12, 2), (2, 10, 3), (2, 2, 2), (2, 4, 4)):
            xq.set_vector_pairs_override(vp)
            xq.set_plan_override(warps, stages)
            y = run_matvec(xq, "q4k", W, None, xq_dev, rows, cols, batch)
            p = xq.last_plan()
            assert p["vector_pairs"] == (vp == 2)
            if vp == 2:
                assert (p["warps"], p["stages"]) == (warps, stages)
            y_ws = xq.linear_ws("q4k", xd, Wd, rows, cols, ws).cpu().numpy()
            assert xq.last_plan()["vector_pairs"] == (vp == 2)
            out.append((y, y_ws))
    finally:
        xq.set_vector_pairs_override(0)
        xq.set_plan_override(0, 0)
    for y, y_ws in out:
        assert np.array_equal(y, out[0][0]) and np.array_equal(y_ws, out[0][0])
    check_y(out[0][0], orc.matvec_q4k(W, orc.quantize_q8(x), rows, cols, batch), "warp pairs")


# ---------------------------------------------------------------- tensor cores
@pytest.mark.parametrize("rows,batch,kind", [(1, 8, "random"), (15, 5, "random"), (129, 6, "random"),
                                             (77, 8, "random"), (1000, 7, "random"),
                                             (4099, 8, "random"), (40000, 6, "random"),
                                             (300, 8, "extreme+"), (130, 5, "extreme-"),
                                             (33, 8, "zeros")])
def test_tensor_cores_are_bit_identical(xq, orc, rows, batch, kind):
    """The tensor-core kernel (tcgen05: 128-row tiles, f16 codes in tensor
    memory, the activation by shared-memory descriptor, exact f32 accumulation
    of each sub-block) gives the dp4a kernel's y bits, with two stages or
    more, on the mat-vec and on the decode step: ragged last tiles, CTAs with
    no tile, and the largest sums the route can form (all codes 15, all
    scales and mins 63, activations all +127 or all -127) included."""
    cols = 4096
    W = synthetic.q4k_weights(rows, cols, 5 * rows + batch)
    if kind == "random":
        x = synthetic.activations(batch, cols, rows + 13, outlier_frac=0.001)
    elif kind == "zeros":
        x = np.zeros((batch, cols), np.float32)
    else:
        W.reshape(rows, -1, 144)[:, :, 4:] = 0xFF
        x = np.full((batch, cols), 127.0 if kind == "extreme+" else -127.0, np.float32)
    xq_dev = run_quantize(xq, x)
    Wd, xd = dev(W), dev(x)
    ws = torch.empty(xq.linear_workspace_bytes(cols, batch), dtype=torch.uint8, device="cuda")
    out = []
    try:
        for tc, stages in ((1, 0), (2, 0), (2, 2), (2, 5)):
            xq.set_tensor_override(tc)
            xq.set_plan_override(0, stages)
            y = run_matvec(xq, "q4k", W, None, xq_dev, rows, cols, batch)
            p = xq.last_plan()
            assert p["tensor"] == (tc == 2)
            if tc == 2:
                assert p["warps"] == 17 and p["stages"] == (stages or 3)
            y_ws = xq.linear_ws("q4k", xd, Wd, rows, cols, ws).cpu().numpy()
            assert xq.last_plan()["tensor"] == (tc == 2)
            out.append((y, y_ws))
    finally:
        xq.set_tensor_override(0)
        xq.set_plan_override(0, 0)
    assert xq.device_status(clear=True) == 0
    for y, y_ws in out:
        assert np.array_equal(y, out[0][0]) and np.array_equal(y_ws, out[0][0])
    y_ref = orc.matvec_q4k(W, orc.quantize_q8(x), rows, cols, batch)
    if kind == "zeros":
        assert np.all(out[0][0] == 0.0)
    else:
        check_y(out[0][0], y_ref, "tensor cores")


# ---------------------------------------------------------------- codebook table forms
@pytest.mark.parametrize("fmt", ["cb4", "cb4r"])
@pytest.mark.parametrize("table", ["seeded", "unsplit", "random0", "random1", "extremes"])
def test_codebook_table_forms_agree(xq, orc, fmt, table):
    """One-vector launches decode with the table split into two lookups (when
    it splits) and batched ones with the select decode; both give the exact
    dots, so a vector's y has the same bits either way, for tables that split
    and for one that does not (an entry 127 beside a negative partner)."""
    import ctypes
    rows, cols, batch = 300, 4096, 2
    if table == "seeded":
        kv = synthetic.cb4_table()
    elif table == "unsplit":
        kv = np.array([-1] * 8 + [127] * 8, np.int8)
    elif table == "extremes":
        kv = np.array([-128, 127, -127, 126, 0, -1, 1, 64, -64, 100, -100, 2, -2, 50, -50, 127],
                      np.int8)
    else:
        kv = np.random.default_rng(int(table[-1])).integers(-128, 128, 16).astype(np.int8)
    lib = ctypes.CDLL(xq.lib_path())
    lib.xq_codebook_split_table.restype = ctypes.c_int32
    splits = lib.xq_codebook_split_table(np.ascontiguousarray(kv).ctypes.data_as(ctypes.c_void_p),
                                         (ctypes.c_uint32 * 4)())
    if table in ("seeded", "unsplit"):
        assert splits == (table == "seeded")
    W = synthetic.cb4_weights(rows, cols, 21)
    x = synthetic.activations(batch, cols, 22, outlier_frac=0.001)
    xq_dev = run_quantize(xq, x)
    Wd = dev(W)
    if fmt == "cb4r":
        Wd = xq.repack_cb4(Wd, rows, cols)
    y2 = getattr(xq, "matvec_" + fmt)(Wd, kv, xq_dev, rows, cols).cpu().numpy()
    for b in range(batch):
        y1 = getattr(xq, "matvec_" + fmt)(Wd, kv, xq_dev[b:b + 1].contiguous(), rows, cols)
        assert np.array_equal(y1.cpu().numpy()[0], y2[b]), b
    d1 = xq.subdots_cb4(dev(W), kv, xq_dev[:1].contiguous(), rows, cols).cpu().numpy()
    xq_ref = orc.quantize_q8(x)
    assert np.array_equal(d1, orc.subdots_cb4(W, kv, xq_ref[:1], rows, cols, 1))
    check_y(y2, orc.matvec_cb4(W, kv, xq_ref, rows, cols, batch), f"{fmt} table {table}")


# ---------------------------------------------------------------- the binding's size checks
def test_binding_rejects_short_buffers(xq):
    """The C ABI takes raw pointers and cannot see allocation sizes; the
    binding checks every buffer against the shape before it calls, so a short
    W, y, dots or q8 buffer raises instead of being read or written past its
    end, and nothing is launched."""
    rows, cols, batch = 64, 1024, 2
    W = dev(synthetic.q4k_weights(rows, cols, 1))
    x = dev(synthetic.activations(batch, cols, 2))
    q8 = xq.quantize_q8(x)
    kv = synthetic.cb4_table()
    ws = torch.empty(xq.linear_workspace_bytes(cols, batch), dtype=torch.uint8, device="cuda")
    short_W = W.reshape(-1)[:-16].contiguous()
    short_y = torch.empty((batch, rows - 1), dtype=torch.float32, device="cuda")
    short_d = torch.empty((batch, rows, cols // 32 - 1), dtype=torch.int32, device="cuda")
    counts = [xq.launch_count(i) for i in range(xq.COUNT_N)]
    calls = [
        lambda: xq.matvec_q4k(short_W, q8, rows, cols),
        lambda: xq.matvec_q4k(W, q8, rows, cols, out=short_y),
        lambda: xq.subdots_q4k(W, q8, rows, cols, out=short_d),
        lambda: xq.linear_q4k(x, short_W, rows, cols),
        lambda: xq.linear_ws("q4k", x, W, rows, cols, ws, out=short_y),
        lambda: xq.matvec_cb4(short_W, kv, q8, rows, cols),
        lambda: xq.quantize_q8(x, out=q8.reshape(-1)[:-1]),
        lambda: xq.matvec_id("q4k", W, torch.tensor([0, 1], dtype=torch.int32, device="cuda"),
                             q8, rows // 2, cols, 3),
        lambda: xq.repack_cb4(W, rows, cols, out=short_W),
    ]
    for k, call in enumerate(calls):
        with pytest.raises(ValueError):
            call()
    torch.cuda.synchronize()
    assert [xq.launch_count(i) for i in range(xq.COUNT_N)] == counts


@pytest.mark.parametrize("fmt", ["q4k", "cb4"])
@pytest.mark.parametrize("rows,cols,batch", [(300, 8192, 2), (257, 7936, 3), (64, 16384, 4), (100, 4096, 8)])
def test_batch_vectors_are_independent(xq, orc, fmt, rows, cols, batch):
    """Each vector of a batch gets the bits it gets alone: the staging of the
    q8 blocks (asynchronous copies from 64 Q4_K blocks a launch, grouped
    loads below; the shapes straddle that threshold), the row blocking and
    the reduction never mix vectors."""
    kv = synthetic.cb4_table()
    W = _weights(fmt, rows, cols, 17)
    x = synthetic.activations(batch, cols, 18)
    xq_dev = run_quantize(xq, x)
    y = run_matvec(xq, fmt, W, kv, xq_dev, rows, cols, batch)
    for b in range(batch):
        yb = run_matvec(xq, fmt, W, kv, xq_dev[b:b + 1].contiguous(), rows, cols, 1)
        assert np.array_equal(y[b], yb[0]), f"vector {b}"
    check_y(y, (orc.matvec_q4k if fmt == "q4k" else
                (lambda W_, q, r, c, n: orc.matvec_cb4(W_, kv, q, r, c, n)))(
        W, orc.quantize_q8(x), rows, cols, batch), f"{fmt} batch {batch}")
