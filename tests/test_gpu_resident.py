"""GPU parity of the resident codebook rows ("25 - Writing XPU Kernels" 25.4:
one resident layout, a row's scale prefix padded to a dword then its 16-byte
payloads; 25.2.1 walks it).

  * xq_repack_cb4: every byte of the resident matrix equals the oracle's
    repack, for whole matrices and for chunks that start and end mid-row,
    from 16-byte aligned and unaligned sources; bytes outside a chunk are
    left alone.
  * the resident mat-vec family: exact int32 dots against the oracle's dots
    of the raw matrix (the resident matrix holds the same weights, a pinned
    oracle property), y within 1e-5 rel + 1e-6 abs of the oracle, and
    bit-identical to the raw-layout kernels (only the staging differs).
"""
import numpy as np
import pytest
import torch

import synthetic
from test_gpu_parity import Guarded, check_y, dev, run_quantize

pytestmark = pytest.mark.gpu

SHAPES = [(1, 256, 1), (31, 512, 2), (33, 1024, 4), (101, 2304, 3), (300, 4096, 1),
          (77, 4096, 8), (64, 14336, 2), (9, 65536, 1)]


@pytest.fixture(scope="module")
def xq():
    import quantized_decode_mat_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    return m


def gpu_repack(xq, W, rows, cols, fill=0xEE, chunks=None, src_shift=0):
    """Repack raw W (uint8 numpy) on the GPU, optionally in chunks
    [(base, n), ...], from a source buffer starting src_shift bytes into an
    allocation (0 keeps it 16-byte aligned)."""
    Wf = np.ascontiguousarray(W).reshape(-1)
    nblk = rows * (cols // 32)
    chunks = chunks or [(0, nblk)]
    out = Guarded((xq.cb4r_bytes(rows, cols),), torch.uint8)
    out.t.fill_(fill)
    before = xq.launch_count(xq.COUNT_REPACK_CB4)
    launched = 0
    for base, n in chunks:
        buf = torch.zeros(src_shift + 18 * n + 16, dtype=torch.uint8, device="cuda")
        buf[src_shift:src_shift + 18 * n] = dev(Wf[18 * base:18 * (base + n)])
        xq.repack_cb4(buf, rows, cols, out=out.t, block_base=base, n_blocks=n,
                      src_offset=src_shift)
        launched += 1 if n > 0 else 0
    torch.cuda.synchronize()
    out.check_guard()
    assert xq.launch_count(xq.COUNT_REPACK_CB4) == before + launched
    return out.t.cpu().numpy()


def oracle_repack(orc, W, rows, cols, fill=0xEE, chunks=None):
    Wf = np.ascontiguousarray(W).reshape(-1)
    nblk = rows * (cols // 32)
    dst = np.full(orc.cb4r_row_bytes(cols) * rows, fill, np.uint8)
    for base, n in chunks or [(0, nblk)]:
        if n:
            orc.repack_cb4(Wf[18 * base:18 * (base + n)], dst, base, n, cols)
    return dst


@pytest.mark.parametrize("rows,cols,batch", SHAPES)
@pytest.mark.parametrize("src_shift", [0, 2, 7])
def test_repack_bit_exact(xq, orc, rows, cols, batch, src_shift):
    W = synthetic.cb4_weights(rows, cols, rows + cols)
    got = gpu_repack(xq, W, rows, cols, src_shift=src_shift)
    want = oracle_repack(orc, W, rows, cols)
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} bytes differ, first at {bad[:4].ravel().tolist()}"


@pytest.mark.parametrize("rows,cols", [(3, 256), (5, 1024), (4, 4096), (3, 14336)])
def test_repack_chunks_mid_row(xq, orc, rows, cols):
    """Chunks that start and end inside rows, repacked out of order, one of
    them empty (no launch) and one of a single block: each writes exactly its
    blocks' bytes; together they give the whole repack."""
    bpr = cols // 32
    nblk = rows * bpr
    W = synthetic.cb4_weights(rows, cols, 5 * rows + cols)
    cuts = sorted({1, bpr // 2 + 3, bpr + 5, nblk - 257 if nblk > 300 else nblk // 2,
                   nblk - 1})
    bounds = [0, *[c for c in cuts if 0 < c < nblk], nblk]
    pieces = [(a, b - a) for a, b in zip(bounds[:-1], bounds[1:])]
    order = pieces[::-1] + [(bpr, 0)]
    got = gpu_repack(xq, W, rows, cols, chunks=order, src_shift=4)
    assert np.array_equal(got, oracle_repack(orc, W, rows, cols))
    # one chunk alone leaves every other byte at the fill value
    a, n = pieces[len(pieces) // 2]
    got1 = gpu_repack(xq, W, rows, cols, chunks=[(a, n)])
    assert np.array_equal(got1, oracle_repack(orc, W, rows, cols, chunks=[(a, n)]))


def _resident(orc, W, rows, cols):
    return orc.repack_cb4_whole(np.ascontiguousarray(W).reshape(-1), rows, cols)


@pytest.mark.parametrize("rows,cols,batch", SHAPES)
def test_subdots_cb4r_bit_exact(xq, orc, rows, cols, batch):
    seed = rows * 7 + cols + batch
    W = synthetic.cb4_weights(rows, cols, seed)
    kv = synthetic.cb4_table()
    x = synthetic.activations(batch, cols, seed + 1)
    xq_dev = run_quantize(xq, x)
    out = Guarded((batch, rows, cols // 32), torch.int32)
    before = xq.launch_count(xq.COUNT_SUBDOTS_CB4R)
    xq.subdots_cb4r(dev(_resident(orc, W, rows, cols)), kv, xq_dev, rows, cols, out=out.t)
    torch.cuda.synchronize()
    out.check_guard()
    assert xq.launch_count(xq.COUNT_SUBDOTS_CB4R) == before + 1
    ref = orc.subdots_cb4(W, kv, orc.quantize_q8(x), rows, cols, batch)
    diff = np.argwhere(out.t.cpu().numpy() != ref)
    assert diff.size == 0, f"{len(diff)} dots differ, first at {diff[:4].tolist()}"


@pytest.mark.parametrize("rows,cols,batch", SHAPES)
def test_matvec_cb4r(xq, orc, rows, cols, batch):
    seed = rows * 11 + cols + batch
    W = synthetic.cb4_weights(rows, cols, seed)
    kv = synthetic.cb4_table()
    x = synthetic.activations(batch, cols, seed + 1, outlier_frac=0.001)
    xq_dev = run_quantize(xq, x)
    out = Guarded((batch, rows), torch.float32)
    before = xq.launch_count(xq.COUNT_MATVEC_CB4R)
    xq.matvec_cb4r(dev(_resident(orc, W, rows, cols)), kv, xq_dev, rows, cols, out=out.t)
    torch.cuda.synchronize()
    out.check_guard()
    assert xq.launch_count(xq.COUNT_MATVEC_CB4R) == before + xq.last_plan()["launches"]
    y = out.t.cpu().numpy()
    check_y(y, orc.matvec_cb4(W, kv, orc.quantize_q8(x), rows, cols, batch),
            f"cb4r {rows}x{cols} b{batch}")
    y_raw = xq.matvec_cb4(dev(W), kv, xq_dev, rows, cols)
    torch.cuda.synchronize()
    assert np.array_equal(y, y_raw.cpu().numpy())


@pytest.mark.parametrize("rows,cols,batch", [(1, 256, 1), (101, 1024, 2), (77, 4096, 8),
                                             (300, 4096, 1), (64, 14336, 3)])
def test_fused_cb4r_are_the_two_call_paths(xq, orc, rows, cols, batch):
    """linear_cb4r = quantise then matvec_cb4r and norm_linear_cb4r =
    rmsnorm_q8 then matvec_cb4r, bit for bit."""
    seed = rows + cols + 3 * batch
    W = synthetic.cb4_weights(rows, cols, seed)
    Wr = dev(_resident(orc, W, rows, cols))
    kv = synthetic.cb4_table()
    x = synthetic.activations(batch, cols, seed + 1, outlier_frac=0.001)
    xd = dev(x)
    y2 = xq.matvec_cb4r(Wr, kv, run_quantize(xq, x), rows, cols)
    before = xq.launch_count(xq.COUNT_LINEAR_CB4R)
    y1 = xq.linear_cb4r(xd, Wr, kv, rows, cols)
    torch.cuda.synchronize()
    assert xq.launch_count(xq.COUNT_LINEAR_CB4R) == before + xq.last_plan()["launches"]
    assert torch.equal(y1, y2)
    check_y(y1.cpu().numpy(), orc.matvec_cb4(W, kv, orc.quantize_q8(x), rows, cols, batch),
            "linear cb4r")
    xn = xq.rmsnorm_q8(xd)
    y4 = xq.matvec_cb4r(Wr, kv, xn, rows, cols)
    before = xq.launch_count(xq.COUNT_NORM_LINEAR_CB4R)
    y3 = xq.norm_linear_cb4r(xd, Wr, kv, rows, cols)
    torch.cuda.synchronize()
    assert xq.launch_count(xq.COUNT_NORM_LINEAR_CB4R) == before + xq.last_plan()["launches"]
    assert torch.equal(y3, y4)
    xn_ref, _ = orc.rmsnorm_q8(x)
    check_y(y3.cpu().numpy(), orc.matvec_cb4(W, kv, xn_ref, rows, cols, batch),
            "norm linear cb4r")


@pytest.mark.parametrize("rpe,cols", [(64, 2048), (45, 4096), (20, 14336)])
@pytest.mark.parametrize("x_per_slot", [False, True])
def test_matvec_cb4r_id(xq, orc, rpe, cols, x_per_slot):
    """The grouped launch over a resident slab equals one dense resident
    launch per selected expert, bit for bit."""
    E, ids = 5, [2, 4, 0]
    used = len(ids)
    kv = synthetic.cb4_table()
    raws = [synthetic.cb4_weights(rpe, cols, rpe + cols + 17 * e) for e in range(E)]
    slab_r = np.concatenate([_resident(orc, w, rpe, cols) for w in raws])
    nvec = used if x_per_slot else 1
    x = synthetic.activations(nvec, cols, cols + 3)
    xq_dev = run_quantize(xq, x)
    sel = torch.tensor(ids, dtype=torch.int32, device="cuda")
    before = xq.launch_count(xq.COUNT_MATVEC_ID_CB4R)
    y_id = xq.matvec_id("cb4r", dev(slab_r), sel, xq_dev, rpe, cols, E, table=kv,
                        x_per_slot=x_per_slot)
    torch.cuda.synchronize()
    assert xq.launch_count(xq.COUNT_MATVEC_ID_CB4R) == before + 1
    y_id = y_id.cpu().numpy()
    xq_ref = orc.quantize_q8(x)
    for kk, e in enumerate(ids):
        v = kk if x_per_slot else 0
        y_dense = xq.matvec_cb4r(dev(_resident(orc, raws[e], rpe, cols)), kv,
                                 xq_dev[v:v + 1].contiguous(), rpe, cols)
        torch.cuda.synchronize()
        assert np.array_equal(y_id[kk], y_dense.cpu().numpy()[0]), f"slot {kk}"
        check_y(y_id[kk:kk + 1], orc.matvec_cb4(raws[e], kv, xq_ref[v:v + 1], rpe, cols, 1),
                f"id cb4r slot {kk}")


@pytest.mark.parametrize("name", ["c4_cb4_4096x4096_b1", "c4_cb4_11008x4096_b1"])
def test_config4_resident_end_to_end(xq, orc, name):
    """The codebook configurations at full size: raw blocks repacked on the
    GPU in four chunks, then every output of the resident mat-vec against the
    oracle, and bit-identical to the raw-layout kernel."""
    c = synthetic.CASES[name]
    W, x = c.weights(), c.x()
    kv = synthetic.cb4_table()
    nblk = c.rows * (c.cols // 32)
    q = nblk // 4 + 5
    chunks = [(0, q), (q, q), (2 * q, q), (3 * q, nblk - 3 * q)]
    Wr = gpu_repack(xq, W, c.rows, c.cols, chunks=chunks)
    assert np.array_equal(Wr, oracle_repack(orc, W, c.rows, c.cols))
    xq_dev = run_quantize(xq, x)
    y = xq.matvec_cb4r(dev(Wr), kv, xq_dev, c.rows, c.cols)
    y_raw = xq.matvec_cb4(dev(W), kv, xq_dev, c.rows, c.cols)
    torch.cuda.synchronize()
    assert torch.equal(y, y_raw)
    check_y(y.cpu().numpy(), orc.matvec_cb4(W, kv, orc.quantize_q8(x), c.rows, c.cols, 1), name)
