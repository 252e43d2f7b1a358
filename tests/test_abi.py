"""The C ABI without a GPU: the library builds and loads, exports every symbol
include/xq.h declares, and its host-side argument checks, size functions and
launch planner behave as documented.  Argument checks run before any CUDA
call, so fake (never dereferenced) pointers are enough here."""
import ctypes
import os
import re

import numpy as np
import pytest

import synthetic

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "xq.h")

P = 0x10000  # a 16-byte aligned fake device address (never dereferenced)


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__

    __graft_entry__._xq_build_module().build()
    import quantized_decode_mat_gb300 as xq
    return xq


@pytest.fixture(scope="module")
def raw(lib):
    return ctypes.CDLL(lib.lib_path())


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(xq_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("xq_quantize_q8", "xq_matvec_q4k", "xq_matvec_cb4", "xq_linear_q4k",
                 "xq_linear_cb4", "xq_rmsnorm_q8", "xq_norm_linear_q4k",
                 "xq_norm_linear_cb4", "xq_subdots_q4k",
                 "xq_subdots_cb4", "xq_q8_bytes", "xq_status_string", "xq_last_error"):
        assert must in names


def test_every_declared_symbol_is_exported(raw):
    missing = [n for n in declared_functions() if not hasattr(raw, n)]
    assert not missing, missing


def test_sizes_match_the_formats(lib):
    import oracle
    assert lib.q8_bytes(256, 1) == oracle.Q8_BYTES == 320
    assert lib.q8_bytes(4096, 8) == 8 * 16 * 320
    assert lib.q4k_bytes(1, 256) == oracle.Q4K_BYTES == 144
    assert lib.cb4_bytes(1, 256) == 8 * oracle.CB4_BYTES
    assert lib.q4k_bytes(128256, 4096) == 295_501_824
    assert lib.cb4_bytes(11008, 4096) == 25_362_432
    assert lib.q8_bytes(100, 1) == 0 and lib.q4k_bytes(4, 0) == 0


def _call(raw, name, *args):
    fn = getattr(raw, name)
    fn.restype = ctypes.c_int
    return fn(*args)


I64 = ctypes.c_int64
V = ctypes.c_void_p


@pytest.mark.parametrize("args,status", [
    ((V(0), V(P), V(P), I64(32), I64(256), I64(1), V(0)), 1),         # null W
    ((V(P), V(P), V(0), I64(32), I64(256), I64(1), V(0)), 1),         # null y
    ((V(P), V(P), V(P * 8), I64(32), I64(100), I64(1), V(0)), 3),     # cols % 256
    ((V(P), V(P), V(P * 8), I64(32), I64(0), I64(1), V(0)), 3),       # cols 0
    ((V(P), V(P), V(P * 8), I64(0), I64(256), I64(1), V(0)), 3),      # rows 0
    ((V(P), V(P), V(P * 8), I64(32), I64(256), I64(0), V(0)), 3),     # batch 0
    ((V(P), V(P), V(P * 8), I64(32), I64(256), I64(9), V(0)), 3),     # batch 9
    ((V(P + 8), V(P), V(P * 8), I64(32), I64(256), I64(1), V(0)), 2),  # W misaligned
    ((V(P), V(P + 4), V(P * 8), I64(32), I64(256), I64(1), V(0)), 2),  # xq misaligned
    ((V(P), V(P * 4), V(P + 2), I64(32), I64(256), I64(1), V(0)), 2),  # y misaligned
    ((V(P), V(P * 4), V(P + 16), I64(32), I64(256), I64(1), V(0)), 1),  # y overlaps W
])
def test_matvec_q4k_argument_checks(raw, args, status):
    assert _call(raw, "xq_matvec_q4k", *args) == status
    err = ctypes.CDLL(raw._name).xq_last_error
    err.restype = ctypes.c_char_p
    assert err()


def test_linear_argument_checks(raw):
    assert _call(raw, "xq_linear_q4k", V(0), V(P), V(P * 8), I64(32), I64(256), I64(1), V(0)) == 1
    assert _call(raw, "xq_linear_q4k", V(P + 4), V(P * 4), V(P * 8), I64(32), I64(256), I64(1),
                 V(0)) == 2
    assert _call(raw, "xq_linear_q4k", V(P), V(P * 4), V(P * 8), I64(32), I64(300), I64(1),
                 V(0)) == 3
    # y overlapping x (1 x 256 f32 = 1024 bytes from P)
    assert _call(raw, "xq_linear_q4k", V(P), V(P * 4), V(P + 512), I64(32), I64(256), I64(1),
                 V(0)) == 1
    assert _call(raw, "xq_linear_cb4", V(P), V(P * 4), V(0), V(P * 8), I64(32), I64(256),
                 I64(1), V(0)) == 1


def test_matvec_id_argument_checks(raw):
    fn = "xq_matvec_q4k_id"
    I32 = ctypes.c_int32
    # W, sel, xq, y, rows_per_expert, cols, n_experts, used, x_per_slot, stream
    ok = (V(P), V(P * 2), V(P * 3), V(P * 8), I64(16), I64(256), I64(4), I64(2), I32(0), V(0))
    assert _call(raw, fn, V(P), V(0), *ok[2:]) == 1                         # null sel
    assert _call(raw, fn, V(P), V(P * 2 + 2), *ok[2:]) == 2                 # sel misaligned
    assert _call(raw, fn, *ok[:6], I64(0), *ok[7:]) == 3                    # no experts
    assert _call(raw, fn, *ok[:7], I64(9), I32(1), V(0)) == 3               # 9 per-slot vectors
    assert _call(raw, fn, *ok[:7], I64(0), *ok[8:]) == 3                    # used 0
    assert _call(raw, "xq_matvec_cb4_id", V(P), V(0), *ok[1:]) == 1         # null table


def test_cb4_needs_a_table(raw):
    assert _call(raw, "xq_matvec_cb4", V(P), V(0), V(P * 2), V(P * 8), I64(32), I64(256),
                 I64(1), V(0)) == 1


def test_quantize_argument_checks(raw):
    assert _call(raw, "xq_quantize_q8", V(0), V(P), I64(256), I64(1), V(0)) == 1
    assert _call(raw, "xq_quantize_q8", V(P + 4), V(P * 4), I64(256), I64(1), V(0)) == 2
    assert _call(raw, "xq_quantize_q8", V(P), V(P * 4), I64(300), I64(1), V(0)) == 3
    assert _call(raw, "xq_quantize_q8", V(P), V(P + 512), I64(256), I64(1), V(0)) == 1


def test_rmsnorm_argument_checks(raw):
    assert _call(raw, "xq_rmsnorm_q8", V(0), V(P), V(0), I64(256), I64(1), V(0)) == 1
    assert _call(raw, "xq_rmsnorm_q8", V(P + 4), V(P * 4), V(0), I64(256), I64(1), V(0)) == 2
    assert _call(raw, "xq_rmsnorm_q8", V(P), V(P * 4), V(P * 8 + 4), I64(256), I64(1), V(0)) == 2
    assert _call(raw, "xq_rmsnorm_q8", V(P), V(P * 4), V(0), I64(300), I64(1), V(0)) == 3
    assert _call(raw, "xq_rmsnorm_q8", V(P), V(P * 4), V(0), I64(256), I64(9), V(0)) == 3
    assert _call(raw, "xq_rmsnorm_q8", V(P), V(P + 512), V(0), I64(256), I64(1), V(0)) == 1
    assert _call(raw, "xq_rmsnorm_q8", V(P), V(P * 4), V(P + 512), I64(256), I64(1), V(0)) == 1
    assert _call(raw, "xq_norm_linear_q4k", V(0), V(P), V(P * 8), I64(32), I64(256), I64(1),
                 V(0)) == 1
    assert _call(raw, "xq_norm_linear_cb4", V(P), V(P * 4), V(0), V(P * 8), I64(32), I64(256),
                 I64(1), V(0)) == 1


def test_subdots_need_16_byte_aligned_output(raw):
    assert _call(raw, "xq_subdots_q4k", V(P), V(P * 2), V(P * 8 + 4), I64(32), I64(256),
                 I64(1), V(0)) == 2


def test_status_strings(raw):
    fn = raw.xq_status_string
    fn.restype = ctypes.c_char_p
    for s in range(6):
        assert fn(s).startswith(b"XQ_")
    assert raw.xq_version() == 3


@pytest.mark.parametrize("fmt,rows,cols,batch,warps,grid,R,spr,launches,M", [
    ("q4k", 128256, 4096, 1, 16, 152, 2, 1, 1, 1), ("q4k", 128256, 4096, 8, 16, 152, 2, 1, 1, 2),
    ("q4k", 4096, 4096, 1, 14, 152, 2, 1, 1, 1), ("q4k", 14336, 4096, 4, 8, 152, 2, 1, 1, 2),
    ("q4k", 4096, 14336, 1, 20, 152, 1, 2, 1, 1), ("q4k", 4096, 14336, 8, 8, 152, 1, 2, 1, 2),
    ("q4k", 4096, 14336, 4, 8, 152, 1, 2, 1, 2), ("q4k", 14336, 4096, 2, 12, 152, 2, 1, 1, 2),
    ("q4k", 4096, 14336, 2, 8, 152, 1, 2, 1, 2),
    ("q4k", 256, 1024, 1, 1, 32, 8, 1, 1, 1), ("cb4", 11008, 4096, 1, 20, 152, 2, 1, 1, 1),
    ("cb4", 4096, 4096, 1, 14, 152, 2, 1, 1, 1), ("q4k", 33, 256, 2, 1, 1, 32, 1, 1, 2),
    ("q4k", 1, 512, 1, 1, 1, 16, 1, 1, 1), ("q4k", 100, 2304, 1, 1, 100, 1, 1, 1, 1),
    ("q4k", 1000, 65536, 8, 6, 152, 1, 8, 4, 1), ("cb4", 14336, 4096, 8, 8, 152, 2, 1, 1, 1), ("cb4", 11008, 4096, 4, 16, 152, 2, 1, 1, 1),
    ("cb4r", 300, 2304, 2, 2, 152, 1, 1, 1, 1)])
def test_plan(lib, fmt, rows, cols, batch, warps, grid, R, spr, launches, M):
    p = lib.plan_matvec(rows, cols, batch, fmt=fmt, sm_count=152, smem_optin=232448)
    assert (p["warps"], p["grid"], p["rows_per_group"], p["segments"], p["launches"],
            p["row_block"]) == (warps, grid, R, spr, launches, M), p
    nb = cols // 256
    assert p["chunks_per_row"] == nb
    assert p["groups"] == -(-rows // R)
    assert p["grid"] == min(-(-p["groups"] // M), 152)
    # a work unit is whole rows in one 4608-byte box, or one row in 32-chunk boxes
    assert (R > 1 and R * nb == 32 and spr == 1) or (R == 1 and spr == -(-nb // 32))
    act = -(-p["batch_per_launch"] * nb * 336 // 128) * 128
    if p["vector_pairs"]:
        # warp pairs: 16 warps, two stages a pair, a 2304-byte reduction
        # scratch a warp
        assert fmt == "q4k" and M == 2 and nb == 16 and batch == 8
        assert p["warps"] == 16 and p["stages"] == 2
        assert p["smem_bytes"] == act + 8 * 2 * M * 4608 + 16 * 2304 + 128
    else:
        # two stages, or one where two-box stages for every warp do not fit
        two = act + p["warps"] * 2 * M * 4608 + 128
        assert p["stages"] == (2 if two <= 232448 or M == 1 else 1)
        assert p["smem_bytes"] == act + p["warps"] * p["stages"] * M * 4608 + 128
    assert p["smem_bytes"] <= 232448
    assert p["batch_per_launch"] * (p["launches"] - 1) < batch <= p["batch_per_launch"] * p["launches"]


def test_row_block_override(lib):
    try:
        lib.set_row_block_override(1)
        p = lib.plan_matvec(128256, 4096, 8)
        assert p["row_block"] == 1 and p["warps"] == 8 and p["grid"] == 152
        lib.set_row_block_override(2)
        assert lib.plan_matvec(128256, 4096, 1)["row_block"] == 1  # batch 1 has one
        assert lib.plan_matvec(4096, 4096, 2, fmt="cb4")["row_block"] == 1
    finally:
        lib.set_row_block_override(0)
    assert lib.plan_matvec(128256, 4096, 8)["row_block"] == 2


def test_vector_pairs_plan(lib):
    """Warp pairs only for the Q4_K mat-vec on q8 blocks with rows of 16
    chunks at 8 vectors; the override turns them off or on."""
    assert lib.plan_matvec(128256, 4096, 8)["vector_pairs"] == 1
    assert lib.plan_matvec(128256, 4096, 6)["vector_pairs"] == 0
    # at least 16 units (four rows each) for each of the 152 x 8 pairs
    assert lib.plan_matvec(4 * 16 * 152 * 8, 4096, 8)["vector_pairs"] == 1
    assert lib.plan_matvec(4 * 16 * 152 * 8 - 4, 4096, 8)["vector_pairs"] == 0
    for rows, cols, batch, fmt in ((14336, 4096, 4, "q4k"), (128256, 4096, 1, "q4k"),
                                   (14336, 4096, 8, "q4k"), (14336, 4096, 6, "q4k"),
                                   (4096, 14336, 8, "q4k"), (11008, 4096, 8, "cb4"),
                                   (1000, 2048, 8, "q4k"), (14336, 4096, 7, "q4k")):
        assert lib.plan_matvec(rows, cols, batch, fmt=fmt)["vector_pairs"] == 0
    try:
        lib.set_vector_pairs_override(1)
        p = lib.plan_matvec(128256, 4096, 8)
        assert p["vector_pairs"] == 0 and p["warps"] == 8
        lib.set_vector_pairs_override(2)  # forced: any size
        p = lib.plan_matvec(100, 4096, 8)
        assert p["vector_pairs"] == 1 and (p["warps"], p["stages"]) == (16, 2)
        assert lib.plan_matvec(100, 4096, 6)["vector_pairs"] == 0
        lib.set_plan_override(warps=11, stages=3)  # forced: the overrides size the pairs
        p = lib.plan_matvec(14336, 4096, 8)
        act = 8 * 16 * 336
        assert p["vector_pairs"] == 1 and (p["warps"], p["stages"]) == (10, 3)
        assert p["smem_bytes"] == act + 5 * 3 * 2 * 4608 + 10 * 2304 + 128
        lib.set_plan_override(warps=16, stages=3)  # does not fit: no pairs
        assert lib.plan_matvec(14336, 4096, 8)["vector_pairs"] == 0
        lib.set_vector_pairs_override(0)
        lib.set_plan_override(warps=8, stages=2)  # a warp or stage override turns them off
        assert lib.plan_matvec(128256, 4096, 8)["vector_pairs"] == 0
    finally:
        lib.set_vector_pairs_override(0)
        lib.set_plan_override(0, 0)


def _prmt_lookup(words, sel_nibble):
    """One byte of a byte permute in its generic mode: the nibble's low three
    bits pick a byte of the two words, bit 3 replicates that byte's sign."""
    b = ((words[0] | (words[1] << 32)) >> (8 * (sel_nibble & 7))) & 0xFF
    v = b - 256 if b >= 128 else b
    return (-1 if v < 0 else 0) if sel_nibble & 8 else v


def _split_exists(a, b):
    """Brute force: some signed bytes l, h with a = l + rep(h), b = rep(l) + h."""
    for l in range(-128, 128):
        for sh in (0, -1):
            h = b - (-1 if l < 0 else 0)
            if -128 <= h <= 127 and (-1 if h < 0 else 0) == sh and l + sh == a:
                return True
    return False


def test_codebook_split_table(raw):
    """The one-vector codebook decode's table split: the two lookups of every
    nibble (n in one table, n ^ 8 in the other) sum to the table entry, for
    the seeded table, random tables and edge tables; no split is reported
    exactly when none exists."""
    fn = raw.xq_codebook_split_table
    fn.restype = ctypes.c_int32
    rng = np.random.default_rng(5)
    tables = [synthetic.cb4_table(), np.arange(-8, 8, dtype=np.int8),
              np.full(16, -128, np.int8), np.full(16, 127, np.int8), np.zeros(16, np.int8),
              np.array([-127] * 8 + [127] * 8, np.int8), np.array([127] * 8 + [-1] * 8, np.int8),
              np.array([-1] * 8 + [-1] * 8, np.int8), np.array([0] * 8 + [-128] * 8, np.int8)]
    tables += [rng.integers(-128, 128, 16).astype(np.int8) for _ in range(300)]
    splits = 0
    for t in tables:
        t = np.ascontiguousarray(t, np.int8)
        out = (ctypes.c_uint32 * 4)()
        ok = fn(t.ctypes.data_as(ctypes.c_void_p), out)
        exists = all(_split_exists(int(t[i]), int(t[i + 8])) for i in range(8))
        assert bool(ok) == exists, t
        if ok:
            splits += 1
            L, H = (out[0], out[1]), (out[2], out[3])
            for n in range(16):
                assert _prmt_lookup(L, n) + _prmt_lookup(H, n ^ 8) == t[n], (t, n)
    assert splits > 250
    ok = fn(np.ascontiguousarray(synthetic.cb4_table()).ctypes.data_as(ctypes.c_void_p),
            (ctypes.c_uint32 * 4)())
    assert ok == 1  # the seeded workload's table takes the split decode


def test_tensor_plan(lib):
    """The tensor-core plan: forced on, for the Q4_K mat-vec on q8 blocks with
    rows of 16 chunks at 5..8 vectors only; one CTA of seventeen warps an SM
    on 128-row tiles, three stages unless a stage override sizes it."""
    act = 16 * 16 * 256 + 16 * 8 * 4 + 16 * 8 * 16
    try:
        lib.set_tensor_override(2)
        p = lib.plan_matvec(128256, 4096, 8)
        assert p["tensor"] == 1 and (p["warps"], p["stages"], p["grid"]) == (17, 3, 152)
        assert (p["groups"], p["rows_per_group"], p["segments"], p["row_block"]) == (1002, 128, 16, 1)
        assert p["smem_bytes"] == act + 3 * 128 * 144 + 64 + 1024
        assert lib.plan_matvec(300, 4096, 5)["grid"] == 3
        for rows, cols, batch, fmt in ((14336, 4096, 4, "q4k"), (4096, 14336, 8, "q4k"),
                                       (11008, 4096, 8, "cb4"), (128256, 4096, 1, "q4k")):
            assert lib.plan_matvec(rows, cols, batch, fmt=fmt)["tensor"] == 0
        lib.set_plan_override(stages=5)
        p = lib.plan_matvec(14336, 4096, 6)
        assert p["tensor"] == 1 and (p["warps"], p["stages"]) == (17, 5)
        assert p["smem_bytes"] == act + 5 * 128 * 144 + 64 + 1024
        lib.set_plan_override(stages=1)  # below two: the default three
        assert lib.plan_matvec(14336, 4096, 6)["stages"] == 3
        lib.set_tensor_override(1)
        lib.set_plan_override(0, 0)
        assert lib.plan_matvec(128256, 4096, 8)["tensor"] == 0
    finally:
        lib.set_tensor_override(0)
        lib.set_plan_override(0, 0)


def test_plan_override_is_clamped(lib):
    try:
        lib.set_plan_override(warps=32, stages=64)
        p = lib.plan_matvec(1000, 1024, 1)
        assert p["warps"] == 20 and p["stages"] <= 8 and p["smem_bytes"] <= 232448
        p = lib.plan_matvec(1000, 1024, 2)
        assert p["warps"] == 12
        p = lib.plan_matvec(1000, 1024, 3)
        assert p["warps"] == 8
        lib.set_plan_override(warps=2, stages=3)
        p = lib.plan_matvec(1000, 4096, 1)
        assert p["warps"] == 2 and p["stages"] == 3
    finally:
        lib.set_plan_override(0, 0)


def test_python_binding_rejects_host_tensors(lib):
    import torch
    with pytest.raises(TypeError):
        lib.quantize_q8(torch.zeros(1, 256))


def test_no_kernel_spills(lib):
    """Spill is invisible to timing ("25 - Writing XPU Kernels" 25.5, the
    manifest before the wall clock): no kernel of the library spills or keeps
    a per-thread array in local memory (a stack frame) -- every
    mat-vec build (each format, batch 1..8, with or without the dots, every
    fused form, the grouped form, one or two row groups a unit, the
    whole-row builds) and the quantise, RMSNorm and repack kernels."""
    import __graft_entry__
    rep = __graft_entry__._xq_build_module().ptxas_report()
    assert rep, "no ptxas report"
    matvec = [n for n in rep if "xq_matvec_kernel" in n]
    # format x batch x (dots, fused quantise, fused RMSNorm, plain) + the grouped
    # form (3 formats, batch 1) + the Q4_K row-blocked builds (7 batches x 4
    # kinds x 2 box shapes) + the whole-row batch-1 codebook builds (2 formats x
    # plain, fused quantise, fused RMSNorm) + the warp-pair build (batch 8) +
    # the split-table batch-1 codebook builds (2 formats x (plain, dots, fused
    # quantise, fused RMSNorm, grouped, and the 3 whole-row forms))
    assert len(matvec) == 3 * 8 * 4 + 3 + 7 * 4 * 2 + 2 * 3 + 1 + 2 * 8, len(matvec)
    assert len([n for n in rep if "xq_tc_q4k_kernel" in n]) == 4  # tensor cores, batch 5..8
    for helper in ("q8_quantize_kernel", "rmsnorm_q8_kernel", "repack_cb4_kernel"):
        assert any(helper in n for n in rep), helper
    for name, r in rep.items():
        assert r["registers"] > 0, (name, r)
        assert r["spill_stores"] == 0 and r["spill_loads"] == 0, (name, r)
        assert r["stack_frame"] == 0, (name, r)  # no per-thread array in local memory


def test_oracle_and_product_share_no_code():
    """The oracle and the CUDA path are independent: neither includes or
    imports the other."""
    pkg = os.path.join(ROOT, "quantized_decode_mat_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f
                assert "xq_oracle" not in text, f
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith((".py", ".c", ".h")):
            text = open(os.path.join(ROOT, "oracle", f)).read()
            assert not re.search(r"^\s*(import|from)\s+quantized_decode_mat_gb300\b", text,
                                 re.M), f
            assert "xq_internal" not in text and '#include "xq' not in text, f


def test_repack_argument_checks(raw):
    fn = "xq_repack_cb4"
    # src, Wr, block_base, n_blocks, rows, cols, stream; the 4 x 256 matrix has 32 blocks
    ok = dict(src=P * 64, wr=P, base=0, n=32, rows=4, cols=256)

    def call(**kw):
        a = {**ok, **kw}
        return _call(raw, fn, V(a["src"]), V(a["wr"]), I64(a["base"]), I64(a["n"]),
                     I64(a["rows"]), I64(a["cols"]), V(0))
    assert call(src=0) == 1                       # null src
    assert call(wr=0) == 1                        # null Wr
    assert call(wr=P + 4) == 2                    # Wr misaligned
    assert call(cols=300) == 3                    # cols % 256
    assert call(base=-1) == 3                     # chunk before the matrix
    assert call(base=1, n=32) == 3                # chunk past the end
    assert call(n=-1) == 3
    assert call(src=P + 100) == 1                 # src inside Wr
    # an empty chunk is accepted and launches nothing (no GPU is touched)
    before = raw.xq_launch_count(12)
    assert call(n=0) == 0
    assert raw.xq_launch_count(12) == before


def test_resident_entry_points_check_arguments(raw):
    assert _call(raw, "xq_matvec_cb4r", V(P), V(0), V(P * 2), V(P * 8), I64(32), I64(256),
                 I64(1), V(0)) == 1
    tbl = (ctypes.c_int8 * 16)()
    assert _call(raw, "xq_matvec_cb4r", V(P + 8), tbl, V(P * 2), V(P * 8), I64(32), I64(256),
                 I64(1), V(0)) == 2
    assert _call(raw, "xq_linear_cb4r", V(P), V(P * 4), tbl, V(P * 8), I64(32), I64(300),
                 I64(1), V(0)) == 3
    assert _call(raw, "xq_norm_linear_cb4r", V(0), V(P * 4), tbl, V(P * 8), I64(32), I64(256),
                 I64(1), V(0)) == 1
    assert _call(raw, "xq_subdots_cb4r", V(P), tbl, V(P * 2), V(P * 8 + 4), I64(32), I64(256),
                 I64(1), V(0)) == 2


def test_resident_sizes(lib):
    import oracle
    o = oracle.get()
    for rows, cols in ((1, 256), (7, 4096), (11008, 4096), (3, 14336)):
        assert lib.cb4r_bytes(rows, cols) == rows * o.cb4r_row_bytes(cols) == \
            lib.cb4_bytes(rows, cols)
    # the same boxes, units and plan (20 warps at batch 1 for both layouts)
    p = lib.plan_matvec(11008, 4096, 1, fmt="cb4r")
    assert p["warps"] == 20
    assert p == lib.plan_matvec(11008, 4096, 1, fmt="cb4")


def test_linear_ws_argument_checks(raw, lib):
    SZ = ctypes.c_size_t
    need = lib.linear_workspace_bytes(256, 1)
    assert need == 320 and lib.linear_workspace_bytes(4096, 8) == 40960 == lib.q8_bytes(4096, 8)
    assert lib.linear_workspace_bytes(300, 1) == 0 and lib.linear_workspace_bytes(256, 9) == 0
    args = lambda ws, n: (V(P), V(P * 4), V(P * 8), I64(32), I64(256), I64(1), V(ws), SZ(n), V(0))
    assert _call(raw, "xq_linear_q4k_ws", *args(0, need)) == 1            # null workspace
    assert _call(raw, "xq_linear_q4k_ws", *args(P * 16, need - 1)) == 1   # too small
    assert _call(raw, "xq_linear_q4k_ws", *args(P * 16 + 8, need)) == 2   # misaligned
    assert _call(raw, "xq_linear_q4k_ws", *args(P * 8, need)) == 1        # overlaps y
    tbl = (ctypes.c_int8 * 16)()
    assert _call(raw, "xq_linear_cb4_ws", V(P), V(P * 4), V(0), V(P * 8), I64(32), I64(256),
                 I64(1), V(P * 16), SZ(need), V(0)) == 1                   # null table
    assert _call(raw, "xq_linear_cb4r_ws", V(P), V(P * 4), tbl, V(P * 8), I64(32), I64(300),
                 I64(1), V(P * 16), SZ(need), V(0)) == 3                   # cols % 256


def test_plan_reports_the_workspace_choice(lib):
    assert lib.plan_matvec(128256, 4096, 1)["quantise_once"] == 0   # 16 blocks: per CTA
    assert lib.plan_matvec(4096, 14336, 1)["quantise_once"] == 1    # 56 blocks: once
    assert lib.plan_matvec(14336, 4096, 2)["quantise_once"] == 0    # 32 blocks: per CTA
    assert lib.plan_matvec(14336, 4096, 3)["quantise_once"] == 1    # 48 blocks: once
    assert lib.plan_matvec(4096, 8448, 1)["quantise_once"] == 1     # 33 blocks: once
    assert lib.plan_matvec(4096, 7936, 1)["quantise_once"] == 0     # 31 blocks: per CTA
    assert lib.plan_matvec(14336, 4096, 8)["quantise_once"] == 1    # 128 blocks
    try:
        lib.set_quantise_once_override(2)
        assert lib.plan_matvec(128256, 4096, 1)["quantise_once"] == 1
        lib.set_quantise_once_override(1)
        assert lib.plan_matvec(4096, 14336, 8)["quantise_once"] == 0
    finally:
        lib.set_quantise_once_override(0)


def test_widest_rows_that_fit(lib):
    """One q8 vector (cols/256 blocks at 336 bytes of shared memory each) must
    fit beside two 4608-byte stages: cols 169984 is the widest on GB300."""
    p = lib.plan_matvec(7, 169984, 2, sm_count=152, smem_optin=232448)
    assert p["batch_per_launch"] == 1 and p["launches"] == 2 and p["segments"] == 21
    assert p["smem_bytes"] <= 232448
    with pytest.raises(lib.XQError) as e:
        lib.plan_matvec(7, 169984 + 256, 1, sm_count=152, smem_optin=232448)
    assert e.value.status == 3 and "shared memory" in e.value.detail
