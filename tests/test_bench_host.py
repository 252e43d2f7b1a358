"""Host logic of bench.py without a GPU: the N>1 path (replicas, barrier and
max-over-ranks timing) on two gloo ranks on the CPU, the reference arm's rank
handling, and the algorithmic byte counts."""
import io
import json
import multiprocessing as mp
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist = bench.dist_init(world, "gloo")
    bench.barrier(dist)
    # each rank reports a different step time; every rank must see the slowest
    slowest = bench.max_over_ranks(0.5 + rank, dist)
    bench.barrier(dist)
    q.put((rank, slowest, dist.get_world_size()))
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(0, 1.5, 2), (1, 1.5, 2)]


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.dist_init(1, "gloo") is None
    assert bench.max_over_ranks(2.5, None) == 2.5


def test_reference_arm_prints_only_on_rank_zero(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3", "--gpus", "2"])
    assert buf.getvalue() == ""


def test_reference_arm_line(monkeypatch):
    """A short reference-arm run on a small case prints one JSON line with the
    contract's keys."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main(["--impl", "reference", "--steps", "2", "--warmup", "3",
                    "--case", "c1_q4k_256x1024_b1"])
    lines = [l for l in buf.getvalue().splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    for k in ("affinity_cores", "cpu_model", "hostname"):
        assert k in d["cpu_baseline"], k
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["steps"] == 2 and d["warmup"] == 3 and d["higher_is_better"] is True


def test_algorithmic_bytes():
    """The metric's bytes of one mat-vec: the weights once and the activation
    as q8 blocks; the y write and the f32 activation are listed, not counted."""
    sys.path.insert(0, ROOT)
    import bench
    import synthetic
    c = synthetic.CASES["c5_q4k_128256x4096_b1"]
    b = bench.step_bytes(c)
    assert b["weights"] == 128256 * 16 * 144 == 295_501_824
    assert b["q8"] == 16 * 320
    assert b["algorithmic"] == 295_501_824 + 16 * 320
    assert b["y"] == 4 * 128256 and b["x"] == 4 * 4096
    c8 = synthetic.CASES["c5_q4k_128256x4096_b8"]
    assert bench.step_bytes(c8)["algorithmic"] == 295_501_824 + 8 * 16 * 320
    cb = synthetic.CASES["hbm_cb4_128256x4096_b1"]
    assert bench.step_bytes(cb)["weights"] == 128256 * 128 * 18 == 295_501_824


def test_host_context():
    sys.path.insert(0, ROOT)
    import bench
    assert 1 <= bench.host_cores() <= (os.cpu_count() or 1)
    assert isinstance(bench.cpu_model(), str) and bench.cpu_model()


def test_warmup_floor():
    sys.path.insert(0, ROOT)
    import bench
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])
