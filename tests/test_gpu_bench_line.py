"""The bench's JSON line on a small case: one line, the keys the measurement
contract asks for, and figures that agree with one another (device time,
roofline, end to end with the host copies counted, launches, clocks)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


def test_bench_line_contract():
    d = _run("--case", "c2_q4k_4096x4096_b1", "--steps", "200", "--warmup", "5",
             "--rounds", "4", "--cpu-seconds", "0.2")
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 200 and d["warmup"] == 5
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert "workload" in d["config"]
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    e = d["e2e"]
    assert e["value"] > 0 and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 4 * 4096 and e["d2h_bytes_per_step"] == 4 * 4096
    assert e["ms_per_step"] <= e["median_ms_per_step"]
    assert d["gpu_launches"] >= d["steps"]
    rd = d["rounds"]
    assert rd["n"] == 4 and len(rd["step_us"]) == 4 and len(rd["matvec_us"]) == 4
    assert rd["min_us"] <= rd["median_us"] <= rd["max_us"]
    assert abs(rd["median_us"] - d["ms_per_step"] * 1e3) < 1e-3
    b = d["bytes"]
    assert b["per_step"] == b["weights"] + b["q8"] == 9437184 + 16 * 320
    assert abs(d["value"] - b["per_step"] / (d["ms_per_step"] * 1e-3) / 1e9) < 1e-6 * d["value"]
    c = d["cpu_baseline"]
    assert c["kind"] == "oracle" and c["cores"] >= 1 and c["value"] > 0
    assert c["cores"] == c["affinity_cores"] and c["cpu_model"] and c["hostname"]
    assert c["single_thread"]["value"] > 0
    assert d["clocks"]["sm_mhz"] > 0
    assert d["device_status"] == 0


def test_bench_line_tensor_opt_in():
    """--tensor on times the tcgen05 form of the batch-8 mat-vec and says so;
    the planner's line names the dp4a kernel."""
    d = _run("--case", "c3_q4k_up_14336x4096_b8", "--steps", "100", "--warmup", "5",
             "--rounds", "2", "--cpu-seconds", "0.1", "--tensor", "on")
    assert d["plan"]["tensor"] == 1 and d["config"]["tensor"].startswith("tcgen05")
    assert "xq_tc_q4k_kernel" in d["roofline"]["kernel"] and "tcgen05" in d["dtype"]
    assert d["device_status"] == 0
    d = _run("--case", "c3_q4k_up_14336x4096_b8", "--steps", "100", "--warmup", "5",
             "--rounds", "2", "--cpu-seconds", "0.1")
    assert d["plan"]["tensor"] == 0 and "tensor" not in d["config"]
    assert "xq_matvec_kernel" in d["roofline"]["kernel"] and "dp4a" in d["dtype"]


def test_reference_arm_line():
    d = _run("--impl", "reference", "--case", "c1_q4k_256x1024_b1", "--steps", "3",
             "--warmup", "3")
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0
