"""Builds the CUDA library ``_build/libxq.so`` in-tree with nvcc for sm_103a.

The translation units are compiled in parallel (one -gencode each), then
linked into one shared library with the CUDA runtime linked statically, so the
library needs only the NVIDIA driver at run time.  ptxas resource reports are
kept beside the objects (``_build/*.ptxas.log``) for the spill gate.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(BUILD, "libxq.so")
SOURCES = ["xq_api.cu", "xq_matvec_q4k.cu", "xq_matvec_q4k_rb2.cu", "xq_matvec_q4k_tc.cu",
           "xq_matvec_cb4.cu", "xq_matvec_cb4r.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
              f"-I{INCLUDE}"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def _inputs() -> list[str]:
    return (glob.glob(os.path.join(CSRC, "*")) + [os.path.join(INCLUDE, "xq.h"),
                                                  os.path.abspath(__file__)])


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if stale) and return the path of libxq.so."""
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    procs = []
    for src in SOURCES:
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        log = open(os.path.join(BUILD, src.replace(".cu", ".ptxas.log")), "w")
        cmd = [nvcc(), *ARCH, *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        procs.append((src, obj, log, subprocess.Popen(cmd, stdout=log, stderr=subprocess.STDOUT)))
    failed = []
    for src, obj, log, p in procs:
        p.wait()
        log.close()
        if p.returncode != 0:
            failed.append(src)
    if failed:
        msgs = []
        for src in failed:
            with open(os.path.join(BUILD, src.replace(".cu", ".ptxas.log"))) as f:
                msgs.append(f"--- {src}\n" + f.read()[-4000:])
        raise RuntimeError("nvcc failed:\n" + "\n".join(msgs))
    tmp = LIB + f".tmp{os.getpid()}"
    objs = [os.path.join(BUILD, s.replace(".cu", ".o")) for s in SOURCES]
    subprocess.run([nvcc(), *ARCH, "-shared", "--cudart", "static", "-o", tmp, *objs],
                   check=True)
    os.replace(tmp, LIB)
    if verbose:
        print(f"built {LIB}", file=sys.stderr)
    return LIB


def ptxas_report() -> dict[str, dict[str, int]]:
    """Registers, spill bytes and stack-frame bytes (local arrays) per kernel,
    parsed from the ptxas logs."""
    out: dict[str, dict[str, int]] = {}
    for log in glob.glob(os.path.join(BUILD, "*.ptxas.log")):
        current = None
        with open(log) as f:
            for line in f:
                if "Compiling entry function" in line:
                    current = line.split("'")[1]
                    out[current] = {"registers": -1, "spill_stores": 0, "spill_loads": 0,
                                    "stack_frame": 0}
                elif current and "spill stores" in line:
                    parts = line.replace(",", "").split()
                    out[current]["spill_stores"] = int(parts[parts.index("spill") - 2])
                    out[current]["spill_loads"] = int(parts[parts.index("loads") - 3])
                    if "stack" in parts:
                        out[current]["stack_frame"] = int(parts[parts.index("stack") - 2])
                elif current and "Used" in line and "registers" in line:
                    parts = line.replace(",", " ").split()
                    out[current]["registers"] = int(parts[parts.index("registers") - 1])
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
