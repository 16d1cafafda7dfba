"""Build libssd.so (in-tree) with nvcc for sm_103a.

Each CUDA source is compiled in parallel, then linked into one shared
library beside this file.  Usage: ``python -m mamba_ssd_chunked_scan_gb300.build``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libssd.so")
SOURCES = ["ssd_api.cu", "ssd_simt.cu", "ssd_tc.cu", "ssd_agg.cu", "ssd_step.cu", "ssd_bwd.cu", "ssd_bwd_tc.cu", "ssd_gate_norm.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for c in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def _deps():
    ds = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    ds.append(os.path.join(ROOT, "include", "ssd.h"))
    ds.append(os.path.abspath(__file__))
    return ds


def build(force: bool = False, verbose: bool = False, extra=()) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    deps = _deps()
    objs, procs = [], []
    for src in SOURCES:
        path = os.path.join(CSRC, src)
        if not os.path.exists(path):
            continue
        obj = os.path.join(OUT_DIR, src.replace(".cu", ".o"))
        objs.append(obj)
        if force or _stale(obj, deps):
            cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", path, "-o", obj]
            if verbose:
                print(" ".join(cmd), flush=True)
            procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for cmd, pr in procs:
        out, _ = pr.communicate()
        if pr.returncode != 0 or verbose:
            sys.stderr.write(out.decode(errors="replace"))
        if pr.returncode != 0:
            failed.append(cmd)
    if failed:
        raise RuntimeError(f"nvcc failed: {failed[0]}")
    if force or procs or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.check_call([nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"])
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv,
          extra=["-Xptxas", "-v"] if "--ptxas" in sys.argv else [])
    print(LIB)
