"""Compile the CUDA library in-tree for sm_103a: libbsm_fa.so next to this file.

Usage: python -m block_sparse_masked_gb300.build [-f] [--checked]
       (or build() / build(checked=True) from Python)

``checked=True`` builds the debug variant libbsm_fa_checked.so with
-DBSM_CHECKED: every plan-derived global index in the planner, forward and
backward kernels is checked against the plan's exact sizes; a violation sets
bit 4 of the device error word (fa_device_error_flags) and the access is
redirected or skipped instead of faulting.  The binding loads it when
BSM_FA_CHECKED=1 is set in the environment.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "libbsm_fa.so")
OUT_CHECKED = os.path.join(HERE, "libbsm_fa_checked.so")
BUILD_DIR = os.path.join(os.path.dirname(HERE), "_build")
SOURCES = ["fa_api.cu", "planner.cu", "attn_fwd.cu", "attn_fwd_pair.cu", "attn_fwd_kt.cu", "attn_bwd.cu",
           "attn_decode.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "--expt-relaxed-constexpr", "-Xptxas", "-v"]


def nvcc() -> str:
    cand = [os.environ.get("NVCC", ""), shutil.which("nvcc") or "", "/usr/local/cuda/bin/nvcc"]
    for c in cand:
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _compile(src: str, verbose: bool, obj_dir: str, extra: list) -> str:
    obj = os.path.join(obj_dir, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    log = r.stdout + r.stderr
    with open(obj + ".log", "w") as f:
        f.write(" ".join(cmd) + "\n" + log)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{log}")
    if verbose:
        print(log, file=sys.stderr)
    return obj


def build(verbose: bool = False, force: bool = False, checked: bool = False) -> str:
    out = OUT_CHECKED if checked else OUT
    obj_dir = os.path.join(BUILD_DIR, "checked") if checked else BUILD_DIR
    extra = ["-DBSM_CHECKED"] if checked else []
    os.makedirs(obj_dir, exist_ok=True)
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    deps = srcs + [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".h", ".cuh"))]
    deps.append(os.path.join(os.path.dirname(HERE), "include", "fa.h"))
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) > max(os.path.getmtime(d) for d in deps)):
        return out
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, obj_dir, extra), SOURCES))
    tmp = out + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv, checked="--checked" in sys.argv))
