"""Build ``libattnres.so`` in-tree with nvcc for GB300 (sm_103a).

The translation units compile in parallel into ``_build/`` at the repository
root and link into ``depth_wise_attention_block_gb300/libattnres.so`` with
the CUDA runtime linked statically.  Usage: ``python -m
depth_wise_attention_block_gb300.build [-v] [--ptxas-info]``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_PATH = os.path.join(PKG_DIR, "libattnres.so")
SOURCES = ["aggregate.cu", "ring_fixed_s.cu", "ring_fixed_s_fused.cu", "ring_fixed_s_fused_noprev.cu",
           "aggregate_multi.cu", "aggregate_split.cu",
           "backward.cu", "twophase.cu", "twophase_tc.cu", "elementwise.cu", "api.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC,-O2,-Wall",
                     "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: libattnres needs the CUDA toolkit to build")


def _run(cmd: list[str], verbose: bool) -> str:
    if verbose:
        print(" ".join(cmd), flush=True)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"command failed ({res.returncode}): {' '.join(cmd)}\n{res.stdout}\n{res.stderr}")
    return res.stdout + res.stderr


def build(verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile and link; returns the path of the shared library."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    nv = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    jobs = []
    for src in SOURCES:
        obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
        jobs.append((obj, [nv, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]))
    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        logs = list(ex.map(lambda j: _run(j[1], verbose), jobs))
    if ptxas_info:
        for (obj, _), log in zip(jobs, logs):
            print(f"== {os.path.basename(obj)}\n{log}")
    tmp = LIB_PATH + ".tmp"
    _run([nv, *ARCH, "-shared", "-o", tmp, *[o for o, _ in jobs]], verbose)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, ptxas_info="--ptxas-info" in sys.argv))
