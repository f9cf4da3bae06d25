"""Builds libmxgemm.so in-tree with nvcc for sm_103a.

    python -m mxfp8_norm_quant_gb300.build [--force] [-v]

Each .cu file is compiled separately and in parallel into _build/, then linked
into mxfp8_norm_quant_gb300/libmxgemm.so with the CUDA runtime linked
statically (the library needs only libc/libstdc++ at load time; the driver
API is reached through cudaGetDriverEntryPointByVersion).
"""

from __future__ import annotations

import argparse
import os
import platform
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmxgemm.so")

SOURCES = ["k_rowquant.cu", "k_rownorm_sp.cu", "k_rownorm_bf16.cu", "k_gemm.cu", "api.cu"]
HEADERS = ["mx_ptx.cuh", "mx_kernels.h", "norm_plan.h", "row_common.cuh", "row_lb.cuh", "quant_lb.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-fvisibility=hidden", "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        raise RuntimeError("nvcc not found; the CUDA 13 toolkit is required to build libmxgemm")
    return nvcc


def _deps_mtime() -> float:
    paths = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "mxgemm.h"), __file__]
    return max(os.path.getmtime(p) for p in paths)


def _compile(nvcc: str, src: str, force: bool, verbose: bool, ptxas_v: bool) -> str:
    obj = os.path.join(BUILD, src.replace(".cu", ".o"))
    src_path = os.path.join(CSRC, src)
    if (not force and os.path.exists(obj)
            and os.path.getmtime(obj) >= max(os.path.getmtime(src_path), _deps_mtime())):
        return obj
    cmd = [nvcc, *ARCH, *CFLAGS, "-I", INCLUDE, "-I", CSRC, "-c", src_path, "-o", obj]
    if ptxas_v:
        cmd += ["-Xptxas", "-v"]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if verbose or ptxas_v:
        sys.stdout.write(r.stdout + r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False, ptxas_v: bool = False) -> str:
    """Compile (if out of date) and link libmxgemm.so; returns its path."""
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    # objects built on another machine type (x86 here, aarch64 on the GPU machine)
    # are never reused
    stamp = os.path.join(BUILD, "MACHINE")
    machine = platform.machine()
    if not os.path.exists(stamp) or open(stamp).read().strip() != machine:
        force = True
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(nvcc, s, force, verbose, ptxas_v), SOURCES))
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < max(os.path.getmtime(o) for o in objs):
        cmd = [nvcc, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", LIB + ".tmp", *objs]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link of libmxgemm.so failed:\n{r.stdout}\n{r.stderr}")
        os.replace(LIB + ".tmp", LIB)
    with open(stamp, "w") as f:
        f.write(machine + "\n")
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("-v", "--verbose", action="store_true")
    ap.add_argument("--ptxas-v", action="store_true", help="print register / shared-memory usage")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose, ptxas_v=a.ptxas_v))
