"""Build ``libflash_mca.so`` in-tree with nvcc for sm_103a.

Three translation units compile in parallel (the C-ABI layer, the SIMT kernels
and the tensor-core kernels) and link into one shared library next to this
file.  The CUDA runtime is linked statically and the driver's tensor-map
encoder is looked up at run time, so the library loads on a machine without a
GPU driver (only calls that touch the device need one).

The package runs ``build()`` on import (a no-op when the library is newer than
its sources); ``python -m flash_mixed_chunk_gb300.build [--force] [-v]`` runs
it by hand.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libflash_mca.so")

SOURCES = ["api.cpp", "simt.cu", "tc.cu", "noalloc.cu", "decode.cu", "backward.cu"]
HEADERS = ["launch.h", "ptx.cuh", "tc_common.cuh", "tc_prep.cuh", "tc_attn.cuh", "tc_fused.cuh", "tc_walk.cuh", "tc_pair.cuh", "tc_gemm.cuh", "tc_bgemm.cuh", "tc_bwd.cuh", "tc_backward.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libflash_mca.so")


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    deps.append(os.path.join(INCLUDE, "flash_mca.h"))
    deps.append(os.path.abspath(__file__))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(BUILD, src.rsplit(".", 1)[0] + ".o")
        objs.append(obj)
        cmd = [cc, *ARCH, *COMMON, "-c", os.path.join(CSRC, src), "-o", obj]
        if src.endswith(".cu"):
            cmd += ["-Xptxas", "-v"] if verbose else []
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode != 0:
            sys.stdout.write(out.decode(errors="replace"))
        if p.returncode != 0:
            failed.append(src)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    tmp = LIB + f".tmp{os.getpid()}"
    link = [cc, *ARCH, "-shared", "-o", tmp, *objs]
    subprocess.run(link, check=True)
    os.replace(tmp, LIB)
    return LIB

