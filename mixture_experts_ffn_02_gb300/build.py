"""Builds the sm_103a shared library ``_build/libmoe_gb300.so`` in-tree.

Each CUDA translation unit is compiled in parallel with nvcc for
``-gencode arch=compute_103a,code=sm_103a`` and linked into one shared object
that exports the C ABI of ``include/moe.h``.  No CMake, no torch extension
machinery: plain nvcc, so the same command works on x86 and on Arm hosts.

``build(debug=True)`` builds the checking variant ``_build/libmoe_gb300_debug.so``
(objects under ``_build/debug``) with ``-DMOE_DEBUG_BOUNDS``: its kernels check
every row index they read from ``inv`` and the segment table against the rows
that exist, latch MOE_ERR_BOUNDS in the status word and skip the access.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libmoe_gb300.so")
LIB_DEBUG = os.path.join(BUILD, "libmoe_gb300_debug.so")
SOURCES = ["moe_api.cu", "moe_dispatch.cu", "moe_gemm.cu", "moe_mx.cu", "moe_router_tc.cu",
           "moe_static.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(extra=()):
    return [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
            "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC, *extra]


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    deps = [src] + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    deps.append(os.path.join(INCLUDE, "moe.h"))
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, ptxas_info: bool = False, force: bool = False,
          debug: bool = False) -> str:
    objdir = os.path.join(BUILD, "debug") if debug else BUILD
    lib = LIB_DEBUG if debug else LIB
    os.makedirs(objdir, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    if debug:
        extra.append("-DMOE_DEBUG_BOUNDS")

    def compile_one(src):
        path = os.path.join(CSRC, src)
        obj = os.path.join(objdir, src.replace(".cu", ".o"))
        if not force and not ptxas_info and not _stale(obj, path):
            return obj, ""
        cmd = [cc, *_flags(extra), "-c", path, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    objs = [o for o, _ in results]
    if verbose or ptxas_info:
        for _, log in results:
            if log:
                print(log, file=sys.stderr)
    if force or not os.path.exists(lib) or any(os.path.getmtime(o) > os.path.getmtime(lib)
                                                for o in objs):
        cmd = [cc, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", lib, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    return lib


if __name__ == "__main__":
    print(build(verbose=True, ptxas_info="-v" in sys.argv, force="-f" in sys.argv,
                debug="--debug" in sys.argv))
