"""Builds libsi_moe.so in-tree with nvcc for sm_103a (GB300).

Each translation unit is compiled in parallel into ``_build/``; the shared
library is linked next to this file. Rebuilds only when a source or header is
newer than the library.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libsi_moe.so")
SOURCES = ["quant_norm.cu", "router.cu", "ffn.cu", "batched.cu", "stack.cu", "requant.cu", "api.cu"]
HEADERS = [os.path.join(CSRC, "common.cuh"), os.path.join(CSRC, "host.hpp"),
           os.path.join(CSRC, "topk.cuh"), os.path.join(CSRC, "tc.cuh"), os.path.join(CSRC, "norm.cuh"),
           os.path.join(ROOT, "include", "si_moe.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libsi_moe.so")


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, build_dir: str = BUILD, extra=()) -> str:
    obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
    path = os.path.join(CSRC, src)
    if _stale(obj, [path] + HEADERS):
        cmd = [nvcc()] + FLAGS + list(extra) + ["-c", path, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj


def build(force: bool = False, verbose: bool = False, trace: bool = False) -> str:
    """Compile every translation unit and link libsi_moe.so; return its path.

    trace=True builds libsi_moe_trace.so instead, with per-phase timestamp
    recording (-DSI_TRACE) for profiling; the product library never has it.
    """
    build_dir = BUILD + ("_trace" if trace else "")
    lib = LIB.replace(".so", "_trace.so") if trace else LIB
    extra = ["-DSI_TRACE"] if trace else []
    os.makedirs(build_dir, exist_ok=True)
    if force:
        for f in os.listdir(build_dir):
            os.remove(os.path.join(build_dir, f))
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda src: _compile(src, build_dir, extra), SOURCES))
    if force or _stale(lib, objs):
        tmp = lib + ".tmp"
        cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    if verbose:
        print("built", lib)
    return lib


if __name__ == "__main__":
    build(verbose=True)
