"""Build libqoq.so in-tree for sm_103a with nvcc (no cmake, no torch extension).

Each .cu file is compiled to an object in parallel, then linked into
``w4a8_quantized_serving_qoq_gb300/_lib/libqoq.so``; the bounds-check build
(the same sources compiled with QOQ_DEBUG_BOUNDS) goes to ``libqoq_debug.so``
beside it.  Rebuilds a library only when a source or header is newer than it.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "libqoq.so")
LIB_DEBUG = os.path.join(LIBDIR, "libqoq_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libqoq.so")
    return cand


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list[str]:
    return sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(CSRC, "*.inc")) + [
        os.path.join(ROOT, "include", "qoq.h"), os.path.abspath(__file__)]


def library(debug: bool) -> str:
    return LIB_DEBUG if debug else LIB


def up_to_date(debug: bool = False) -> bool:
    lib = library(debug)
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, debug: bool | None = None) -> str:
    """Build the release library (debug=False), the bounds-check one
    (debug=True) or both (None, the default; all objects compile in one
    parallel pool).  Returns the path of the release library, or of the
    bounds-check one when only it was asked for."""
    variants = [False, True] if debug is None else [debug]
    variants = [d for d in variants if force or not up_to_date(d)]
    if variants:
        os.makedirs(LIBDIR, exist_ok=True)
        nvcc = _nvcc()

        def compile_one(job: tuple[str, bool]) -> str:
            src, dbg = job
            objdir = os.path.join(LIBDIR, "obj_debug" if dbg else "obj")
            os.makedirs(objdir, exist_ok=True)
            obj = os.path.join(objdir, os.path.basename(src) + ".o")
            extra = ["-DQOQ_DEBUG_BOUNDS"] if dbg else []
            cmd = [nvcc, *ARCH, *FLAGS, *extra, "-I", os.path.join(ROOT, "include"), "-c", src, "-o", obj]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
            if verbose and (r.stdout or r.stderr):
                print(r.stdout, r.stderr)
            return obj

        # largest sources first: the two tensor-core GEMM files set the build time
        jobs = [(src, d) for src in sorted(sources(), key=os.path.getsize, reverse=True) for d in variants]
        with cf.ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1))) as ex:
            objs = list(ex.map(compile_one, jobs))
        for d in variants:
            lib = library(d)
            mine = [o for o, (_, dj) in zip(objs, jobs) if dj == d]
            tmp = lib + f".{os.getpid()}.tmp"
            r = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *mine], capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
            os.replace(tmp, lib)
    return LIB_DEBUG if debug else LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
