"""Builds liblaneformer.so (the C-ABI engine) in-tree for sm_103a with nvcc.

Translation units are compiled in parallel into ``_build/`` and linked into
``decode_persistent_sm_gb300/liblaneformer.so``.  No CMake, no torch
extension machinery: the library exports plain C symbols (include/laneformer.h).
``build(debug=True)`` makes ``liblaneformer_debug.so`` from the same sources
with ``-DLF_DEBUG`` (device-side bounds checks, canaries around the engine's
buffers) in ``_build_debug/``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "liblaneformer.so")
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "liblaneformer_debug.so")
SOURCES = ["lf_plan.cpp", "lf_kernel.cu", "lf_runtime.cu", "lf_noalloc.cu", "lf_tc_gemm.cu", "lf_prefill.cu",
           "lf_pf_attn_tc.cu", "lf_sample.cu", "lf_gemv_tc.cu", "lf_batch.cu", "lf_stream.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "laneformer.h"))
    return files


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in _deps())


def _compile(src: str, verbose: bool, debug: bool) -> str:
    obj = os.path.join(BUILD_DEBUG if debug else BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), "-c", os.path.join(CSRC, src), "-o", obj, "-O3", "-std=c++17", "-lineinfo",
           *ARCH, "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]
    if debug:
        cmd += ["-DLF_DEBUG"]
    if src.endswith(".cu"):
        cmd += ["--expt-relaxed-constexpr"]
        if verbose:
            cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        print(r.stdout + r.stderr, file=sys.stderr)
    return obj


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile (if sources changed) and return the path of liblaneformer.so
    (liblaneformer_debug.so with debug=True)."""
    lib = LIB_DEBUG if debug else LIB
    if not force and not _stale(lib):
        return lib
    os.makedirs(BUILD_DEBUG if debug else BUILD, exist_ok=True)
    with cf.ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, debug), SOURCES))
    tmp = lib + ".tmp"
    r = subprocess.run([nvcc(), "-shared", *ARCH, "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


def build_all(force: bool = False, verbose: bool = False):
    """Both libraries, compiled side by side."""
    with cf.ThreadPoolExecutor(2) as ex:
        return list(ex.map(lambda d: build(force, verbose, d), (False, True)))


if __name__ == "__main__":
    print(build_all(force="--force" in sys.argv, verbose="-v" in sys.argv))
