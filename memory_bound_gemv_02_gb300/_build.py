"""In-tree build of the GEMV C-ABI library ``_lib/libgemv.so`` with nvcc.

Each translation unit is compiled for sm_103a in parallel, then linked into a
shared library with the CUDA runtime linked statically (so the library does
not depend on which libcudart the host process loaded).  No torch extension
ABI is involved: the Python side talks to the library through ctypes.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJDIR = os.path.join(ROOT, "_build", "gemv")
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "libgemv.so")
HOST_TOOL_SRC = "bench_tool_main.cu"
HOST_TOOL = os.path.join(LIBDIR, "gemv_bench_tool")  # native host-overhead and read-ceiling measurements

SOURCES = ["gemv_api.cu", "gemv_kernels_f16.cu", "gemv_kernels_bf16.cu", "gemv_bulk_f16.cu", "gemv_bulk_bf16.cu",
           "gla_decode.cu"]
HEADERS = [os.path.join(CSRC, h) for h in ("gemv_internal.h", "gemv_kernels.cuh", "gemv_tiles.cuh",
                                           "gemv_bulk.cuh")] + \
    [os.path.join(INCLUDE, "gemv.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-I" + INCLUDE, "-I" + CSRC]

_lock = threading.Lock()


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the GEMV library needs the CUDA toolkit to build")
    return cand


def _stale() -> bool:
    if not os.path.exists(LIB) or not os.path.exists(HOST_TOOL):
        return True
    t = min(os.path.getmtime(LIB), os.path.getmtime(HOST_TOOL))
    deps = [os.path.join(CSRC, s) for s in SOURCES + [HOST_TOOL_SRC]] + HEADERS + [os.path.abspath(__file__)]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile (if needed) and return the path of ``libgemv.so``."""
    with _lock:
        if not force and not _stale():
            return LIB
        os.makedirs(OBJDIR, exist_ok=True)
        os.makedirs(LIBDIR, exist_ok=True)
        exe = nvcc()

        def compile_one(src):
            obj = os.path.join(OBJDIR, os.path.splitext(src)[0] + ".o")
            cmd = [exe, *NVCC_FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
            if verbose and (r.stdout or r.stderr):
                print(r.stdout + r.stderr)
            return obj

        with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
            objs = list(ex.map(compile_one, SOURCES))
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [exe, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-cudart", "static", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
        # the native measurement tool, linked against the library just built
        tmp = HOST_TOOL + f".tmp{os.getpid()}"
        cmd = [exe, *NVCC_FLAGS, *extra_flags, os.path.join(CSRC, HOST_TOOL_SRC), "-o", tmp,
               "-L" + LIBDIR, "-lgemv", "-Xlinker", "-rpath,$ORIGIN"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"measurement tool build failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, HOST_TOOL)
        return LIB


def ensure_built() -> str:
    return build(force=False)


def lib_path() -> str:
    return LIB
