"""Build libqoq.so (sm_103a) in-tree with nvcc.

Each .cu file compiles to an object in parallel, then nvcc links the shared
library (CUDA runtime linked statically, so the library loads without a GPU
and without libcudart on the loader path).  Output:
w4a8_quantized_serving_gb300/_build/libqoq.so, and beside it libqoq_probe.so,
the benchmark's streaming-read probe (not part of the W4A8 path).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
PKG = os.path.dirname(HERE)
ROOT = os.path.dirname(PKG)
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libqoq.so")
SOURCES = ["api.cu", "act_quant.cu", "pack.cu", "gemm.cu", "gemm_decode.cu", "gemm_no_alloc.cu"]
PROBE_LIB = os.path.join(BUILD, "libqoq_probe.so")
PROBE_SOURCES = ["probe_stream.cu", "probe_mma.cu"]
HEADERS = ["internal.h", "ptx.cuh", "gemm_common.cuh", os.path.join("..", "..", "include", "qoq.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O3",
                     "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None) -> str:
    os.makedirs(BUILD, exist_ok=True)
    headers = [os.path.join(HERE, h) for h in HEADERS]
    flags = NVCC_FLAGS + list(extra_flags or [])
    nv = nvcc()

    def compile_one(src: str) -> str:
        path = os.path.join(HERE, src)
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        if force or _stale(obj, [path] + headers):
            cmd = [nv, *flags, "-c", path, "-o", obj + ".tmp"]
            if verbose:
                print(" ".join(cmd), flush=True)
            subprocess.check_call(cmd)
            os.replace(obj + ".tmp", obj)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES) + len(PROBE_SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES + PROBE_SOURCES))

    def link(target: str, parts: list[str]) -> None:
        if force or _stale(target, parts):
            tmp = target + f".{os.getpid()}.tmp"
            cmd = [nv, *ARCH, "-shared", "-o", tmp, *parts]
            if verbose:
                print(" ".join(cmd), flush=True)
            subprocess.check_call(cmd)
            os.replace(tmp, target)

    link(LIB, objs[: len(SOURCES)])
    link(PROBE_LIB, objs[len(SOURCES):])
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
