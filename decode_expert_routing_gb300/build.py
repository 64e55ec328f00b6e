"""Builds the CUDA library libmoe_route.so in-tree with nvcc (sm_103a only).

Each translation unit compiles in its own nvcc process, in parallel, then one
nvcc call links the shared library against the shared CUDA runtime (the same
libcudart PyTorch loads, so streams pass between them).  No cmake.
"""

from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmoe_route.so")
INCLUDE = os.path.join(ROOT, "include")

SOURCES = ["abi.cu", "kernels_gemv.cu", "kernels_aux.cu", "kernel_route.cu", "kernel_route_spw6.cu",
           "kernel_route_spw7.cu", "kernel_tc_gemv.cu", "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# No --use_fast_math: the quantiser and the sigmoid recipe need IEEE rounding
# and subnormals (no flush to zero).
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-Xcompiler", "-fno-strict-aliasing", "-I" + INCLUDE]


def nvcc() -> str:
    for cand in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        p = os.path.join(cand, "bin", "nvcc") if cand else ""
        if p and os.path.exists(p):
            return p
    return "nvcc"


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "moe_route.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


TRACE_LIB = os.path.join(HERE, "libmoe_route_trace.so")


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          trace: bool = False) -> str:
    """Compile and link libmoe_route.so; returns its path.  trace=True builds
    libmoe_route_trace.so instead, with per-CTA phase stamps (-DMR_TRACE)."""
    lib = TRACE_LIB if trace else LIB
    if not force and up_to_date(lib):
        return lib
    bdir = BUILD + ("_trace" if trace else "")
    os.makedirs(bdir, exist_ok=True)
    cc = nvcc()
    extra = (["-Xptxas", "-v"] if ptxas_info else []) + (["-DMR_TRACE"] if trace else [])

    def compile_one(src):
        obj = os.path.join(bdir, os.path.splitext(src)[0] + ".o")
        cmd = [cc, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose or ptxas_info:
        for _, log in results:
            if log.strip():
                sys.stderr.write(log)
    objs = [o for o, _ in results]
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                trace="--trace" in sys.argv))
