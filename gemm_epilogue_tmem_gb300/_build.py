"""Build libgf.so (the C-ABI library) in-tree with nvcc for sm_103a.

Each kernel family is its own translation unit, compiled in parallel; the
CUDA runtime is linked statically with its symbols hidden, so the library
exports exactly the gf_* entry points of include/gf.h.
"""
from __future__ import annotations

import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libgf.so")

SOURCES = ["runtime.cu", "k_none_bias.cu", "k_relu.cu", "k_drelu.cu", "k_gelu.cu", "k_swiglu.cu", "noalloc.cu"]
HEADERS = ["ptx.cuh", "gemm_kernel.cuh", "gemm_kernel_2sm.cuh", "dispatch.cuh", "launch.h",
           "params.h", "runtime_internal.h"]

NVCC_FLAGS = [
    "-std=c++17", "-O3", "-lineinfo",
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-Xcompiler", "-fPIC,-fvisibility=hidden",
    "-I", INCLUDE, "-I", CSRC,
]


def _newest_input() -> float:
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(INCLUDE, "gf.h"),
                                                                 __file__]
    return max(os.path.getmtime(f) for f in files)


def compile_cmd(src: str, obj: str, extra=()) -> list[str]:
    return ["nvcc", *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _newest_input():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    objs = [os.path.join(BUILD, os.path.splitext(s)[0] + ".o") for s in SOURCES]

    def one(args):
        src, obj = args
        r = subprocess.run(compile_cmd(src, obj, extra), capture_output=True, text=True)
        return src, r

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(one, zip(SOURCES, objs)))
    for src, r in results:
        if verbose or ptxas_info:
            print(r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    link = ["nvcc", "-shared", "-gencode", "arch=compute_103a,code=sm_103a", "-o", LIB + ".tmp",
            *objs, "-Xlinker", "--exclude-libs,ALL", "-Xlinker", "-Bsymbolic"]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
