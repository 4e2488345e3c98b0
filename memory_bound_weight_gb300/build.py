"""Compile the CUDA sources of this package into libmbw.so (sm_103a only).

One nvcc process per translation unit, run in parallel, then one link step.
The library is built in-tree (memory_bound_weight_gb300/libmbw.so) and loaded
with ctypes by the binding.
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
LIB = os.path.join(PKG, "libmbw.so")
GEN_LIB = os.path.join(PKG, "libmbw_inputs.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
                     "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]

# translation units of libmbw.so (the product) and of the input generator
LIB_SOURCES = ["abi.cu", "plan.cu", "gemv_simt.cu", "gemv_mma.cu", "gemv_tma.cu", "gemv_lat.cu", "gemm_tc.cu",
               "gemv_awq_batch.cu", "quantize.cu"]
GEN_SOURCES = ["gen_inputs.cu"]


def _nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _stale(out: str, deps: list[str]) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def _headers() -> list[str]:
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    return hs + [os.path.join(INCLUDE, "mbw.h")]


def _compile(src: str, ptxas_v: bool) -> str:
    obj = os.path.join(BUILD, os.path.basename(src) + ".o")
    if _stale(obj, [src] + _headers()):
        cmd = [_nvcc(), *NVCC_FLAGS, "-c", src, "-o", obj]
        if ptxas_v:
            cmd += ["-Xptxas", "-v"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if ptxas_v:
            sys.stderr.write(r.stderr)
    return obj


def _link(objs: list[str], out: str) -> None:
    if not _stale(out, objs):
        return
    tmp = out + ".tmp"
    cmd = [_nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)


def build(ptxas_v: bool = False) -> str:
    """Build libmbw.so and libmbw_inputs.so; returns the path of libmbw.so."""
    os.makedirs(BUILD, exist_ok=True)
    srcs = [os.path.join(CSRC, f) for f in LIB_SOURCES + GEN_SOURCES]
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(lambda s: _compile(s, ptxas_v), srcs))
    _link(objs[: len(LIB_SOURCES)], LIB)
    _link(objs[len(LIB_SOURCES):], GEN_LIB)
    return LIB


if __name__ == "__main__":
    print(build(ptxas_v="-v" in sys.argv))
