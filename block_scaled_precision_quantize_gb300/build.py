"""Build the CUDA library (libbsq.so) in-tree for sm_103a with nvcc.

Each translation unit is compiled in parallel, then linked into a shared
library under block_scaled_precision_quantize_gb300/_build/. No fast math:
IEEE division and reciprocals and no flush-to-zero, as the bit-exact
quantizer contract requires.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libbsq.so")
SOURCES = ["api.cu", "quant.cu", "requant.cu", "gemm_fp4.cu", "moe.cu", "ceiling.cu"]
HEADERS = ["common.cuh", "kernels.h", "tc_ptx.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-ftz=false", "-prec-div=true",
              "-prec-sqrt=true", "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    files.append(os.path.join(ROOT, "include", "bsq.h"))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, extra_flags=None) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    flags = NVCC_FLAGS + list(extra_flags or [])

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        cmd = [cc, *ARCH, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    r = subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


STALL_LIB = os.path.join(BUILD, "libbsq_gemm_stall.so")


def build_gemm_stall_test_lib() -> str:
    """A test-only copy of the library whose grouped GEMM is compiled with
    BSQ_GEMM_STALL_HOOK: its producer never issues a copy and its waits give
    up after a few thousand polls, so a test can watch the bounded-wait
    timeout path end with BSQ_DEV_TIMEOUT while nothing asynchronous is in
    flight.  The other objects are the product build's."""
    build()
    src = os.path.join(CSRC, "gemm_fp4.cu")
    if os.path.exists(STALL_LIB) and os.path.getmtime(STALL_LIB) >= os.path.getmtime(LIB):
        return STALL_LIB
    cc = nvcc()
    obj = os.path.join(BUILD, "gemm_fp4_stall.o")
    r = subprocess.run([cc, *ARCH, *NVCC_FLAGS, "-DBSQ_GEMM_STALL_HOOK", "-c", src, "-o", obj],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for the stall-hook GEMM:\n{r.stdout}\n{r.stderr}")
    objs = [os.path.join(BUILD, os.path.splitext(x)[0] + ".o") for x in SOURCES if x != "gemm_fp4.cu"] + [obj]
    tmp = STALL_LIB + f".tmp{os.getpid()}"
    r = subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, STALL_LIB)
    return STALL_LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
