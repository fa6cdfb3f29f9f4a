"""Builds libom_gpu.so (the C-ABI CUDA library) in-tree for sm_103a with nvcc.

Each translation unit under csrc/ compiles to an object in parallel, then
nvcc links the shared library into ``_lib/``. Flags: one -gencode for
sm_103a, -lineinfo, -O3, -fmad=false (no contraction of a*b+c anywhere; the
kernels also use explicitly rounded intrinsics; the same switch is passed to
ptxas), and no -ftz / fast-math, so
subnormals are computed and every operation rounds to nearest even.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_DIR = os.path.join(HERE, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libom_gpu.so")

SOURCES = ["om_api.cu", "simple_kernels.cu", "sgemm_tiled.cu", "conv_implicit.cu", "conv_rows.cu",
           "conv_direct.cu", "gemv.cu", "gemm_tf32x3.cu", "gemm_no_alloc.cu", "selftest.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-lineinfo", "-O3", "-std=c++17", "-fmad=false", "-Xptxas", "--fmad=false",
                     "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
                     f"-I{INCLUDE}", "-Xptxas", "-v"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libom_gpu.so")


def _inputs() -> list[str]:
    files = [os.path.join(INCLUDE, "om.h"), os.path.abspath(__file__)]
    for f in os.listdir(CSRC):
        if f.endswith((".cu", ".cuh", ".h")):
            files.append(os.path.join(CSRC, f))
    return files


def _stamp() -> str:
    return " ".join(_extra_flags())


def is_stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    stamp = LIB_PATH + ".flags"
    if (open(stamp).read() if os.path.exists(stamp) else "") != _stamp():
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(f) > t for f in _inputs())


def _extra_flags() -> list[str]:
    """Extra nvcc flags for tuning builds (OM_EXTRA_NVCC_FLAGS, space separated)."""
    return os.environ.get("OM_EXTRA_NVCC_FLAGS", "").split()


def _compile(src: str) -> str:
    obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
    cmd = [nvcc(), *NVCC_FLAGS, *_extra_flags(), "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    with open(os.path.join(BUILD_DIR, src + ".ptxas.txt"), "w") as f:
        f.write(r.stderr)
    return obj


def build(force: bool = False) -> str:
    """Compile and link libom_gpu.so unless it is newer than every source."""
    if not force and not is_stale():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(_compile, SOURCES))
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    with open(LIB_PATH + ".flags", "w") as f:
        f.write(_stamp())
    return LIB_PATH
