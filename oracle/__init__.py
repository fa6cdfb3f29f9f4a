"""CPU oracle for the fp32 matrix product and NCHW convolution (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. The product path never does: it has no CPU
fallback, and this code shares nothing with the CUDA library.

The arithmetic lives in ``om_oracle.c`` (plain C loops written from the
OneModel "Exact mode" page, sections "Matrix product" and "Convolution", and
the "Fast mode" section of the matrix-product kernels page). This module
compiles it with gcc and wraps it with ctypes and numpy.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "om_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

EXACT = 0
FAST = 1

_lock = threading.Lock()
_lib = None

# Flags that keep every float operation a single binary32 operation:
# no contraction of a*b+c, no fast-math reassociation, ISO excess-precision rules.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
          "-fexcess-precision=standard", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile ``om_oracle.c`` into ``_build/liboracle.so`` (OpenMP if gcc has it)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            i64, fp, dp, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int
            L.oracle_selfcheck.restype = ci
            L.oracle_abi_version.restype = ci
            L.oracle_conv_out_dim.restype = i64
            L.oracle_conv_out_dim.argtypes = [i64] * 6
            L.oracle_gemm_f32.restype = None
            L.oracle_gemm_f32.argtypes = [i64, i64, i64, fp, i64, fp, i64, fp, i64, ci, ci]
            L.oracle_gemm_f64.restype = None
            L.oracle_gemm_f64.argtypes = [i64, i64, i64, fp, i64, fp, i64, dp, dp, i64, ci]
            L.oracle_conv2d_f32.restype = None
            L.oracle_conv2d_f32.argtypes = [i64] * 16 + [fp, fp, fp, ci, ci]
            L.oracle_conv2d_f64.restype = None
            L.oracle_conv2d_f64.argtypes = [i64] * 16 + [fp, fp, dp, dp, ci]
            L.oracle_epilogue_f32.restype = None
            L.oracle_epilogue_f32.argtypes = [i64, i64, i64, fp, fp, fp, ci]
            rc = L.oracle_selfcheck()
            if rc != 0:
                raise RuntimeError(f"oracle self-check failed with code {rc}: host float "
                                   "arithmetic is not plain binary32 RNE with subnormals")
            _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def gemm_raw(m, n, k, A, lda, B, ldb, C, ldc, mode, threads=1):
    """C[:m, :n] (row stride ldc) = A * B on flat or 2-D float32 buffers."""
    for arr in (A, B, C):
        assert arr.dtype == np.float32 and arr.flags.c_contiguous
    lib().oracle_gemm_f32(m, n, k, _ptr(A), lda, _ptr(B), ldb, _ptr(C), ldc, int(mode), int(threads))
    return C


def gemm(A: np.ndarray, B: np.ndarray, mode: int = EXACT, threads: int = 1) -> np.ndarray:
    A = np.ascontiguousarray(A, dtype=np.float32)
    B = np.ascontiguousarray(B, dtype=np.float32)
    m, k = A.shape
    k2, n = B.shape
    assert k == k2
    C = np.zeros((m, n), dtype=np.float32)
    if m and n:
        gemm_raw(m, n, k, A if A.size else np.zeros(1, np.float32), max(k, 1),
                 B if B.size else np.zeros(1, np.float32), max(n, 1), C, n, mode, threads)
    return C


def gemm_f64(A: np.ndarray, B: np.ndarray, threads: int = 1):
    """(sum a*b, sum |a*b|) per output in binary64, for error bounds."""
    A = np.ascontiguousarray(A, dtype=np.float32)
    B = np.ascontiguousarray(B, dtype=np.float32)
    m, k = A.shape
    n = B.shape[1]
    ref = np.zeros((m, n), np.float64)
    mag = np.zeros((m, n), np.float64)
    if m and n and k:
        lib().oracle_gemm_f64(m, n, k, _ptr(A), k, _ptr(B), n, _ptr(ref), _ptr(mag), n, threads)
    return ref, mag


def conv_out_dim(size, ksize, stride, pad_before, pad_after, dil) -> int:
    return int(lib().oracle_conv_out_dim(size, ksize, stride, pad_before, pad_after, dil))


def _conv_args(x, w, stride, pad, dil, groups):
    N, Cin, H, W = x.shape
    Cout, cg, KH, KW = w.shape
    sH, sW = (stride, stride) if np.isscalar(stride) else stride
    dH, dW = (dil, dil) if np.isscalar(dil) else dil
    if np.isscalar(pad):
        pT = pL = pB = pR = pad
    else:
        pT, pL, pB, pR = pad
    assert Cin == cg * groups and Cout % groups == 0
    OH = conv_out_dim(H, KH, sH, pT, pB, dH)
    OW = conv_out_dim(W, KW, sW, pL, pR, dW)
    return (N, Cin, H, W, Cout, groups, KH, KW, sH, sW, pT, pL, pB, pR, dH, dW), (N, Cout, OH, OW)


def conv2d(x: np.ndarray, w: np.ndarray, stride=1, pad=0, dil=1, groups: int = 1,
           mode: int = EXACT, threads: int = 1) -> np.ndarray:
    """NCHW convolution; ``pad`` is a scalar or (top, left, bottom, right)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    args, yshape = _conv_args(x, w, stride, pad, dil, groups)
    y = np.zeros(yshape, dtype=np.float32)
    if y.size:
        xb = x if x.size else np.zeros(1, np.float32)
        wb = w if w.size else np.zeros(1, np.float32)
        lib().oracle_conv2d_f32(*args, _ptr(xb), _ptr(wb), _ptr(y), int(mode), int(threads))
    return y


def conv2d_f64(x, w, stride=1, pad=0, dil=1, groups=1, threads=1):
    x = np.ascontiguousarray(x, dtype=np.float32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    args, yshape = _conv_args(x, w, stride, pad, dil, groups)
    ref = np.zeros(yshape, np.float64)
    mag = np.zeros(yshape, np.float64)
    if ref.size and x.size and w.size:
        lib().oracle_conv2d_f64(*args, _ptr(x), _ptr(w), _ptr(ref), _ptr(mag), threads)
    return ref, mag


RELU = 1


def epilogue(y: np.ndarray, bias=None, res=None, activation: int = 0, channel_axis: int = 1):
    """Bias (per channel_axis index), then residual, then activation, on a copy
    of y (a product's output with channel_axis=1 for per-column bias of a 2-D
    matrix, or a convolution's NCHW output with channel_axis=1)."""
    y = np.ascontiguousarray(y, dtype=np.float32).copy()
    if y.size == 0:
        return y
    channels = y.shape[channel_axis]
    plane = int(np.prod(y.shape[channel_axis + 1:])) if y.ndim > channel_axis + 1 else 1
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    r = None if res is None else np.ascontiguousarray(res, dtype=np.float32)
    lib().oracle_epilogue_f32(y.size, plane, channels, _ptr(y), None if b is None else _ptr(b),
                              None if r is None else _ptr(r), int(activation))
    return y
