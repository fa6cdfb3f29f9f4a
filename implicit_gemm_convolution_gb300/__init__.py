"""GB300 (sm_103a) fp32 matrix product and implicit-GEMM NCHW convolution.

A thin Python binding over the C ABI of ``libom_gpu.so`` (declared in
include/om.h): it only marshals arguments. Every step of the computation
runs in the library's CUDA kernels; there is no CPU fallback, and the
functions raise if the library has not been built.

Semantics (OneModel documentation, "Exact mode" page, sections "Matrix
product" and "Convolution"; "Matrix product and convolution kernels" page,
section "Fast mode"): one accumulator per output from +0, terms in
increasing k (convolution taps in channel, kernel row, kernel column order),
NaN stored as 0x7FC00000, subnormals kept. ``mode="exact"`` rounds each
product and each sum; ``mode="fast"`` uses one fused multiply-add per term.
Both are bit-reproducible.

PyTorch is used for device memory and streams: tensors must be CUDA float32
with unit stride in the last dimension; calls run on the current stream.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

from . import _build

OM_OK = 0
STATUS_NAMES = {
    0: "OM_OK", 1: "OM_ERR_INVALID_ARG", 2: "OM_ERR_NULL_PTR", 3: "OM_ERR_ALIAS",
    4: "OM_ERR_UNSUPPORTED", 5: "OM_ERR_CUDA", 6: "OM_ERR_TIMEOUT", 7: "OM_ERR_ALIGNMENT",
    8: "OM_ERR_TOO_LARGE",
}
MODES = {"exact": 0, "fast": 1, "tf32x3": 2}
ACTIVATIONS = {None: 0, "none": 0, "relu": 1}

_lock = threading.Lock()
_lib = None


class OmError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")


def library_path() -> str:
    return _build.LIB_PATH


def build(force: bool = False) -> str:
    return _build.build(force=force)


def header_functions() -> list[str]:
    """Names of the functions include/om.h declares."""
    text = open(os.path.join(_build.INCLUDE, "om.h")).read()
    return re.findall(r"^OM_API\s+[\w\s\*]*?\b(om_\w+)\s*\(", text, flags=re.M)


def lib() -> ctypes.CDLL:
    """The loaded C library. Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_build.LIB_PATH):
                raise RuntimeError(
                    f"{_build.LIB_PATH} is missing: build the CUDA library first "
                    "(implicit_gemm_convolution_gb300.build())")
            L = ctypes.CDLL(_build.LIB_PATH)
            i64, vp, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
            L.om_version.restype = ci
            L.om_status_string.restype = ctypes.c_char_p
            L.om_status_string.argtypes = [ci]
            L.om_conv_out_dim.restype = i64
            L.om_conv_out_dim.argtypes = [i64] * 5
            L.om_gemm_f32.restype = ci
            L.om_gemm_f32.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, ci, vp]
            L.om_conv2d_f32.restype = ci
            L.om_conv2d_f32.argtypes = [i64] * 11 + [vp, vp, vp, ci, vp]
            L.om_conv2d_f32_packed.restype = ci
            L.om_conv2d_f32_packed.argtypes = [i64] * 11 + [vp, vp, vp, ci, vp]
            L.om_pack_conv_weights.restype = ci
            L.om_pack_conv_weights.argtypes = [i64] * 5 + [vp, vp, ctypes.POINTER(ctypes.c_size_t), vp]
            L.om_device_status.restype = ci
            L.om_device_status.argtypes = [vp]
            L.om_selftest_wait_timeout.argtypes = [ci, ci, vp]
            L.om_selftest_wait_timeout_ws.restype = ci
            L.om_selftest_wait_timeout_ws.argtypes = [ci, ci, vp, ctypes.c_size_t, vp]
            L.om_workspace_status.restype = ci
            L.om_workspace_status.argtypes = [vp, ctypes.c_size_t, vp]
            L.om_workspace_bytes.restype = ctypes.c_size_t
            L.om_gemm_f32_ex.restype = ci
            L.om_gemm_f32_ex.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, vp, vp, i64, ci,
                                         ci, vp, ctypes.c_size_t, vp]
            L.om_conv2d_f32_ex.restype = ci
            L.om_conv2d_f32_ex.argtypes = [i64] * 11 + [vp, vp, ci, vp, vp, ci, vp, ci, vp,
                                                        ctypes.c_size_t, vp]
            L.om_gemm_f32_ws.restype = ci
            L.om_gemm_f32_ws.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, ci, vp,
                                         ctypes.c_size_t, vp]
            L.om_conv2d_f32_ws.restype = ci
            L.om_conv2d_f32_ws.argtypes = [i64] * 11 + [vp, vp, vp, ci, vp, ctypes.c_size_t, vp]
            L.om_conv2d_f32_packed_ws.restype = ci
            L.om_conv2d_f32_packed_ws.argtypes = [i64] * 11 + [vp, vp, vp, ci, vp,
                                                  ctypes.c_size_t, vp]
            _lib = L
    return _lib


def _mode(mode) -> int:
    if isinstance(mode, str):
        if mode not in MODES:
            raise ValueError(f"unknown mode {mode!r}")
        return MODES[mode]
    return int(mode)


def _check(status: int, what: str) -> None:
    if status != OM_OK:
        raise OmError(status, what)


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) or None


def _require(t, name, ndim):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda or t.dtype != torch.float32:
        raise TypeError(f"{name} must be a CUDA float32 tensor")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions")


def conv_out_dim(size: int, ksize: int, stride: int = 1, pad: int = 0, dil: int = 1) -> int:
    v = lib().om_conv_out_dim(size, ksize, stride, pad, dil)
    if v < 0:
        raise ValueError("invalid convolution geometry")
    return int(v)


def workspace_bytes() -> int:
    """Device scratch bytes the balanced-schedule entry points need."""
    return int(lib().om_workspace_bytes())


def new_workspace(device=None):
    """A device tensor usable as the workspace of the *_ws entry points."""
    import torch
    return torch.zeros((workspace_bytes() + 3) // 4, dtype=torch.int32, device=device or "cuda")


def _ws_args(workspace):
    return workspace.data_ptr(), workspace.numel() * workspace.element_size()


def gemm_raw(m, n, k, A_ptr, lda, B_ptr, ldb, C_ptr, ldc, mode="exact", stream=None,
             workspace=None) -> int:
    """Calls om_gemm_f32 (om_gemm_f32_ws when a workspace tensor is given) on
    raw device pointers; returns the status code."""
    if workspace is None:
        return lib().om_gemm_f32(m, n, k, A_ptr, lda, B_ptr, ldb, C_ptr, ldc, _mode(mode),
                                 _stream_handle(stream))
    return lib().om_gemm_f32_ws(m, n, k, A_ptr, lda, B_ptr, ldb, C_ptr, ldc, _mode(mode),
                                *_ws_args(workspace), _stream_handle(stream))


def gemm(A, B, out=None, mode="exact", stream=None, workspace=None):
    """C = A @ B (row-major views; leading dimensions from the row strides)."""
    import torch
    _require(A, "A", 2)
    _require(B, "B", 2)
    m, k = A.shape
    k2, n = B.shape
    if k != k2:
        raise ValueError("inner dimensions differ")
    if out is None:
        out = torch.empty((m, n), dtype=torch.float32, device=A.device)
    _require(out, "out", 2)
    if tuple(out.shape) != (m, n):
        raise ValueError("out has the wrong shape")
    for t, name in ((A, "A"), (B, "B"), (out, "out")):
        if t.shape[1] > 1 and t.stride(1) != 1:
            raise ValueError(f"{name} needs unit stride along its rows")
    lda = A.stride(0) if m > 1 else max(k, 1)
    ldb = B.stride(0) if k > 1 else max(n, 1)
    ldc = out.stride(0) if m > 1 else max(n, 1)
    _check(gemm_raw(m, n, k, A.data_ptr(), lda, B.data_ptr(), ldb, out.data_ptr(), ldc, mode,
                    stream, workspace), "om_gemm_f32")
    return out


def _conv_geom(x, w_shape, stride, padding, dilation, groups):
    N, Cin, H, W = x.shape
    Cout, cg, KH, KW = w_shape
    if cg * groups != Cin:
        raise ValueError("weights do not match Cin/groups")
    OH = conv_out_dim(H, KH, stride, padding, dilation)
    OW = conv_out_dim(W, KW, stride, padding, dilation)
    return (N, Cin, H, W, Cout, groups, KH, KW, stride, padding, dilation), (N, Cout, OH, OW)


def conv2d(x, w, stride: int = 1, padding: int = 0, dilation: int = 1, groups: int = 1,
           out=None, mode="exact", stream=None, workspace=None):
    """NCHW convolution without bias (implicit GEMM on the GPU)."""
    import torch
    _require(x, "x", 4)
    _require(w, "w", 4)
    if not x.is_contiguous() or not w.is_contiguous():
        raise ValueError("x and w must be contiguous")
    args, yshape = _conv_geom(x, tuple(w.shape), stride, padding, dilation, groups)
    if out is None:
        out = torch.empty(yshape, dtype=torch.float32, device=x.device)
    _require(out, "out", 4)
    if tuple(out.shape) != yshape or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor of the output shape")
    if workspace is None:
        st = lib().om_conv2d_f32(*args, x.data_ptr(), w.data_ptr(), out.data_ptr(), _mode(mode),
                                 _stream_handle(stream))
    else:
        st = lib().om_conv2d_f32_ws(*args, x.data_ptr(), w.data_ptr(), out.data_ptr(), _mode(mode),
                                    *_ws_args(workspace), _stream_handle(stream))
    _check(st, "om_conv2d_f32")
    return out


def packed_weight_bytes(Cout, Cin, groups, KH, KW) -> int:
    size = ctypes.c_size_t(0)
    _check(lib().om_pack_conv_weights(Cout, Cin, groups, KH, KW, None, None, ctypes.byref(size),
                                      None), "om_pack_conv_weights")
    return int(size.value)


def pack_conv_weights(w, groups: int = 1, stream=None):
    """Packs [Cout, Cin/G, KH, KW] weights for conv2d_packed (a flat float32 tensor)."""
    import torch
    _require(w, "w", 4)
    if not w.is_contiguous():
        raise ValueError("w must be contiguous")
    Cout, cg, KH, KW = w.shape
    nbytes = packed_weight_bytes(Cout, cg * groups, groups, KH, KW)
    out = torch.empty(max(nbytes // 4, 4), dtype=torch.float32, device=w.device)
    size = ctypes.c_size_t(0)
    _check(lib().om_pack_conv_weights(Cout, cg * groups, groups, KH, KW, w.data_ptr(),
                                      out.data_ptr(), ctypes.byref(size), _stream_handle(stream)),
           "om_pack_conv_weights")
    return out[: nbytes // 4]


def conv2d_packed(x, w_packed, w_shape, stride: int = 1, padding: int = 0, dilation: int = 1,
                  groups: int = 1, out=None, mode="exact", stream=None, workspace=None):
    """conv2d with weights from pack_conv_weights (w_shape = the unpacked shape)."""
    import torch
    _require(x, "x", 4)
    _require(w_packed, "w_packed", 1)
    args, yshape = _conv_geom(x, tuple(w_shape), stride, padding, dilation, groups)
    if out is None:
        out = torch.empty(yshape, dtype=torch.float32, device=x.device)
    if workspace is None:
        st = lib().om_conv2d_f32_packed(*args, x.data_ptr(), w_packed.data_ptr(), out.data_ptr(),
                                        _mode(mode), _stream_handle(stream))
    else:
        st = lib().om_conv2d_f32_packed_ws(*args, x.data_ptr(), w_packed.data_ptr(),
                                           out.data_ptr(), _mode(mode), *_ws_args(workspace),
                                           _stream_handle(stream))
    _check(st, "om_conv2d_f32_packed")
    return out


def device_status(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device-wide status
    words (timeouts of calls made without a workspace)."""
    return int(lib().om_device_status(_stream_handle(stream)))


def workspace_status(workspace, stream=None) -> int:
    """Synchronises the stream and returns (and clears) the status word of a
    workspace: timeouts of the calls that were given this workspace."""
    return int(lib().om_workspace_status(*_ws_args(workspace), _stream_handle(stream)))


def _ptr_or_none(t):
    return None if t is None else t.data_ptr()


def gemm_ex(A, B, bias=None, residual=None, activation=None, out=None, mode="exact",
            stream=None, workspace=None):
    """act(A @ B + bias + residual): bias per column (n,), residual (m, n)."""
    import torch
    _require(A, "A", 2)
    _require(B, "B", 2)
    m, k = A.shape
    n = B.shape[1]
    if out is None:
        out = torch.empty((m, n), dtype=torch.float32, device=A.device)
    if bias is not None:
        _require(bias, "bias", 1)
    if residual is not None:
        _require(residual, "residual", 2)
    lda = A.stride(0) if m > 1 else max(k, 1)
    ldb = B.stride(0) if k > 1 else max(n, 1)
    ldc = out.stride(0) if m > 1 else max(n, 1)
    ldr = (residual.stride(0) if m > 1 else max(n, 1)) if residual is not None else 0
    ws = (None, 0) if workspace is None else _ws_args(workspace)
    _check(lib().om_gemm_f32_ex(m, n, k, A.data_ptr(), lda, B.data_ptr(), ldb, out.data_ptr(), ldc,
                                _ptr_or_none(bias), _ptr_or_none(residual), ldr,
                                ACTIVATIONS[activation], _mode(mode), ws[0], ws[1],
                                _stream_handle(stream)), "om_gemm_f32_ex")
    return out


def conv2d_ex(x, w, stride: int = 1, padding: int = 0, dilation: int = 1, groups: int = 1,
              bias=None, residual=None, activation=None, out=None, mode="exact", stream=None,
              workspace=None, w_packed=None):
    """act(conv2d(x, w) + bias[oc] + residual), NCHW. With w_packed given, w is
    only used for its shape."""
    import torch
    _require(x, "x", 4)
    args, yshape = _conv_geom(x, tuple(w.shape), stride, padding, dilation, groups)
    if out is None:
        out = torch.empty(yshape, dtype=torch.float32, device=x.device)
    wsrc = w if w_packed is None else w_packed
    ws = (None, 0) if workspace is None else _ws_args(workspace)
    _check(lib().om_conv2d_f32_ex(*args, x.data_ptr(), wsrc.data_ptr(), int(w_packed is not None),
                                  _ptr_or_none(bias), _ptr_or_none(residual),
                                  ACTIVATIONS[activation], out.data_ptr(), _mode(mode), ws[0],
                                  ws[1], _stream_handle(stream)), "om_conv2d_f32_ex")
    return out
