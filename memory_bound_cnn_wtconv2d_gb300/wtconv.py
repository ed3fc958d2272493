"""Thin ctypes binding of libwtconv.so (include/wtconv.h).

Argument marshalling only: every step of the layer runs in the library's
CUDA kernels.  The functions keep the C names (``wtconv_fwd``,
``wtconv_bwd_data``, ``wtconv_bwd_weight``, ``wtconv_workspace_size``) and
take torch CUDA tensors; tensors are only used as device memory, and the
work is enqueued on the current torch stream unless ``stream`` is given.
If the library is missing this module raises instead of falling back.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libwtconv.so")

WTCONV_OK, WTCONV_ERR_INVALID_ARG, WTCONV_ERR_UNSUPPORTED = 0, 1, 2
WTCONV_ERR_MISALIGNED, WTCONV_ERR_WORKSPACE, WTCONV_ERR_CUDA = 3, 4, 5
OP_FWD, OP_BWD_DATA, OP_BWD_WEIGHT, OP_BWD = 0, 1, 2, 3
DTYPE_CODES = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}

# entry points declared in include/wtconv.h
EXPORTS = ("wtconv_workspace_size", "wtconv_fwd", "wtconv_bwd_data", "wtconv_bwd_weight", "wtconv_bwd",
           "wtconv_bwd_weight_noalloc", "wtconv_status_string", "wtconv_last_error",
           "wtconv_device_faults")


class WtconvDesc(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int), ("C", ctypes.c_int), ("H", ctypes.c_int), ("W", ctypes.c_int),
                ("levels", ctypes.c_int), ("k", ctypes.c_int), ("dtype", ctypes.c_int)]


class WtconvError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


_LIB = None


def lib() -> ctypes.CDLL:
    """Load libwtconv.so (built in-tree by ``build.build()``)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        vp, sz = ctypes.c_void_p, ctypes.c_size_t
        dp = ctypes.POINTER(WtconvDesc)
        L.wtconv_workspace_size.argtypes = [dp, ctypes.c_int]
        L.wtconv_workspace_size.restype = sz
        L.wtconv_fwd.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.wtconv_fwd.restype = ctypes.c_int
        L.wtconv_bwd_data.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.wtconv_bwd_data.restype = ctypes.c_int
        L.wtconv_bwd_weight.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.wtconv_bwd_weight.restype = ctypes.c_int
        L.wtconv_bwd.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.wtconv_bwd.restype = ctypes.c_int
        L.wtconv_bwd_weight_noalloc.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.wtconv_bwd_weight_noalloc.restype = ctypes.c_int
        L.wtconv_status_string.argtypes = [ctypes.c_int]
        L.wtconv_status_string.restype = ctypes.c_char_p
        L.wtconv_last_error.argtypes = []
        L.wtconv_last_error.restype = ctypes.c_char_p
        L.wtconv_device_faults.argtypes = []
        L.wtconv_device_faults.restype = ctypes.c_uint
        _LIB = L
    return _LIB


def _check(status: int):
    if status != WTCONV_OK:
        L = lib()
        name = L.wtconv_status_string(status).decode()
        raise WtconvError(status, f"{name}: {L.wtconv_last_error().decode()}")


def make_desc(N, C, H, W, levels, k, dtype) -> WtconvDesc:
    code = DTYPE_CODES[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return WtconvDesc(int(N), int(C), int(H), int(W), int(levels), int(k), code)


def desc_for(x: torch.Tensor, levels: int, k: int) -> WtconvDesc:
    if x.dim() != 4:
        raise ValueError("activations must be NCHW")
    return make_desc(*x.shape, levels, k, x.dtype)


def wtconv_workspace_size(desc: WtconvDesc, op: int) -> int:
    return int(lib().wtconv_workspace_size(ctypes.byref(desc), int(op)))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _act(t, name):
    if not (t.is_cuda and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    return t


def _param(t, name, optional=False):
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    if not (t.is_cuda and t.is_contiguous() and t.dtype == torch.float32):
        raise ValueError(f"{name} must be a contiguous float32 CUDA tensor")
    return t


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def wtconv_fwd(x, w_base, b_base, w_sub, base_scale, wavelet_scale, levels, k, y=None, stream=None):
    """y = WTConv2d(x)."""
    _act(x, "x")
    desc = desc_for(x, levels, k)
    y = torch.empty_like(x) if y is None else _act(y, "y")
    _check(lib().wtconv_fwd(ctypes.byref(desc), _ptr(x), _ptr(_param(w_base, "w_base")),
                            _ptr(_param(b_base, "b_base", True)), _ptr(_param(w_sub, "w_sub")),
                            _ptr(_param(base_scale, "base_scale")),
                            _ptr(_param(wavelet_scale, "wavelet_scale")), _ptr(y), None, 0, _stream(stream)))
    return y


def wtconv_bwd_data(dy, w_base, w_sub, base_scale, wavelet_scale, levels, k, dx=None, stream=None):
    """dx = dL/dx for upstream gradient dy."""
    _act(dy, "dy")
    desc = desc_for(dy, levels, k)
    dx = torch.empty_like(dy) if dx is None else _act(dx, "dx")
    _check(lib().wtconv_bwd_data(ctypes.byref(desc), _ptr(dy), _ptr(_param(w_base, "w_base")),
                                 _ptr(_param(w_sub, "w_sub")), _ptr(_param(base_scale, "base_scale")),
                                 _ptr(_param(wavelet_scale, "wavelet_scale")), _ptr(dx), None, 0,
                                 _stream(stream)))
    return dx


def wtconv_bwd_weight(x, dy, w_base, b_base, w_sub, base_scale, wavelet_scale, levels, k,
                      grads=None, workspace=None, stream=None):
    """Parameter gradients as a dict: dw_base, db_base (None without bias), dw_sub,
    dbase_scale, dwavelet_scale (float32, overwritten)."""
    _act(x, "x")
    _act(dy, "dy")
    desc = desc_for(x, levels, k)
    dev = x.device
    if grads is None:
        grads = dict(dw_base=torch.empty_like(w_base),
                     db_base=None if b_base is None else torch.empty_like(b_base),
                     dw_sub=torch.empty_like(w_sub), dbase_scale=torch.empty_like(base_scale),
                     dwavelet_scale=torch.empty_like(wavelet_scale))
    if workspace is None:  # a caller-provided workspace is checked by the library itself
        need = wtconv_workspace_size(desc, OP_BWD_WEIGHT)
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _check(lib().wtconv_bwd_weight(
        ctypes.byref(desc), _ptr(x), _ptr(dy), _ptr(_param(w_base, "w_base")),
        _ptr(_param(b_base, "b_base", True)), _ptr(_param(w_sub, "w_sub")),
        _ptr(_param(base_scale, "base_scale")), _ptr(_param(wavelet_scale, "wavelet_scale")),
        _ptr(grads["dw_base"]), _ptr(grads["db_base"]), _ptr(grads["dw_sub"]), _ptr(grads["dbase_scale"]),
        _ptr(grads["dwavelet_scale"]), _ptr(workspace), workspace.numel(), _stream(stream)))
    return grads


def wtconv_bwd(x, dy, w_base, b_base, w_sub, base_scale, wavelet_scale, levels, k,
               dx=None, grads=None, workspace=None, stream=None):
    """The whole backward in one call (one kernel over x and dy where the planes
    fit): returns (dx, grads) with grads as from wtconv_bwd_weight."""
    _act(x, "x")
    _act(dy, "dy")
    desc = desc_for(x, levels, k)
    dev = x.device
    dx = torch.empty_like(dy) if dx is None else _act(dx, "dx")
    if grads is None:
        grads = dict(dw_base=torch.empty_like(w_base),
                     db_base=None if b_base is None else torch.empty_like(b_base),
                     dw_sub=torch.empty_like(w_sub), dbase_scale=torch.empty_like(base_scale),
                     dwavelet_scale=torch.empty_like(wavelet_scale))
    if workspace is None:  # a caller-provided workspace is checked by the library itself
        need = wtconv_workspace_size(desc, OP_BWD)
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _check(lib().wtconv_bwd(
        ctypes.byref(desc), _ptr(x), _ptr(dy), _ptr(_param(w_base, "w_base")),
        _ptr(_param(b_base, "b_base", True)), _ptr(_param(w_sub, "w_sub")),
        _ptr(_param(base_scale, "base_scale")), _ptr(_param(wavelet_scale, "wavelet_scale")), _ptr(dx),
        _ptr(grads["dw_base"]), _ptr(grads["db_base"]), _ptr(grads["dw_sub"]), _ptr(grads["dbase_scale"]),
        _ptr(grads["dwavelet_scale"]), _ptr(workspace), workspace.numel(), _stream(stream)))
    return dx, grads


def wtconv_bwd_weight_noalloc(x, dy, w_base, b_base, w_sub, base_scale, wavelet_scale, levels, k,
                              grads=None, stream=None):
    """Parameter gradients through the entry point that allocates nothing: the
    library's built-in 4 MiB device scratch replaces the workspace.  For callers
    that cannot allocate device memory; concurrent calls race on the scratch."""
    _act(x, "x")
    _act(dy, "dy")
    desc = desc_for(x, levels, k)
    if grads is None:
        grads = dict(dw_base=torch.empty_like(w_base),
                     db_base=None if b_base is None else torch.empty_like(b_base),
                     dw_sub=torch.empty_like(w_sub), dbase_scale=torch.empty_like(base_scale),
                     dwavelet_scale=torch.empty_like(wavelet_scale))
    _check(lib().wtconv_bwd_weight_noalloc(
        ctypes.byref(desc), _ptr(x), _ptr(dy), _ptr(_param(w_base, "w_base")),
        _ptr(_param(b_base, "b_base", True)), _ptr(_param(w_sub, "w_sub")),
        _ptr(_param(base_scale, "base_scale")), _ptr(_param(wavelet_scale, "wavelet_scale")),
        _ptr(grads["dw_base"]), _ptr(grads["db_base"]), _ptr(grads["dw_sub"]), _ptr(grads["dbase_scale"]),
        _ptr(grads["dwavelet_scale"]), _stream(stream)))
    return grads


def wtconv_device_faults() -> int:
    """In-kernel bounded waits that gave up since the previous call (0 in
    normal operation); synchronises the device and resets the count."""
    return int(lib().wtconv_device_faults())
