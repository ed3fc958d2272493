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
PARAM_NAMES = ("w_base", "b_base", "w_sub", "base_scale", "wavelet_scale")
GRAD_NAMES = ("dw_base", "db_base", "dw_sub", "dbase_scale", "dwavelet_scale")

# entry points declared in include/wtconv.h
EXPORTS = ("wtconv_workspace_size", "wtconv_fwd", "wtconv_bwd_data", "wtconv_bwd_weight", "wtconv_bwd",
           "wtconv_bwd_weight_noalloc", "wtconv_status_string", "wtconv_last_error",
           "wtconv_device_faults", "wtconv_test_copy_timeout")


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
        L.wtconv_test_copy_timeout.argtypes = [ctypes.c_int]
        L.wtconv_test_copy_timeout.restype = None
        _LIB = L
    return _LIB


def _check(status: int):
    if status != WTCONV_OK:
        L = lib()
        name = L.wtconv_status_string(status).decode()
        raise WtconvError(status, f"{name}: {L.wtconv_last_error().decode()}")


def make_desc(N, C, H, W, levels, k, dtype) -> WtconvDesc:
    if isinstance(dtype, torch.dtype) and dtype not in DTYPE_CODES:
        raise ValueError(f"activations must be float32, float16 or bfloat16, got {dtype}")
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


# The library sees plain pointers, so every size it relies on is checked
# here: a tensor smaller than the layer implies would be read or written past
# its end by the kernels.  Outputs must not overlap inputs or each other
# (include/wtconv.h, "Aliasing"), which is checked here too.


def _on_cuda(t):
    return t.is_cuda


def _act(t, name, like=None):
    """An activation: contiguous CUDA; `like` (x) fixes shape, dtype and device."""
    if not (isinstance(t, torch.Tensor) and _on_cuda(t) and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if like is not None and (t.shape != like.shape or t.dtype != like.dtype or t.device != like.device):
        raise ValueError(f"{name} must be {tuple(like.shape)} {like.dtype} on {like.device}, "
                         f"got {tuple(t.shape)} {t.dtype} on {t.device}")
    return t


def _param(t, name, numel, device, optional=False):
    """A parameter or gradient: contiguous float32 on `device` with `numel`
    elements (any shape: [C,k,k] and the depthwise [C,1,k,k] both work)."""
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    if not (isinstance(t, torch.Tensor) and _on_cuda(t) and t.is_contiguous() and t.dtype == torch.float32):
        raise ValueError(f"{name} must be a contiguous float32 CUDA tensor")
    if t.device != device or t.numel() != numel:
        raise ValueError(f"{name} must hold {numel} elements on {device}, got {t.numel()} on {t.device}")
    return t


def _param_sizes(x, levels, k):
    """Element counts of w_base, b_base, w_sub, base_scale, wavelet_scale."""
    C, L, kk = x.shape[1], int(levels), int(k) * int(k)
    return C * kk, C, L * 4 * C * kk, C, L * 4 * C


def _params(x, levels, k, w_base, b_base, w_sub, base_scale, wavelet_scale):
    n = _param_sizes(x, levels, k)
    d = x.device
    return (_param(w_base, "w_base", n[0], d), _param(b_base, "b_base", n[1], d, True),
            _param(w_sub, "w_sub", n[2], d), _param(base_scale, "base_scale", n[3], d),
            _param(wavelet_scale, "wavelet_scale", n[4], d))


def _grads(grads, params):
    """The caller's gradient buffers (checked), or new ones shaped like the
    parameters.  Without a bias db_base may be absent or None; a db_base that
    is given still receives the gradient a bias would have (s_base * sum dy)."""
    if grads is None:
        return {n: None if p is None else torch.empty_like(p) for n, p in zip(GRAD_NAMES, params)}
    C = params[3].numel()
    for n, p in zip(GRAD_NAMES, params):
        if p is not None:
            _param(grads.get(n), n, p.numel(), p.device)
        elif grads.get(n) is not None:
            _param(grads[n], n, C, params[0].device)
    return grads if "db_base" in grads else dict(grads, db_base=None)


def _workspace_bytes(ws, device):
    if not (isinstance(ws, torch.Tensor) and _on_cuda(ws) and ws.is_contiguous() and ws.device == device):
        raise ValueError(f"workspace must be a contiguous CUDA tensor on {device}")
    return ws.numel() * ws.element_size()


def _disjoint(outs, ins):
    """Raise if an output's memory overlaps an input's or another output's.
    outs, ins: (name, tensor or None) pairs."""
    def span(t):
        p = t.data_ptr()
        return p, p + t.numel() * t.element_size()
    o = [(n, span(t)) for n, t in outs if t is not None and t.numel()]
    every = o + [(n, span(t)) for n, t in ins if t is not None and t.numel()]
    for i, (n, (a0, a1)) in enumerate(o):
        for m, (b0, b1) in every[i + 1:]:
            if a0 < b1 and b0 < a1:
                raise ValueError(f"{n} overlaps {m}: outputs may not share memory with inputs or other outputs")


def _stream(stream, device):
    """The stream handle for a call on `device`: the given stream, else that
    device's current torch stream."""
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _device_ctx(device):
    """Makes `device` the current CUDA device for the duration of a call: the
    library launches on the current device and picks per-device state (plan
    caches, the no-alloc scratch) by it, so it must be the device that holds
    the tensors."""
    return torch.cuda.device(device)


# Workspace bytes of the forward and input-gradient passes, per (layer,
# pass): nonzero only for layers computed as a fine pass plus a coarse layer
# (include/wtconv.h, "Limits"); the size does not depend on the device.
_FWD_WS = {}


def _fwd_workspace(desc, op, device, workspace):
    """The workspace a forward / input-gradient call needs and its size in
    bytes: the caller's, else a new one when the layer needs any, else
    (None, 0).  The caller keeps the tensor alive until the call is enqueued."""
    if workspace is not None:
        return workspace, _workspace_bytes(workspace, device)
    key = (desc.N, desc.C, desc.H, desc.W, desc.levels, desc.k, desc.dtype, op)
    need = _FWD_WS.get(key)
    if need is None:
        need = _FWD_WS[key] = wtconv_workspace_size(desc, op)
    if need == 0:
        return None, 0
    return torch.empty(need, dtype=torch.uint8, device=device), need


def wtconv_fwd(x, w_base, b_base, w_sub, base_scale, wavelet_scale, levels, k, y=None, stream=None,
               workspace=None):
    """y = WTConv2d(x)."""
    _act(x, "x")
    desc = desc_for(x, levels, k)
    ps = _params(x, levels, k, w_base, b_base, w_sub, base_scale, wavelet_scale)
    y = torch.empty_like(x) if y is None else _act(y, "y", like=x)
    outs = [("y", y)] + ([("workspace", workspace)] if workspace is not None else [])
    _disjoint(outs, [("x", x), *zip(PARAM_NAMES, ps)])
    with _device_ctx(x.device):
        wt, wn = _fwd_workspace(desc, OP_FWD, x.device, workspace)
        _check(lib().wtconv_fwd(ctypes.byref(desc), _ptr(x), *map(_ptr, ps), _ptr(y), _ptr(wt), wn,
                                _stream(stream, x.device)))
    return y


def wtconv_bwd_data(dy, w_base, w_sub, base_scale, wavelet_scale, levels, k, dx=None, stream=None,
                    workspace=None):
    """dx = dL/dx for upstream gradient dy."""
    _act(dy, "dy")
    desc = desc_for(dy, levels, k)
    wb, _, ws_, sb, sw = _params(dy, levels, k, w_base, None, w_sub, base_scale, wavelet_scale)
    dx = torch.empty_like(dy) if dx is None else _act(dx, "dx", like=dy)
    outs = [("dx", dx)] + ([("workspace", workspace)] if workspace is not None else [])
    _disjoint(outs, [("dy", dy), ("w_base", wb), ("w_sub", ws_), ("base_scale", sb), ("wavelet_scale", sw)])
    with _device_ctx(dy.device):
        wt, wn = _fwd_workspace(desc, OP_BWD_DATA, dy.device, workspace)
        _check(lib().wtconv_bwd_data(ctypes.byref(desc), _ptr(dy), _ptr(wb), _ptr(ws_), _ptr(sb), _ptr(sw), _ptr(dx),
                                     _ptr(wt), wn, _stream(stream, dy.device)))
    return dx


def wtconv_bwd_weight(x, dy, w_base, b_base, w_sub, base_scale, wavelet_scale, levels, k,
                      grads=None, workspace=None, stream=None):
    """Parameter gradients as a dict: dw_base, db_base (None without bias), dw_sub,
    dbase_scale, dwavelet_scale (float32, overwritten)."""
    _act(x, "x")
    _act(dy, "dy", like=x)
    desc = desc_for(x, levels, k)
    ps = _params(x, levels, k, w_base, b_base, w_sub, base_scale, wavelet_scale)
    grads = _grads(grads, ps)
    if workspace is None:  # a caller-provided workspace's size is checked by the library itself
        with _device_ctx(x.device):  # the size follows the device's occupancy
            need = wtconv_workspace_size(desc, OP_BWD_WEIGHT)
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device)
    ws_bytes = _workspace_bytes(workspace, x.device)
    _disjoint([*((n, grads.get(n)) for n in GRAD_NAMES), ("workspace", workspace)],
              [("x", x), ("dy", dy), *zip(PARAM_NAMES, ps)])
    with _device_ctx(x.device):
        _check(lib().wtconv_bwd_weight(
            ctypes.byref(desc), _ptr(x), _ptr(dy), *map(_ptr, ps),
            _ptr(grads["dw_base"]), _ptr(grads["db_base"]), _ptr(grads["dw_sub"]), _ptr(grads["dbase_scale"]),
            _ptr(grads["dwavelet_scale"]), _ptr(workspace), ws_bytes, _stream(stream, x.device)))
    return grads


def wtconv_bwd(x, dy, w_base, b_base, w_sub, base_scale, wavelet_scale, levels, k,
               dx=None, grads=None, workspace=None, stream=None):
    """The whole backward in one call (one kernel over x and dy where the planes
    fit): returns (dx, grads) with grads as from wtconv_bwd_weight."""
    _act(x, "x")
    _act(dy, "dy", like=x)
    desc = desc_for(x, levels, k)
    ps = _params(x, levels, k, w_base, b_base, w_sub, base_scale, wavelet_scale)
    dx = torch.empty_like(dy) if dx is None else _act(dx, "dx", like=x)
    grads = _grads(grads, ps)
    if workspace is None:  # a caller-provided workspace's size is checked by the library itself
        with _device_ctx(x.device):  # the size follows the device's occupancy
            need = wtconv_workspace_size(desc, OP_BWD)
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device)
    ws_bytes = _workspace_bytes(workspace, x.device)
    _disjoint([("dx", dx), *((n, grads.get(n)) for n in GRAD_NAMES), ("workspace", workspace)],
              [("x", x), ("dy", dy), *zip(PARAM_NAMES, ps)])
    with _device_ctx(x.device):
        _check(lib().wtconv_bwd(
            ctypes.byref(desc), _ptr(x), _ptr(dy), *map(_ptr, ps), _ptr(dx),
            _ptr(grads["dw_base"]), _ptr(grads["db_base"]), _ptr(grads["dw_sub"]), _ptr(grads["dbase_scale"]),
            _ptr(grads["dwavelet_scale"]), _ptr(workspace), ws_bytes, _stream(stream, x.device)))
    return dx, grads


def wtconv_bwd_weight_noalloc(x, dy, w_base, b_base, w_sub, base_scale, wavelet_scale, levels, k,
                              grads=None, stream=None):
    """Parameter gradients through the entry point that allocates nothing: the
    library's built-in 4 MiB device scratch replaces the workspace.  For callers
    that cannot allocate device memory; concurrent calls race on the scratch."""
    _act(x, "x")
    _act(dy, "dy", like=x)
    desc = desc_for(x, levels, k)
    ps = _params(x, levels, k, w_base, b_base, w_sub, base_scale, wavelet_scale)
    grads = _grads(grads, ps)
    _disjoint([(n, grads.get(n)) for n in GRAD_NAMES], [("x", x), ("dy", dy), *zip(PARAM_NAMES, ps)])
    with _device_ctx(x.device):
        _check(lib().wtconv_bwd_weight_noalloc(
            ctypes.byref(desc), _ptr(x), _ptr(dy), *map(_ptr, ps),
            _ptr(grads["dw_base"]), _ptr(grads["db_base"]), _ptr(grads["dw_sub"]), _ptr(grads["dbase_scale"]),
            _ptr(grads["dwavelet_scale"]), _stream(stream, x.device)))
    return grads


def wtconv_device_faults() -> int:
    """In-kernel bounded waits that gave up since the previous call (0 in
    normal operation); synchronises the device and resets the count."""
    return int(lib().wtconv_device_faults())


def wtconv_test_copy_timeout(enable: bool) -> None:
    """Test support: while on, the kernels' bounded waits for their plane copies
    run out on purpose (see include/wtconv.h); off restores normal operation."""
    lib().wtconv_test_copy_timeout(1 if enable else 0)
