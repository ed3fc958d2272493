"""WTConv2d as a torch autograd function / module on top of the C ABI.

A drop-in replacement for a depthwise k x k convolution ("Fast and
Memory-Efficient Wavelet Convolutions via I/O-Aware Reformulation",
arXiv 2608.10805, technical summary "Problem statement").  Forward runs
``wtconv_fwd``; backward runs ``wtconv_bwd`` (input and parameter gradients
in one fused call), or ``wtconv_bwd_data`` / ``wtconv_bwd_weight`` alone when
only one of them is needed.
"""
from __future__ import annotations

import threading
from collections import OrderedDict

import torch

from . import wtconv as _c

# Gradient workspaces, one per (device, stream, layer shape, dtype, call),
# reused across steps: the library overwrites every byte it reads, so a
# workspace needs no clearing, and reusing it spares each backward step a
# size query (a full launch plan) and an allocation.  Calls on one stream
# run in order, so sharing a workspace between them is safe.  The cache keeps
# the most recently used MAX_WORKSPACES entries, so a process that meets many
# shapes (varying batch sizes) does not grow it without bound.  Dropping an
# entry is safe while a kernel may still use it: the workspace was allocated
# on the stream it serves, and PyTorch's caching allocator hands a freed
# block only to later work on that stream.
MAX_WORKSPACES = 64
_WORKSPACES: "OrderedDict" = OrderedDict()
_WS_LOCK = threading.Lock()


def _workspace(x, levels, k, op):
    stream = torch.cuda.current_stream(x.device)
    key = (x.device, stream.cuda_stream, tuple(x.shape), x.dtype, levels, k, op)
    with _WS_LOCK:
        ws = _WORKSPACES.get(key)
        if ws is not None:
            _WORKSPACES.move_to_end(key)
    if ws is None:
        with _c._device_ctx(x.device):  # the size follows that device's occupancy
            need = _c.wtconv_workspace_size(_c.desc_for(x, levels, k), op)
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device)
        with _WS_LOCK:
            _WORKSPACES[key] = ws
            while len(_WORKSPACES) > MAX_WORKSPACES:
                _WORKSPACES.popitem(last=False)
    return ws


class WTConv2dFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, w_base, b_base, w_sub, base_scale, wavelet_scale, levels, k):
        x = x.contiguous()
        y = _c.wtconv_fwd(x, w_base, b_base, w_sub, base_scale, wavelet_scale, levels, k)
        ctx.save_for_backward(x, w_base, b_base, w_sub, base_scale, wavelet_scale)
        ctx.levels, ctx.k, ctx.has_bias = levels, k, b_base is not None
        return y

    @staticmethod
    def backward(ctx, dy):
        x, w_base, b_base, w_sub, base_scale, wavelet_scale = ctx.saved_tensors
        dy = dy.contiguous().to(x.dtype)
        b = b_base if ctx.has_bias else None
        need_dx = ctx.needs_input_grad[0]
        need_params = any(ctx.needs_input_grad[1:6])
        dx, g = None, None
        if need_dx and need_params:  # one call: the fused backward
            dx, g = _c.wtconv_bwd(x, dy, w_base, b, w_sub, base_scale, wavelet_scale, ctx.levels, ctx.k,
                                  workspace=_workspace(x, ctx.levels, ctx.k, _c.OP_BWD))
        elif need_dx:
            dx = _c.wtconv_bwd_data(dy, w_base, w_sub, base_scale, wavelet_scale, ctx.levels, ctx.k)
        elif need_params:
            g = _c.wtconv_bwd_weight(x, dy, w_base, b, w_sub, base_scale, wavelet_scale, ctx.levels, ctx.k,
                                     workspace=_workspace(x, ctx.levels, ctx.k, _c.OP_BWD_WEIGHT))
        if g is None:
            return (dx, None, None, None, None, None, None, None)
        return (dx, g["dw_base"], g["db_base"], g["dw_sub"], g["dbase_scale"], g["dwavelet_scale"],
                None, None)


class WTConv2d(torch.nn.Module):
    """Wavelet convolution on C channels with `levels` Haar levels and k x k kernels.

    Parameters (float32): weight [C,k,k] and bias [C] of the base depthwise
    conv, base_scale [C] (init 1), wavelet_weight [L,4C,k,k] (subband channel
    4c+b), wavelet_scale [L,4C] (init 0.1).
    """

    def __init__(self, channels: int, kernel_size: int = 5, levels: int = 1, bias: bool = True,
                 device=None):
        super().__init__()
        C, k, L = channels, kernel_size, levels
        # the library's limits (include/wtconv.h), checked here so that a bad
        # layer fails when it is built rather than at its first call
        if not (isinstance(k, int) and 3 <= k <= 9 and k % 2 == 1):
            raise ValueError(f"kernel_size must be odd and in [3, 9], got {k}")
        if not (isinstance(L, int) and 1 <= L <= 8):
            raise ValueError(f"levels must be in [1, 8], got {L}")
        if not (isinstance(C, int) and C >= 1):
            raise ValueError(f"channels must be a positive int, got {C}")
        f = dict(device=device, dtype=torch.float32)
        bound = 1.0 / k
        self.levels, self.k = L, k
        self.weight = torch.nn.Parameter(torch.empty(C, k, k, **f).uniform_(-bound, bound))
        self.bias = torch.nn.Parameter(torch.zeros(C, **f)) if bias else None
        self.base_scale = torch.nn.Parameter(torch.ones(C, **f))
        self.wavelet_weight = torch.nn.Parameter(torch.empty(L, 4 * C, k, k, **f).uniform_(-bound, bound))
        self.wavelet_scale = torch.nn.Parameter(torch.full((L, 4 * C), 0.1, **f))

    def extra_repr(self):
        return (f"channels={self.weight.shape[0]}, kernel_size={self.k}, levels={self.levels}, "
                f"bias={self.bias is not None}")

    def forward(self, x):
        return WTConv2dFunction.apply(x, self.weight, self.bias, self.wavelet_weight, self.base_scale,
                                      self.wavelet_scale, self.levels, self.k)
