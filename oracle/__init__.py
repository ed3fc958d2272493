"""WTConv2d CPU oracle -- TEST INFRASTRUCTURE ONLY.

A plain float64 C++ statement of the WTConv2d layer (forward and backward)
from "Fast and Memory-Efficient Wavelet Convolutions via I/O-Aware
Reformulation" (arXiv 2608.10805; technical summary on gist.science,
"Methodology").  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package.  The product path
(``memory_bound_cnn_wtconv2d_gb300``) never imports it and shares no code
with it; the only thing both sides use is the seeded input generator
``memory_bound_cnn_wtconv2d_gb300.synth``, which holds no layer arithmetic.

Functions (numpy in, float64 numpy out):

* ``fwd(inp, form)`` / ``bwd(inp, form)``: the whole layer; ``form`` is
  ``"cascade"`` (unfused stages in the pages' order, hand-written adjoints)
  or ``"direct"`` (direct block sums, the closed-form bit-indexed synthesis,
  brute-force transpose for dx; tiny shapes only).
* ``haar_analysis`` / ``haar_synthesis``: one level of the Haar pair.

Parity status: pinned (see ``tests/test_oracle_pins.py``); no function here
is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "wtconv_oracle.cpp")
_SO = os.path.join(_HERE, "liboracle.so")
_LOCK = threading.Lock()
_LIB = None

_D = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (-O2, strict IEEE float64, no -march)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.run(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-fno-fast-math",
                        "-ffp-contract=off", _SRC, "-o", tmp], check=True)
        os.replace(tmp, _SO)
    return _SO


def _lib():
    global _LIB
    with _LOCK:
        if _LIB is None:
            lib = ctypes.CDLL(build())
            i = ctypes.c_int
            fwd_args = [i, i, i, i, i, i, _D, _D, _D, _D, _D, _D, _D]
            bwd_args = [i, i, i, i, i, i, _D, _D, _D, _D, _D, _D, _D, _D, _D, _D, _D, _D, _D]
            for name in ("oracle_fwd_cascade", "oracle_fwd_direct"):
                getattr(lib, name).argtypes = fwd_args
                getattr(lib, name).restype = i
            for name in ("oracle_bwd_cascade", "oracle_bwd_direct"):
                getattr(lib, name).argtypes = bwd_args
                getattr(lib, name).restype = i
            lib.oracle_haar_analysis.argtypes = [_D, i, i, _D]
            lib.oracle_haar_analysis.restype = None
            lib.oracle_haar_synthesis.argtypes = [_D, i, i, _D, i, i]
            lib.oracle_haar_synthesis.restype = None
            _LIB = lib
        return _LIB


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def _p(a):
    return None if a is None else a.ctypes.data_as(_D)


def _params(inp):
    return [_f64(inp.w_base), _f64(inp.b_base), _f64(inp.w_sub), _f64(inp.base_scale),
            _f64(inp.wavelet_scale)]


def fwd(inp, form: str = "cascade") -> np.ndarray:
    """y[N,C,H,W] (float64) for a ``synth.LayerInputs``-like object."""
    x = _f64(inp.x)
    N, C, H, W = x.shape
    params = _params(inp)
    y = np.empty_like(x)
    fn = {"cascade": _lib().oracle_fwd_cascade, "direct": _lib().oracle_fwd_direct}[form]
    rc = fn(N, C, H, W, inp.levels, inp.k, _p(x), *[_p(a) for a in params], _p(y))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (rc={rc})")
    return y


def bwd(inp, form: str = "cascade", dy=None) -> dict:
    """dx and every parameter gradient (float64) for upstream gradient ``dy``."""
    x = _f64(inp.x)
    dy = _f64(inp.dy if dy is None else dy)
    N, C, H, W = x.shape
    L, K = inp.levels, inp.k
    params = _params(inp)
    out = dict(
        dx=np.empty_like(x),
        dw_base=np.empty((C, K, K)),
        db_base=np.empty(C) if inp.b_base is not None else None,
        dw_sub=np.empty((L, 4 * C, K, K)),
        dbase_scale=np.empty(C),
        dwavelet_scale=np.empty((L, 4 * C)),
    )
    fn = {"cascade": _lib().oracle_bwd_cascade, "direct": _lib().oracle_bwd_direct}[form]
    rc = fn(N, C, H, W, L, K, _p(x), _p(dy), *[_p(a) for a in params],
            _p(out["dx"]), _p(out["dw_base"]), _p(out["db_base"]), _p(out["dw_sub"]),
            _p(out["dbase_scale"]), _p(out["dwavelet_scale"]))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (rc={rc})")
    return out


def haar_analysis(plane: np.ndarray) -> np.ndarray:
    """One analysis level of an H x W plane -> [4, ceil(H/2), ceil(W/2)]."""
    a = _f64(plane)
    H, W = a.shape
    out = np.empty((4, (H + 1) // 2, (W + 1) // 2))
    _lib().oracle_haar_analysis(_p(a), H, W, _p(out))
    return out


def haar_synthesis(bands: np.ndarray, H: int, W: int) -> np.ndarray:
    """One synthesis level of [4, Hh, Wh] bands, cropped to H x W."""
    b = _f64(bands)
    _, Hh, Wh = b.shape
    out = np.empty((H, W))
    _lib().oracle_haar_synthesis(_p(b), Hh, Wh, _p(out), H, W)
    return out


def _slice(inp, a, b):
    """The layer problem restricted to images a..b-1 (parameters shared)."""
    import copy
    part = copy.copy(inp)
    part.N = b - a
    part.x = inp.x[a:b]
    part.dy = inp.dy[a:b]
    return part


def _bounds(N, workers):
    workers = max(1, min(int(workers), N))
    return [N * i // workers for i in range(workers + 1)]


def fwd_parallel(inp, workers: int | None = None) -> np.ndarray:
    """``fwd`` over the batch split into ``workers`` image slices, each run by
    its own thread (the C calls release the interpreter lock).  Every image is
    computed by the same code as ``fwd``; only the batch is cut."""
    import concurrent.futures
    workers = workers or os.cpu_count() or 1
    if inp.N == 0:
        return fwd(inp)
    _lib()
    b = _bounds(inp.N, workers)
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(b) - 1) as ex:
        parts = list(ex.map(lambda i: fwd(_slice(inp, b[i], b[i + 1])), range(len(b) - 1)))
    return np.concatenate(parts, axis=0)


def bwd_parallel(inp, workers: int | None = None) -> dict:
    """``bwd`` over image slices run in threads: dx is the concatenation of the
    slices' dx; each parameter gradient is a sum over the images of the batch
    (the layer's parameters are shared by every image, and the unfolded
    gradients are linear in the correlation sums), so the slices' gradients
    are added in slice order, in float64."""
    import concurrent.futures
    workers = workers or os.cpu_count() or 1
    if inp.N == 0:
        return bwd(inp)
    _lib()
    b = _bounds(inp.N, workers)
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(b) - 1) as ex:
        parts = list(ex.map(lambda i: bwd(_slice(inp, b[i], b[i + 1])), range(len(b) - 1)))
    out = {"dx": np.concatenate([p["dx"] for p in parts], axis=0)}
    for name in ("dw_base", "db_base", "dw_sub", "dbase_scale", "dwavelet_scale"):
        if parts[0][name] is None:
            out[name] = None
            continue
        acc = parts[0][name].copy()
        for p in parts[1:]:
            acc += p[name]
        out[name] = acc
    return out
