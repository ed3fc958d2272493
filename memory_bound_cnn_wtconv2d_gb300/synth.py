"""Seeded synthetic inputs for the WTConv2d layer.

This module draws random numbers and nothing else: it holds none of the
layer's arithmetic, so both the CUDA path and the CPU oracle may use it.

Distributions (the workloads of "Fast and Memory-Efficient Wavelet
Convolutions via I/O-Aware Reformulation", arXiv 2608.10805, restated as
synthetic draws; the pages measure on WTConvNeXt layer shapes, which these
stand in for):

* activations ``x`` and upstream gradient ``dy``: N(0, 1);
* base weight ``w_base[C,k,k]``, subband weights ``w_sub[L,4C,k,k]`` and
  base bias ``b_base[C]``: N(0, 0.05^2) (standard deviation 0.05);
* ``base_scale[C]`` = 1 + U(-0.1, 0.1);
* ``wavelet_scale[L,4C]`` = 0.1 + U(-0.05, 0.05).

Values are drawn in float64 with numpy's PCG64 generator (bit-identical on
x86 and Arm), then rounded once to the storage type.  Every returned array is
float32 whose values are exactly representable in the storage dtype, so the
device copy (``torch.tensor(..., dtype)``) and the oracle's float64 view hold
the same numbers.
"""
from __future__ import annotations

import dataclasses

import numpy as np

DTYPES = ("f32", "f16", "bf16")


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns float32."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    bits = a.view(np.uint32).astype(np.uint64)
    lsb = (bits >> np.uint64(16)) & np.uint64(1)
    rounded = (bits + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)
    out = rounded.astype(np.uint32).view(np.float32)
    # keep NaN/Inf as they were (never drawn here, but stay safe)
    return np.where(np.isfinite(a), out, a).astype(np.float32)


def quantize(a: np.ndarray, dtype: str) -> np.ndarray:
    """Round to the storage dtype and return the values as float32."""
    if dtype == "f32":
        return a.astype(np.float32)
    if dtype == "f16":
        return a.astype(np.float16).astype(np.float32)
    if dtype == "bf16":
        return round_to_bf16(a.astype(np.float32))
    raise ValueError(f"unknown dtype {dtype!r}")


@dataclasses.dataclass
class LayerInputs:
    """One synthetic WTConv2d problem (host arrays, float32 values)."""

    N: int
    C: int
    H: int
    W: int
    levels: int
    k: int
    dtype: str
    x: np.ndarray            # [N,C,H,W], values exact in `dtype`
    dy: np.ndarray           # [N,C,H,W], values exact in `dtype`
    w_base: np.ndarray       # [C,k,k]
    b_base: np.ndarray | None  # [C] or None
    w_sub: np.ndarray        # [L,4C,k,k], subband channel 4c+b
    base_scale: np.ndarray   # [C]
    wavelet_scale: np.ndarray  # [L,4C]

    @property
    def numel(self) -> int:
        return self.N * self.C * self.H * self.W


def make_inputs(N: int, C: int, H: int, W: int, levels: int, k: int,
                dtype: str = "f32", seed: int = 0, bias: bool = True,
                weight_std: float = 0.05) -> LayerInputs:
    if dtype not in DTYPES:
        raise ValueError(f"dtype must be one of {DTYPES}")
    rng = np.random.Generator(np.random.PCG64(seed))
    L = levels
    # parameters first, so that their values do not depend on the activation size
    w_base = rng.standard_normal((C, k, k)) * weight_std
    b_base = rng.standard_normal(C) * weight_std
    w_sub = rng.standard_normal((L, 4 * C, k, k)) * weight_std
    base_scale = 1.0 + rng.uniform(-0.1, 0.1, size=C)
    wavelet_scale = 0.1 + rng.uniform(-0.05, 0.05, size=(L, 4 * C))
    x = rng.standard_normal((N, C, H, W))
    dy = rng.standard_normal((N, C, H, W))
    return LayerInputs(
        N=N, C=C, H=H, W=W, levels=L, k=k, dtype=dtype,
        x=quantize(x, dtype), dy=quantize(dy, dtype),
        w_base=w_base.astype(np.float32),
        b_base=b_base.astype(np.float32) if bias else None,
        w_sub=w_sub.astype(np.float32),
        base_scale=base_scale.astype(np.float32),
        wavelet_scale=wavelet_scale.astype(np.float32),
    )


# The synthetic workloads: WTConvNeXt-T layer shapes (k = 5 throughout).
WORKLOADS = {
    "tiny": dict(N=2, C=32, H=32, W=32, levels=2, k=5, dtype="f32", seed=0),
    "stage1": dict(N=64, C=96, H=56, W=56, levels=3, k=5, dtype="f32", seed=1000),
    "stage2_f16": dict(N=128, C=192, H=28, W=28, levels=2, k=5, dtype="f16", seed=2000),
    "stage2_bf16": dict(N=128, C=192, H=28, W=28, levels=2, k=5, dtype="bf16", seed=2001),
}

# (C, H=W) shapes of the four WTConvNeXt-T stages and the level sweep.
SWEEP_SHAPES = ((96, 56), (192, 28), (384, 14), (768, 7))
SWEEP_LEVELS = (1, 2, 3, 4, 5)
# All WTConv layers of WTConvNeXt-T at 224x224 input: (C, H=W, depth, levels).
NETWORK_STAGES = ((96, 56, 3, 5), (192, 28, 3, 4), (384, 14, 9, 3), (768, 7, 3, 2))
# Planes larger than one CTA holds (run tile by tile with a halo): a WTConv
# layer at the stem resolution of a 224x224 image for levels 1-4, and larger
# maps.  (N, C, H, W, levels, k, dtype); every tensor is larger than the L2.
LARGE_PLANES = ((16, 64, 224, 224, 1, 5, "f32"), (16, 64, 224, 224, 2, 5, "f32"), (16, 64, 224, 224, 3, 5, "f32"),
                (16, 64, 224, 224, 4, 5, "f32"), (32, 64, 224, 224, 3, 5, "f16"), (32, 96, 128, 128, 3, 5, "f32"),
                (16, 32, 384, 384, 2, 5, "f32"), (8, 32, 512, 512, 2, 5, "f16"),
                # reaches whose tile window does not fit one CTA: a fine pass and a coarse layer
                (16, 64, 224, 224, 5, 5, "f32"), (16, 64, 224, 224, 6, 3, "f16"))


def workload(name: str, **overrides) -> LayerInputs:
    cfg = dict(WORKLOADS[name])
    cfg.update(overrides)
    return make_inputs(**cfg)
