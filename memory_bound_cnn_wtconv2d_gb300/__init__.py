"""GB300-native WTConv2d: fused forward and backward of the wavelet convolution
layer, delivered as the C-ABI library ``libwtconv.so`` (include/wtconv.h) with
hand-written sm_103a kernels, plus this thin Python binding."""
from . import synth  # noqa: F401  (seeded synthetic inputs; no layer arithmetic)

__all__ = ["synth", "wtconv", "layer"]
