"""GPU parity at the descriptor limits, against the float64 oracle.

- The largest plane the library takes, H * W = 2^24 (4096 x 4096), at the
  deepest pyramid (8 levels): tiles with a halo for the fine levels and a
  coarse layer on the level-5 low-pass planes (k = 3).
- Many tiny planes: 2^20 channels of 1 x 1 pixels, so unit, channel and
  record indices run far past the sizes the other tests reach, while every
  band is the zero-padded 1 x 1 block.
Each checks every pass (y, dx from both backward entry points, every
parameter gradient) with the tolerances of the whole-plane tests.
"""
import pytest
import torch

import oracle
from memory_bound_cnn_wtconv2d_gb300 import synth

from test_parity_gpu import GRADS, compare, to_dev, wt  # noqa: F401  (wt is a fixture)

pytestmark = pytest.mark.gpu


def all_passes(wt, inp):
    d = to_dev(inp)
    L, k = inp.levels, inp.k
    ps = [d[n] for n in ("w_base", "b_base", "w_sub", "base_scale", "wavelet_scale")]
    y = wt.wtconv_fwd(d["x"], *ps, L, k)
    dx = wt.wtconv_bwd_data(d["dy"], ps[0], ps[2], ps[3], ps[4], L, k)
    g = wt.wtconv_bwd_weight(d["x"], d["dy"], *ps, L, k)
    dx2, g2 = wt.wtconv_bwd(d["x"], d["dy"], *ps, L, k)
    torch.cuda.synchronize()
    assert wt.wtconv_device_faults() == 0
    compare("y", y.float().cpu().numpy(), oracle.fwd(inp), inp.dtype, False)
    ref = oracle.bwd(inp)
    compare("dx", dx.float().cpu().numpy(), ref["dx"], inp.dtype, False)
    compare("dx (wtconv_bwd)", dx2.float().cpu().numpy(), ref["dx"], inp.dtype, False)
    for n in GRADS:
        compare(n, g[n].cpu().numpy(), ref[n], inp.dtype, True)
        compare(n + " (wtconv_bwd)", g2[n].cpu().numpy(), ref[n], inp.dtype, True)


def test_largest_plane_at_the_deepest_pyramid(wt):
    all_passes(wt, synth.make_inputs(1, 1, 4096, 4096, 8, 3, dtype="f16", seed=4096))


def test_many_single_pixel_channels(wt):
    all_passes(wt, synth.make_inputs(1, 1 << 20, 1, 1, 2, 3, seed=20))
