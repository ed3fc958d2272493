"""GPU parity of the windowed passes (planes whose Haar pyramids do not fit
one CTA) against the float64 oracle: forward, input gradient and every
parameter gradient.

Every shape below is larger than any whole plane the library keeps in one
CTA (at most about 112 x 112 pixels for the forward, 56 x 56 for the
parameter gradient), so the calls run tile by tile with a halo.  The cases
span every window load (float32 box copies, 16-bit box copies widened on
chip, plain loads for rows that are not whole 16-byte chunks or pointers
that are not 16-byte aligned), ragged edge tiles, odd sizes padded at every
level, each kernel size and levels 1 to 5.  Tolerances are those of the
whole-plane tests (relative L2 and elementwise against the largest oracle
magnitude).
"""
import numpy as np
import pytest
import torch

from memory_bound_cnn_wtconv2d_gb300 import synth

from test_parity_gpu import GRADS, check_all, to_dev, wt  # noqa: F401  (wt is a fixture)

pytestmark = pytest.mark.gpu


def fwd_and_dx(wt, inp, d):
    L, k = inp.levels, inp.k
    y = wt.wtconv_fwd(d["x"], d["w_base"], d["b_base"], d["w_sub"], d["base_scale"], d["wavelet_scale"], L, k)
    dx = wt.wtconv_bwd_data(d["dy"], d["w_base"], d["w_sub"], d["base_scale"], d["wavelet_scale"], L, k)
    torch.cuda.synchronize()
    assert wt.wtconv_device_faults() == 0, "an in-kernel bounded wait gave up"
    return y.float().cpu().numpy(), dx.float().cpu().numpy()


# (N, C, H, W, L, k, dtype): the window load each one takes is in the id
WINDOWED = [
    (2, 3, 150, 150, 3, 5, "f32"),   # float32 box copies, ragged last tile
    (1, 2, 113, 129, 3, 5, "f32"),   # W odd: plain loads; odd sizes at every level
    (3, 2, 128, 128, 1, 9, "f32"),   # one level, widest kernel
    (1, 2, 130, 124, 2, 7, "f32"),
    (1, 2, 144, 136, 4, 3, "f32"),   # 4 levels: 32-pixel halo
    (1, 2, 160, 152, 4, 5, "f32"),
    (1, 2, 168, 160, 5, 3, "f32"),   # 5 levels (k = 3)
    (1, 3, 1023, 17, 2, 5, "f32"),   # tall and narrow: one tile column, W not a multiple of 4
    (2, 2, 200, 136, 4, 3, "f16"),   # 16-bit box copies, widened on chip
    (1, 2, 120, 120, 3, 5, "bf16"),
    (1, 2, 131, 125, 3, 7, "f16"),   # 16-bit plain loads
    (1, 2, 256, 256, 2, 9, "bf16"),
]


@pytest.mark.parametrize("case", WINDOWED, ids=lambda s: "x".join(map(str, s)))
def test_windowed_matches_oracle(wt, case):
    N, C, H, W, L, k, dtype = case
    check_all(wt, synth.make_inputs(N, C, H, W, L, k, dtype=dtype, seed=H * 7 + W + L + k))


# Planes the forward still keeps whole but the parameter gradient does not
# (57..112 pixels): whole-plane forward, windowed parameter gradient.
@pytest.mark.parametrize("case", [(2, 3, 64, 64, 3, 5, "f32"), (1, 2, 57, 61, 2, 7, "f32"), (3, 2, 96, 80, 4, 3, "f16"),
                                  (2, 2, 72, 72, 1, 9, "bf16")], ids=lambda s: "x".join(map(str, s)))
def test_windowed_parameter_gradient_only(wt, case):
    N, C, H, W, L, k, dtype = case
    check_all(wt, synth.make_inputs(N, C, H, W, L, k, dtype=dtype, seed=H + W * 3 + L + k))


def test_windowed_without_bias_and_unaligned_pointers(wt):
    # activations one element past a 16-byte boundary: plain scalar loads and stores
    inp = synth.make_inputs(1, 2, 136, 128, 3, 5, seed=11, bias=False)
    d = to_dev(inp)
    for key in ("x", "dy"):
        buf = torch.empty(d[key].numel() + 1, dtype=d[key].dtype, device="cuda")
        view = buf[1:].view_as(d[key])
        view.copy_(d[key])
        d[key] = view
    assert d["x"].data_ptr() % 16 != 0
    check_all(wt, inp, d)


def test_windowed_matches_whole_plane_results_elementwise(wt):
    # The same layer at a plane that still fits one CTA (whole-plane kernel)
    # and embedded in a larger, zero-extended plane (windowed kernel): on the
    # common pixels the outputs are the same sums of the same coefficients
    # up to rounding, so they agree to float32 rounding.
    inp = synth.make_inputs(2, 2, 64, 64, 3, 5, seed=5)
    d = to_dev(inp)
    y_small, dx_small = fwd_and_dx(wt, inp, d)
    big = {k: v for k, v in d.items()}
    for key in ("x", "dy"):
        z = torch.zeros(2, 2, 192, 192, dtype=d[key].dtype, device="cuda")
        z[:, :, :64, :64] = d[key]
        big[key] = z
    y_big, dx_big = fwd_and_dx(wt, inp, big)
    scale = np.abs(y_small).max()
    assert np.abs(y_big[:, :, :64, :64] - y_small).max() <= 1e-5 * scale
    scale = np.abs(dx_small).max()
    assert np.abs(dx_big[:, :, :64, :64] - dx_small).max() <= 1e-5 * scale


def test_windowed_full_size(wt):
    # An ImageNet-stem-sized layer (N=8, C=64, 224 x 224, 3 levels, k=5,
    # float32) in the launch configuration a user gets, every output and
    # every parameter gradient against the oracle.
    check_all(wt, synth.make_inputs(8, 64, 224, 224, 3, 5, seed=224))


def test_windowed_parameter_gradient_is_deterministic_and_noalloc_agrees(wt):
    inp = synth.make_inputs(2, 3, 200, 136, 3, 5, seed=21)
    d = to_dev(inp)
    args = (d["x"], d["dy"], d["w_base"], d["b_base"], d["w_sub"], d["base_scale"], d["wavelet_scale"], 3, 5)
    g1 = wt.wtconv_bwd_weight(*args)
    g2 = wt.wtconv_bwd_weight(*args)
    g3 = wt.wtconv_bwd_weight_noalloc(*args)
    torch.cuda.synchronize()
    assert wt.wtconv_device_faults() == 0
    for name in GRADS:
        assert torch.equal(g1[name], g2[name]), name
        assert torch.equal(g1[name], g3[name]), name


def test_reach_beyond_one_cta_splits(wt):
    # 5 levels at k = 5 need a 64-pixel halo around every tile: even the
    # smallest tile's window does not fit one CTA, so levels 5.. run as a
    # coarse layer on the level-4 low-pass planes (tests/test_split_gpu.py);
    # 4 levels still run tile by tile in one pass.
    check_all(wt, synth.make_inputs(1, 2, 224, 224, 5, 5, seed=3))
    check_all(wt, synth.make_inputs(1, 2, 224, 224, 4, 5, seed=3))