"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Tolerances (relative L2 error against the oracle on the same seeded,
storage-rounded inputs): float32 activations 1e-5 on y and dx, 1e-4 on every
parameter gradient; float16 2e-2; bfloat16 4e-2.  Besides the norm-wise
figure, every element is checked against an elementwise bound scaled by the
largest oracle magnitude of that output.
"""
import numpy as np
import pytest
import torch

import oracle
from memory_bound_cnn_wtconv2d_gb300 import synth

pytestmark = pytest.mark.gpu

TORCH_DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
REL_L2 = {"f32": (1e-5, 1e-4), "f16": (2e-2, 2e-2), "bf16": (4e-2, 4e-2)}
ELEM = {"f32": (2e-5, 2e-4), "f16": (2e-2, 2e-2), "bf16": (4e-2, 4e-2)}
GRADS = ("dw_base", "db_base", "dw_sub", "dbase_scale", "dwavelet_scale")


@pytest.fixture(scope="module")
def wt():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from memory_bound_cnn_wtconv2d_gb300 import build
    build.build()
    from memory_bound_cnn_wtconv2d_gb300 import wtconv
    return wtconv


def to_dev(inp):
    dev = "cuda"
    dt = TORCH_DT[inp.dtype]
    t = lambda a, d=torch.float32: None if a is None else torch.tensor(a, dtype=d, device=dev)
    return dict(x=t(inp.x, dt), dy=t(inp.dy, dt), w_base=t(inp.w_base), b_base=t(inp.b_base),
                w_sub=t(inp.w_sub), base_scale=t(inp.base_scale), wavelet_scale=t(inp.wavelet_scale))


def run_gpu(wt, inp, d=None):
    d = to_dev(inp) if d is None else d
    L, k = inp.levels, inp.k
    y = wt.wtconv_fwd(d["x"], d["w_base"], d["b_base"], d["w_sub"], d["base_scale"], d["wavelet_scale"], L, k)
    dx = wt.wtconv_bwd_data(d["dy"], d["w_base"], d["w_sub"], d["base_scale"], d["wavelet_scale"], L, k)
    g = wt.wtconv_bwd_weight(d["x"], d["dy"], d["w_base"], d["b_base"], d["w_sub"], d["base_scale"],
                             d["wavelet_scale"], L, k)
    torch.cuda.synchronize()
    assert wt.wtconv_device_faults() == 0, "an in-kernel bounded wait gave up"
    out = dict(y=y.float().cpu().numpy(), dx=dx.float().cpu().numpy())
    for name in GRADS:
        out[name] = None if g[name] is None else g[name].cpu().numpy()
    return out


def compare(name, got, ref, dtype, is_grad):
    tol = REL_L2[dtype][1 if is_grad else 0]
    etol = ELEM[dtype][1 if is_grad else 0]
    got = np.asarray(got, np.float64)
    assert got.shape == ref.shape, name
    assert np.isfinite(got).all(), name
    scale = np.abs(ref).max()
    err = np.linalg.norm((got - ref).ravel()) / max(np.linalg.norm(ref.ravel()), 1e-30)
    assert err <= tol, f"{name}: rel-L2 {err:.3g} > {tol}"
    worst = np.abs(got - ref).max()
    assert worst <= etol * max(scale, 1e-30), f"{name}: max abs err {worst:.3g} > {etol} * {scale:.3g}"
    return err


def check_all(wt, inp, d=None):
    got = run_gpu(wt, inp, d)
    y_ref = oracle.fwd(inp)
    g_ref = oracle.bwd(inp)
    errs = {"y": compare("y", got["y"], y_ref, inp.dtype, False),
            "dx": compare("dx", got["dx"], g_ref["dx"], inp.dtype, False)}
    for name in GRADS:
        if g_ref[name] is None:
            assert got[name] is None
            continue
        errs[name] = compare(name, got[name], g_ref[name], inp.dtype, True)
    return errs


# shapes spanning several tiles with ragged tails, odd sizes, deep pyramids
SMALL = [
    (2, 3, 13, 17, 3, 5), (1, 2, 9, 7, 2, 3), (3, 2, 20, 12, 4, 7), (2, 2, 33, 31, 5, 9),
    (1, 1, 1, 1, 1, 3), (1, 2, 1, 9, 2, 5), (2, 3, 7, 7, 5, 5), (2, 4, 56, 56, 3, 5),
    (3, 4, 28, 28, 2, 5), (5, 4, 14, 14, 3, 5), (9, 6, 7, 7, 2, 5), (2, 2, 40, 40, 1, 5),
    (2, 2, 64, 48, 6, 3), (1, 2, 5, 64, 3, 5), (37, 3, 7, 7, 4, 3),
]


def shape_seed(shape):
    return int(sum((i + 1) * v for i, v in enumerate(shape)))


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_small_shapes(wt, shape, dtype):
    inp = synth.make_inputs(*shape, dtype=dtype, seed=shape_seed(shape))
    check_all(wt, inp)


def test_tiny_workload(wt):
    check_all(wt, synth.workload("tiny"))


@pytest.mark.parametrize("k", [3, 5, 7, 9])
def test_kernel_sizes(wt, k):
    check_all(wt, synth.make_inputs(2, 3, 19, 23, 3, k, seed=k))


# Layers whose parameter-gradient plans take each tile variant of the
# whole-plane kernel: one 4-row tile per thread (planes that fill the CTA:
# 7 x 7, 14 x 14; at k = 9 two per thread, the one-tile kernel fitting no
# more CTAs), two 4-row tiles per thread (28 x 28 at 4 levels) and 8-row
# tiles (28 x 28 at 2 levels), each with several units per CTA slot.
TILE_VARIANTS = [(24, 2, 7, 7, 2), (8, 3, 14, 14, 3), (3, 2, 28, 28, 4), (4, 2, 28, 28, 2)]


@pytest.mark.parametrize("shape", TILE_VARIANTS, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("k", [3, 5, 7, 9])
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_gradient_tile_variants(wt, shape, k, dtype):
    check_all(wt, synth.make_inputs(*shape, k, dtype=dtype, seed=shape_seed(shape) + k))


def test_no_bias(wt):
    check_all(wt, synth.make_inputs(2, 3, 21, 18, 3, 5, seed=4, bias=False))


def test_unaligned_pointers_take_scalar_path(wt):
    # activations offset by one element: element-aligned, not 16-byte aligned
    inp = synth.make_inputs(2, 3, 16, 16, 2, 5, seed=8)
    d = to_dev(inp)
    for key in ("x", "dy"):
        buf = torch.empty(d[key].numel() + 1, dtype=d[key].dtype, device="cuda")
        view = buf[1:].view(d[key].shape)
        view.copy_(d[key])
        d[key] = view
    check_all(wt, inp, d)


def test_empty_batch(wt):
    inp = synth.make_inputs(0, 3, 16, 16, 2, 5, seed=1)
    got = run_gpu(wt, inp)
    assert got["y"].shape == (0, 3, 16, 16) and got["dx"].shape == (0, 3, 16, 16)
    for name in GRADS:
        assert np.all(got[name] == 0), name


def test_bwd_weight_is_deterministic(wt):
    inp = synth.make_inputs(16, 8, 28, 28, 3, 5, seed=12)
    d = to_dev(inp)
    a = wt.wtconv_bwd_weight(d["x"], d["dy"], d["w_base"], d["b_base"], d["w_sub"], d["base_scale"],
                             d["wavelet_scale"], 3, 5)
    b = wt.wtconv_bwd_weight(d["x"], d["dy"], d["w_base"], d["b_base"], d["w_sub"], d["base_scale"],
                             d["wavelet_scale"], 3, 5)
    for name in GRADS:
        assert torch.equal(a[name], b[name]), name


def test_autograd_module_matches_oracle(wt):
    from memory_bound_cnn_wtconv2d_gb300.layer import WTConv2d
    torch.manual_seed(0)
    m = WTConv2d(4, kernel_size=5, levels=3, device="cuda")
    x = torch.randn(2, 4, 24, 20, device="cuda", requires_grad=True)
    y = m(x)
    dy = torch.randn_like(y)
    y.backward(dy)
    inp = synth.make_inputs(2, 4, 24, 20, 3, 5)
    inp.x = x.detach().cpu().numpy()
    inp.dy = dy.cpu().numpy()
    inp.w_base = m.weight.detach().cpu().numpy()
    inp.b_base = m.bias.detach().cpu().numpy()
    inp.w_sub = m.wavelet_weight.detach().cpu().numpy()
    inp.base_scale = m.base_scale.detach().cpu().numpy()
    inp.wavelet_scale = m.wavelet_scale.detach().cpu().numpy()
    compare("y", y.detach().cpu().numpy(), oracle.fwd(inp), "f32", False)
    g = oracle.bwd(inp)
    compare("dx", x.grad.cpu().numpy(), g["dx"], "f32", False)
    compare("dw_base", m.weight.grad.cpu().numpy(), g["dw_base"], "f32", True)
    compare("db_base", m.bias.grad.cpu().numpy(), g["db_base"], "f32", True)
    compare("dw_sub", m.wavelet_weight.grad.cpu().numpy(), g["dw_sub"], "f32", True)
    compare("dbase_scale", m.base_scale.grad.cpu().numpy(), g["dbase_scale"], "f32", True)
    compare("dwavelet_scale", m.wavelet_scale.grad.cpu().numpy(), g["dwavelet_scale"], "f32", True)


@pytest.mark.parametrize("which", ["input_only", "params_only"])
def test_autograd_module_single_gradient_paths(wt, which):
    # The module's backward computes only what autograd asks for: dx alone
    # (frozen parameters) runs the input-gradient call, parameter gradients
    # alone (an input that needs no gradient) the parameter-gradient call.
    from memory_bound_cnn_wtconv2d_gb300.layer import WTConv2d
    torch.manual_seed(1)
    m = WTConv2d(4, kernel_size=5, levels=2, device="cuda")
    x = torch.randn(2, 4, 20, 24, device="cuda", requires_grad=(which == "input_only"))
    if which == "input_only":
        for p in m.parameters():
            p.requires_grad_(False)
    y = m(x)
    dy = torch.randn_like(y)
    y.backward(dy)
    inp = synth.make_inputs(2, 4, 20, 24, 2, 5)
    inp.x = x.detach().cpu().numpy()
    inp.dy = dy.cpu().numpy()
    inp.w_base = m.weight.detach().cpu().numpy()
    inp.b_base = m.bias.detach().cpu().numpy()
    inp.w_sub = m.wavelet_weight.detach().cpu().numpy()
    inp.base_scale = m.base_scale.detach().cpu().numpy()
    inp.wavelet_scale = m.wavelet_scale.detach().cpu().numpy()
    g = oracle.bwd(inp)
    if which == "input_only":
        compare("dx", x.grad.cpu().numpy(), g["dx"], "f32", False)
        assert all(p.grad is None for p in m.parameters())
    else:
        assert x.grad is None
        compare("dw_base", m.weight.grad.cpu().numpy(), g["dw_base"], "f32", True)
        compare("db_base", m.bias.grad.cpu().numpy(), g["db_base"], "f32", True)
        compare("dw_sub", m.wavelet_weight.grad.cpu().numpy(), g["dw_sub"], "f32", True)
        compare("dbase_scale", m.base_scale.grad.cpu().numpy(), g["dbase_scale"], "f32", True)
        compare("dwavelet_scale", m.wavelet_scale.grad.cpu().numpy(), g["dwavelet_scale"], "f32", True)


# ---- full-size workloads, in the launch configuration the benchmark times ----

@pytest.mark.parametrize("name", ["stage1", "stage2_f16", "stage2_bf16"])
def test_full_size_workloads(wt, name):
    errs = check_all(wt, synth.workload(name))
    print(name, {k: f"{v:.2e}" for k, v in errs.items()})


@pytest.mark.parametrize("C,H", synth.SWEEP_SHAPES)
@pytest.mark.parametrize("L", synth.SWEEP_LEVELS)
@pytest.mark.parametrize("dtype", ["f32", "f16"])
def test_level_sweep_shapes(wt, C, H, L, dtype):
    # the sweep's (C, H=W, L) shapes at a reduced batch (every plane is
    # independent, so the batch size does not change the per-plane path);
    # covers both input-set layouts, 16-bit staging and both final-tile heights
    check_all(wt, synth.make_inputs(3, C // 8, H, H, L, 5, dtype=dtype, seed=C + H + L))


# The largest planes each pass of this build handles (shared memory per CTA for
# the forward / input-gradient pass; register-resident gradient tiles for the
# parameter-gradient pass), and the deepest pyramids (L = 8: the coarse levels
# are 1x1 planes of zero-padded blocks).
@pytest.mark.parametrize("N,C,H,W,L,k", [(1, 2, 104, 104, 3, 3), (1, 2, 96, 96, 5, 9), (1, 2, 100, 100, 8, 3),
                                         (1, 2, 3, 512, 1, 5), (2, 3, 92, 92, 8, 9)])
def test_forward_and_input_gradient_at_maximum_plane(wt, N, C, H, W, L, k):
    inp = synth.make_inputs(N, C, H, W, L, k, seed=H + W + L + k)
    d = to_dev(inp)
    y = wt.wtconv_fwd(d["x"], d["w_base"], d["b_base"], d["w_sub"], d["base_scale"], d["wavelet_scale"], L, k)
    dx = wt.wtconv_bwd_data(d["dy"], d["w_base"], d["w_sub"], d["base_scale"], d["wavelet_scale"], L, k)
    torch.cuda.synchronize()
    assert wt.wtconv_device_faults() == 0
    compare("y", y.cpu().numpy(), oracle.fwd(inp), "f32", False)
    compare("dx", dx.cpu().numpy(), oracle.bwd(inp)["dx"], "f32", False)


@pytest.mark.parametrize("N,C,H,W,L,k", [(1, 2, 56, 56, 8, 9), (2, 2, 64, 64, 1, 5), (1, 3, 3, 256, 3, 5),
                                         (2, 2, 56, 55, 5, 7)])
def test_all_passes_at_maximum_gradient_plane(wt, N, C, H, W, L, k):
    check_all(wt, synth.make_inputs(N, C, H, W, L, k, seed=H + W + L + k))
