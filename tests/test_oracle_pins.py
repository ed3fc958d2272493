"""Pins for the CPU oracle (CPU only).

Each test ties the oracle to something other than its own arithmetic: the
mathematics of the orthonormal Haar pair, closed forms for delta kernels,
hand-derived fixtures, PyTorch library routines (conv2d, conv_transpose2d and
autograd, float64), linearity, the adjoint identity and finite differences.
The layer follows "Fast and Memory-Efficient Wavelet Convolutions via
I/O-Aware Reformulation" (arXiv 2608.10805), technical summary on
gist.science, "Methodology".
"""
import itertools

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from memory_bound_cnn_wtconv2d_gb300 import synth
from conftest import read_golden

pytestmark = pytest.mark.filterwarnings("ignore")


def rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm((a - b).ravel()) / max(np.linalg.norm(b.ravel()), 1e-300))


def unit_layer(N, C, H, W, L, k, seed=0):
    """Delta kernels, unit scales, zero bias."""
    inp = synth.make_inputs(N, C, H, W, L, k, seed=seed, bias=False)
    r = k // 2
    inp.w_base[:] = 0
    inp.w_base[:, r, r] = 1
    inp.w_sub[:] = 0
    inp.w_sub[:, :, r, r] = 1
    inp.base_scale[:] = 1
    inp.wavelet_scale[:] = 1
    return inp


def block_mean(x, m):
    """Mean of x (zero-extended) over aligned 2^m x 2^m blocks, expanded back and cropped."""
    H, W = x.shape[-2:]
    s = 1 << m
    Hp, Wp = -(-H // s) * s, -(-W // s) * s
    xp = np.zeros(x.shape[:-2] + (Hp, Wp))
    xp[..., :H, :W] = x
    blk = xp.reshape(x.shape[:-2] + (Hp // s, s, Wp // s, s)).mean(axis=(-3, -1))
    up = np.repeat(np.repeat(blk, s, axis=-2), s, axis=-1)
    return up[..., :H, :W]


# ------------------------------------------------------------- Haar pair --

@pytest.mark.parametrize("H,W", [(1, 1), (1, 5), (2, 2), (3, 3), (5, 8), (7, 7), (8, 5), (9, 16), (16, 16), (17, 6)])
def test_perfect_reconstruction(H, W):
    x = np.random.default_rng(H * 100 + W).standard_normal((H, W))
    bands = oracle.haar_analysis(x)
    assert bands.shape == (4, (H + 1) // 2, (W + 1) // 2)
    assert np.abs(oracle.haar_synthesis(bands, H, W) - x).max() < 1e-14


@pytest.mark.parametrize("H,W", [(3, 5), (6, 6), (7, 9)])
def test_parseval(H, W):
    # orthonormal analysis preserves energy (padding adds zeros only)
    x = np.random.default_rng(7).standard_normal((H, W))
    bands = oracle.haar_analysis(x)
    assert abs((bands ** 2).sum() - (x ** 2).sum()) < 1e-12 * (x ** 2).sum()


def test_synthesis_is_transpose_of_analysis():
    rng = np.random.default_rng(3)
    for H, W in [(5, 7), (6, 4)]:
        x = rng.standard_normal((H, W))
        z = rng.standard_normal((4, (H + 1) // 2, (W + 1) // 2))
        lhs = (oracle.haar_analysis(x) * z).sum()
        rhs = (x * oracle.haar_synthesis(z, H, W)).sum()
        assert abs(lhs - rhs) < 1e-12 * abs(lhs)


def test_haar_golden_2x2():
    g = read_golden("haar_2x2_bands.txt")
    x = np.array(g["x"]).reshape(2, 2)
    bands = oracle.haar_analysis(x)
    np.testing.assert_allclose(bands.ravel(), g["bands"], atol=1e-15)
    total = np.zeros((2, 2))
    for b in range(4):
        one = np.zeros_like(bands)
        one[b] = bands[b]
        proj = oracle.haar_synthesis(one, 2, 2)
        np.testing.assert_allclose(proj.ravel(), g[f"proj{b}"], atol=1e-15)
        total += proj
    np.testing.assert_allclose(total, x, atol=1e-15)


# ----------------------------------------------------------- closed forms --

@pytest.mark.parametrize("case", ["caseA", "caseB", "caseC"])
@pytest.mark.parametrize("form", ["cascade", "direct"])
def test_delta_kernel_golden(case, form):
    g = read_golden("delta_kernels.txt")
    H, W = (int(v) for v in g[f"{case}_shape"])
    L = int(g[f"{case}_levels"][0])
    inp = unit_layer(1, 1, H, W, L, 3)
    inp.x = np.array(g[f"{case}_x"], np.float32).reshape(1, 1, H, W)
    y = oracle.fwd(inp, form)
    np.testing.assert_allclose(y.ravel(), g[f"{case}_y"], rtol=0, atol=1e-12)


@pytest.mark.parametrize("H,W,L", [(8, 8, 3), (7, 9, 3), (5, 5, 4), (16, 12, 2), (6, 11, 5)])
@pytest.mark.parametrize("k", [3, 5])
def test_delta_kernel_closed_form(H, W, L, k):
    inp = unit_layer(2, 3, H, W, L, k, seed=H + W)
    x = inp.x.astype(np.float64)
    expect = 2 * x + sum(block_mean(x, m) for m in range(1, L))
    for form in ("cascade", "direct"):
        assert rel(oracle.fwd(inp, form), expect) < 1e-13


@pytest.mark.parametrize("b", [0, 1, 2, 3])
def test_single_band_projection_level1(b):
    # only level-1 band b is a delta (others zero, base zero): y = P_b x, the
    # projection of each 2x2 block onto the band's sign pattern.
    H, W, k = 6, 8, 3
    inp = unit_layer(1, 2, H, W, 2, k, seed=b)
    inp.w_base[:] = 0
    inp.w_sub[:] = 0
    inp.w_sub[0, b::4, 1, 1] = 1
    x = inp.x.astype(np.float64)
    pat = np.array([[1, 1], [1, 1]] if b == 0 else
                   [[1, 1], [-1, -1]] if b == 1 else
                   [[1, -1], [1, -1]] if b == 2 else
                   [[1, -1], [-1, 1]], np.float64)
    blocks = x.reshape(1, 2, H // 2, 2, W // 2, 2)
    coef = np.einsum("ncpuqv,uv->ncpq", blocks, pat) / 4.0
    expect = np.einsum("ncpq,uv->ncpuqv", coef, pat).reshape(x.shape)
    assert rel(oracle.fwd(inp), expect) < 1e-13


def test_coarsest_lowpass_is_block_mean():
    # only the level-L low-pass subband is a delta -> M_L(x)
    H, W, L = 12, 10, 3
    inp = unit_layer(1, 2, H, W, L, 3, seed=5)
    inp.w_base[:] = 0
    inp.w_sub[:] = 0
    inp.w_sub[L - 1, 0::4, 1, 1] = 1
    x = inp.x.astype(np.float64)
    assert rel(oracle.fwd(inp), block_mean(x, L)) < 1e-13


def test_receptive_field():
    # one input impulse only reaches outputs within the level-L block grid
    # dilated by the level-L conv radius (exponential receptive field)
    H = W = 32
    L, k = 2, 3
    inp = synth.make_inputs(1, 1, H, W, L, k, seed=9, bias=False)
    inp.x = np.zeros_like(inp.x)
    inp.x[0, 0, 0, 0] = 1.0
    y = oracle.fwd(inp)
    reach = (1 << L) * (1 + k // 2)  # block of 2^L plus radius in level-L pixels
    assert np.abs(y[0, 0, reach:, :]).max() == 0.0
    assert np.abs(y[0, 0, :, reach:]).max() == 0.0
    assert np.abs(y[0, 0, reach - 1, :]).max() > 0.0


# --------------------------------------------------- torch compositions --

def torch_layer(inp, requires_grad=False):
    """The unfused layer written with PyTorch library ops in float64."""
    t = lambda a: None if a is None else torch.tensor(np.asarray(a, np.float64), requires_grad=requires_grad)
    x, wb, bb, ws, sb, sw = (t(inp.x), t(inp.w_base), t(inp.b_base), t(inp.w_sub),
                             t(inp.base_scale), t(inp.wavelet_scale))
    N, C, H, W = x.shape
    L, k = inp.levels, inp.k
    r = k // 2
    haar = 0.5 * torch.tensor([[[1, 1], [1, 1]], [[1, 1], [-1, -1]], [[1, -1], [1, -1]], [[1, -1], [-1, 1]]],
                              dtype=torch.float64).unsqueeze(1)  # [4,1,2,2]
    filt = haar.repeat(C, 1, 1, 1)  # [4C,1,2,2], channel 4c+b
    cur, Zs, shapes = x, [], []
    for l in range(L):
        h, w = cur.shape[-2:]
        shapes.append((h, w))
        Y = F.conv2d(F.pad(cur, (0, w % 2, 0, h % 2)), filt, stride=2, groups=C)
        Zs.append(F.conv2d(Y, ws[l].unsqueeze(1), padding=r, groups=4 * C) * sw[l].view(1, -1, 1, 1))
        cur = Y.view(N, C, 4, *Y.shape[-2:])[:, :, 0]
    nxt = None
    for l in reversed(range(L)):
        Z = Zs[l]
        if nxt is not None:
            Zv = Z.view(N, C, 4, *Z.shape[-2:])
            Z = torch.cat([Zv[:, :, :1] + nxt.unsqueeze(2), Zv[:, :, 1:]], dim=2).view(Z.shape)
        h, w = shapes[l]
        nxt = F.conv_transpose2d(Z, filt, stride=2, groups=C)[..., :h, :w]
    y = F.conv2d(x, wb.unsqueeze(1), bb, padding=r, groups=C) * sb.view(1, -1, 1, 1) + nxt
    return y, dict(x=x, w_base=wb, b_base=bb, w_sub=ws, base_scale=sb, wavelet_scale=sw)


def test_base_path_equals_grouped_conv():
    inp = synth.make_inputs(2, 3, 9, 7, 2, 5, seed=11)
    inp.wavelet_scale[:] = 0.0
    x = torch.tensor(inp.x, dtype=torch.float64)
    ref = F.conv2d(x, torch.tensor(inp.w_base, dtype=torch.float64).unsqueeze(1),
                   torch.tensor(inp.b_base, dtype=torch.float64), padding=2, groups=3)
    ref = ref * torch.tensor(inp.base_scale, dtype=torch.float64).view(1, -1, 1, 1)
    assert rel(oracle.fwd(inp), ref.numpy()) < 1e-14


SHAPES = [(2, 3, 8, 8, 1, 3), (1, 2, 9, 7, 2, 5), (2, 2, 13, 10, 3, 5), (1, 3, 7, 7, 4, 3),
          (1, 2, 6, 5, 5, 7), (2, 1, 16, 16, 3, 9), (1, 2, 1, 6, 2, 3)]


@pytest.mark.parametrize("shape", SHAPES)
def test_forward_equals_torch_composition(shape):
    inp = synth.make_inputs(*shape, seed=sum(shape))
    y, _ = torch_layer(inp)
    assert rel(oracle.fwd(inp), y.numpy()) < 1e-13


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("bias", [True, False])
def test_backward_equals_torch_autograd(shape, bias):
    inp = synth.make_inputs(*shape, seed=sum(shape) + 1, bias=bias)
    y, leaves = torch_layer(inp, requires_grad=True)
    (y * torch.tensor(inp.dy, dtype=torch.float64)).sum().backward()
    got = oracle.bwd(inp)
    assert rel(got["dx"], leaves["x"].grad.numpy()) < 1e-12
    for name in ("w_base", "w_sub", "base_scale", "wavelet_scale"):
        assert rel(got["d" + name], leaves[name].grad.numpy()) < 1e-12, name
    if bias:
        assert rel(got["db_base"], leaves["b_base"].grad.numpy()) < 1e-12


# ---------------------------------------------------------- Form A == B --

@pytest.mark.parametrize("H,W", [(1, 1), (2, 3), (4, 4), (5, 9), (7, 7), (8, 6), (9, 9), (16, 16)])
@pytest.mark.parametrize("L", [1, 2, 3, 4])
def test_cascade_equals_direct(H, W, L):
    k = 3 if (H * W) % 2 else 5
    inp = synth.make_inputs(1, 2, H, W, L, k, seed=H * 31 + W * 7 + L)
    assert rel(oracle.fwd(inp, "cascade"), oracle.fwd(inp, "direct")) < 1e-12
    if H * W <= 81:
        a, b = oracle.bwd(inp, "cascade"), oracle.bwd(inp, "direct")
        for key in a:
            if a[key] is not None:
                assert rel(a[key], b[key]) < 1e-12, key


# ------------------------------------------------------------ identities --

def test_linearity_in_x():
    inp = synth.make_inputs(2, 2, 11, 9, 3, 5, seed=21, bias=False)
    rng = np.random.default_rng(0)
    x1, x2 = inp.x.astype(np.float64), rng.standard_normal(inp.x.shape)
    alpha, beta = 0.7, -1.3
    inp.x = x1
    y1 = oracle.fwd(inp)
    inp.x = x2
    y2 = oracle.fwd(inp)
    inp.x = alpha * x1 + beta * x2
    assert rel(oracle.fwd(inp), alpha * y1 + beta * y2) < 1e-13


@pytest.mark.parametrize("shape", [(2, 2, 11, 9, 3, 5), (1, 3, 16, 16, 4, 3), (1, 1, 7, 5, 5, 7)])
def test_adjoint_identity(shape):
    inp = synth.make_inputs(*shape, seed=5, bias=False)
    y = oracle.fwd(inp)
    dx = oracle.bwd(inp)["dx"]
    lhs = (y * inp.dy).sum()
    rhs = (inp.x.astype(np.float64) * dx).sum()
    assert abs(lhs - rhs) < 1e-12 * max(abs(lhs), 1.0)


def test_finite_difference_every_parameter():
    # loss = <y, dy> is linear in each single parameter, so a central
    # difference is exact up to rounding.
    inp = synth.make_inputs(1, 2, 8, 8, 2, 3, seed=13)
    g = oracle.bwd(inp)
    dy = inp.dy.astype(np.float64)
    eps = 1e-3

    def loss():
        return float((oracle.fwd(inp) * dy).sum())

    for name, grad in [("w_base", "dw_base"), ("b_base", "db_base"), ("w_sub", "dw_sub"),
                       ("base_scale", "dbase_scale"), ("wavelet_scale", "dwavelet_scale")]:
        arr = getattr(inp, name)
        arr64 = arr.astype(np.float64)
        setattr(inp, name, arr64)
        for idx in itertools.product(*[range(s) for s in arr64.shape]):
            old = arr64[idx]
            arr64[idx] = old + eps
            lp = loss()
            arr64[idx] = old - eps
            lm = loss()
            arr64[idx] = old
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - g[grad][idx]) < 1e-8 * max(1.0, abs(fd)), (name, idx)
        setattr(inp, name, arr)


def test_finite_difference_dx_sample():
    inp = synth.make_inputs(1, 2, 9, 7, 3, 5, seed=17)
    g = oracle.bwd(inp)
    dy = inp.dy.astype(np.float64)
    x = inp.x.astype(np.float64)
    inp.x = x
    rng = np.random.default_rng(1)
    for _ in range(20):
        idx = tuple(int(rng.integers(0, s)) for s in x.shape)
        old = x[idx]
        x[idx] = old + 1e-3
        lp = float((oracle.fwd(inp) * dy).sum())
        x[idx] = old - 1e-3
        lm = float((oracle.fwd(inp) * dy).sum())
        x[idx] = old
        assert abs((lp - lm) / 2e-3 - g["dx"][idx]) < 1e-8


def test_rejects_even_kernel():
    inp = synth.make_inputs(1, 1, 4, 4, 1, 3)
    inp.k = 4
    with pytest.raises(ValueError):
        oracle.fwd(inp)


# ------------------------------------------- comparison arm of the bench --

@pytest.mark.parametrize("shape", [(2, 3, 9, 7, 2, 5), (1, 2, 13, 10, 3, 3), (1, 2, 8, 8, 1, 5)])
def test_bench_unfused_arm_equals_oracle(shape):
    """bench.py's unfused PyTorch composition (a timing comparison arm) computes
    the same layer and gradients as the oracle, so its timings compare like with
    like."""
    import bench
    inp = synth.make_inputs(*shape, seed=sum(shape) + 5)
    t = lambda a: torch.tensor(np.asarray(a, np.float64), requires_grad=True)
    leaves = [t(a) for a in (inp.x, inp.w_base, inp.b_base, inp.w_sub, inp.base_scale, inp.wavelet_scale)]
    y = bench.unfused_torch_layer(*leaves, inp.levels, inp.k)
    assert rel(oracle.fwd(inp), y.detach().numpy()) < 1e-13
    (y * torch.tensor(inp.dy, dtype=torch.float64)).sum().backward()
    got = oracle.bwd(inp)
    assert rel(got["dx"], leaves[0].grad.numpy()) < 1e-12
    assert rel(got["dw_sub"], leaves[3].grad.numpy()) < 1e-12
    assert rel(got["dwavelet_scale"], leaves[5].grad.numpy()) < 1e-12
