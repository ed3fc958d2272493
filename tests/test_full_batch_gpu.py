"""GPU parity at the timed batch sizes: every layer of the shape/level sweep
and of the 18-layer WTConvNeXt-T network at N = 128, element by element
against the float64 oracle.

The planner picks the planes per unit (and with them the tile grid, the
number of input sets and the staging mode) from N, so a reduced batch would
not run the plans the benchmark times.  Here every sweep layer -- (C, H) in
the four WTConvNeXt-T stage shapes x levels 1..5, float32 and float16 -- and
the four distinct network layers (float16, their own seeds) run through
``wtconv_fwd`` + ``wtconv_bwd`` (the benchmark's step) and through the two
separate backward calls, at N = 128.  The oracle runs on image slices in
threads (``oracle.fwd_parallel`` / ``bwd_parallel``: the unchanged oracle on
parts of the batch), which keeps each layer to a second or so on 16 cores.

Tolerances as in test_parity_gpu.py: relative L2 1e-5 (y, dx) / 1e-4
(parameter gradients) for float32 activations, 2e-2 for float16, plus an
elementwise bound scaled by the largest oracle magnitude.
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
N_TIMED = 128


@pytest.fixture(scope="module")
def wt():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from memory_bound_cnn_wtconv2d_gb300 import build
    build.build()
    from memory_bound_cnn_wtconv2d_gb300 import wtconv
    return wtconv


def compare(name, got, ref, dtype, is_grad):
    tol = REL_L2[dtype][1 if is_grad else 0]
    etol = ELEM[dtype][1 if is_grad else 0]
    got = np.asarray(got, np.float64)
    assert got.shape == ref.shape, name
    assert np.isfinite(got).all(), name
    scale = float(np.abs(ref).max())
    err = float(np.linalg.norm((got - ref).ravel()) / max(np.linalg.norm(ref.ravel()), 1e-30))
    assert err <= tol, f"{name}: rel-L2 {err:.3g} > {tol}"
    worst = float(np.abs(got - ref).max())
    assert worst <= etol * max(scale, 1e-30), f"{name}: max abs err {worst:.3g} > {etol} * {scale:.3g}"
    return err


def run_layer(wt, inp):
    dev = "cuda"
    dt = TORCH_DT[inp.dtype]
    t = lambda a, d=torch.float32: None if a is None else torch.tensor(a, dtype=d, device=dev)
    x, dy = t(inp.x, dt), t(inp.dy, dt)
    ps = [t(inp.w_base), t(inp.b_base), t(inp.w_sub), t(inp.base_scale), t(inp.wavelet_scale)]
    L, k = inp.levels, inp.k
    y = wt.wtconv_fwd(x, *ps, L, k)
    dx_f, g_f = wt.wtconv_bwd(x, dy, *ps, L, k)
    dx_s = wt.wtconv_bwd_data(dy, ps[0], ps[2], ps[3], ps[4], L, k)
    g_s = wt.wtconv_bwd_weight(x, dy, *ps, L, k)
    torch.cuda.synchronize()
    assert wt.wtconv_device_faults() == 0, "an in-kernel bounded wait gave up"
    host = lambda a: None if a is None else a.float().cpu().numpy()
    got = {"y": host(y), "dx": host(dx_f), "dx (separate)": host(dx_s)}
    for n in GRADS:
        got[n] = host(g_f[n])
        got[n + " (separate)"] = host(g_s[n])
    del x, dy, y, dx_f, dx_s
    return got


def check_layer(wt, inp):
    got = run_layer(wt, inp)
    y_ref = oracle.fwd_parallel(inp)
    errs = {"y": compare("y", got.pop("y"), y_ref, inp.dtype, False)}
    del y_ref
    g_ref = oracle.bwd_parallel(inp)
    for key, val in got.items():
        base = key.split()[0]
        if g_ref[base] is None:
            assert val is None, key
            continue
        errs[key] = compare(key, val, g_ref[base], inp.dtype, base != "dx")
    return errs


@pytest.mark.parametrize("C,H", synth.SWEEP_SHAPES, ids=lambda v: str(v))
@pytest.mark.parametrize("L", synth.SWEEP_LEVELS)
@pytest.mark.parametrize("dtype", ["f32", "f16"])
def test_sweep_layer_at_timed_batch(wt, C, H, L, dtype):
    inp = synth.make_inputs(N_TIMED, C, H, H, L, 5, dtype=dtype, seed=3000 + 10 * C + L)
    errs = check_layer(wt, inp)
    print(f"sweep C{C} H{H} L{L} {dtype}", {k: f"{v:.2e}" for k, v in errs.items()})


@pytest.mark.parametrize("C,H,depth,L", synth.NETWORK_STAGES, ids=lambda v: str(v))
def test_network_layer_at_timed_batch(wt, C, H, depth, L):
    inp = synth.make_inputs(N_TIMED, C, H, H, L, 5, dtype="f16", seed=4000 + C)
    errs = check_layer(wt, inp)
    print(f"network C{C} H{H} L{L} f16", {k: f"{v:.2e}" for k, v in errs.items()})
