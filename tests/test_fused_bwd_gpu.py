"""GPU parity of wtconv_bwd, the whole backward in one call (one kernel over
x and dy where the planes fit), against the float64 oracle and against the
two separate calls it replaces.

The FUSED shapes are ones the fused kernel takes in float32 (8-row gradient
tiles, planes up to 64 x 64 pixels); the FALLBACK shapes are ones it hands
to the two separate passes, which the call must do transparently: 4-row
gradient tiles (deep pyramids, small planes packed several per unit),
planes beyond one CTA, and a 16-bit layer whose fused working set would
leave one CTA per SM.  Tolerances against the oracle
are those of the other parity tests; against the separate calls (same
float32 arithmetic, other evaluation order) dx and every gradient agree to
a relative 1e-6 of their largest magnitude in float32.
"""
import numpy as np
import pytest
import torch

import oracle
from memory_bound_cnn_wtconv2d_gb300 import synth

from test_parity_gpu import GRADS, compare, to_dev, wt  # noqa: F401  (wt is a fixture)

pytestmark = pytest.mark.gpu

FUSED = [(2, 4, 56, 56, 3, 5), (3, 4, 28, 28, 2, 5), (2, 2, 40, 40, 1, 5), (2, 2, 64, 48, 6, 3),
         (2, 3, 16, 16, 2, 5), (3, 2, 32, 32, 1, 7), (2, 2, 48, 40, 3, 9), (2, 2, 56, 55, 2, 5),
         # ragged last plane group (3 + 1, 3 + 3 + 1, 2 + 2 + 1 planes per unit) and the largest plane
         (4, 4, 28, 28, 2, 5), (7, 2, 32, 32, 1, 7), (5, 3, 40, 40, 1, 5), (2, 2, 64, 64, 1, 5)]
FALLBACK = [(2, 3, 13, 17, 3, 5, "f32"), (9, 6, 7, 7, 2, 5, "f32"), (2, 3, 28, 28, 4, 5, "f16"),
            (2, 2, 130, 124, 2, 5, "f32"), (2, 4, 56, 56, 5, 5, "bf16")]


def run_fused(wt, inp, d):
    L, k = inp.levels, inp.k
    dx, g = wt.wtconv_bwd(d["x"], d["dy"], d["w_base"], d["b_base"], d["w_sub"], d["base_scale"],
                          d["wavelet_scale"], L, k)
    torch.cuda.synchronize()
    assert wt.wtconv_device_faults() == 0, "an in-kernel bounded wait gave up"
    return dx.float().cpu().numpy(), {n: None if g[n] is None else g[n].cpu().numpy() for n in GRADS}


def run_separate(wt, inp, d):
    L, k = inp.levels, inp.k
    dx = wt.wtconv_bwd_data(d["dy"], d["w_base"], d["w_sub"], d["base_scale"], d["wavelet_scale"], L, k)
    g = wt.wtconv_bwd_weight(d["x"], d["dy"], d["w_base"], d["b_base"], d["w_sub"], d["base_scale"],
                             d["wavelet_scale"], L, k)
    torch.cuda.synchronize()
    return dx.float().cpu().numpy(), {n: None if g[n] is None else g[n].cpu().numpy() for n in GRADS}


def check(wt, inp, d=None, against_separate=True):
    d = to_dev(inp) if d is None else d
    dx, g = run_fused(wt, inp, d)
    ref = oracle.bwd(inp)
    compare("dx", dx, ref["dx"], inp.dtype, False)
    for n in GRADS:
        if ref[n] is None:
            assert g[n] is None
        else:
            compare(n, g[n], ref[n], inp.dtype, True)
    if against_separate:
        dx2, g2 = run_separate(wt, inp, d)
        tol = 1e-6 if inp.dtype == "f32" else 2 ** -7
        assert np.abs(dx - dx2).max() <= tol * max(np.abs(dx2).max(), 1e-30)
        for n in GRADS:
            if g2[n] is not None:
                assert np.abs(g[n] - g2[n]).max() <= 1e-6 * max(np.abs(g2[n]).max(), 1e-30), n


@pytest.mark.parametrize("shape", FUSED, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_fused_matches_oracle_and_separate_calls(wt, shape, dtype):
    check(wt, synth.make_inputs(*shape, dtype=dtype, seed=sum(shape) + 7))


@pytest.mark.parametrize("case", FALLBACK, ids=lambda s: "x".join(map(str, s)))
def test_layers_the_fused_kernel_does_not_take(wt, case):
    *shape, dtype = case
    check(wt, synth.make_inputs(*shape, dtype=dtype, seed=sum(shape) + 9))


@pytest.mark.parametrize("name", ["stage1", "stage2_f16"])
def test_full_size_workloads(wt, name):
    check(wt, synth.workload(name))


def test_no_bias_unaligned_pointers_and_determinism(wt):
    inp = synth.make_inputs(2, 4, 56, 56, 3, 5, seed=31, bias=False)
    d = to_dev(inp)
    for key in ("x", "dy"):  # one element past a 16-byte boundary: plain loads instead of box copies
        buf = torch.empty(d[key].numel() + 1, dtype=d[key].dtype, device="cuda")
        view = buf[1:].view_as(d[key])
        view.copy_(d[key])
        d[key] = view
    check(wt, inp, d)
    dx1, g1 = run_fused(wt, inp, d)
    dx2, g2 = run_fused(wt, inp, d)
    assert np.array_equal(dx1, dx2)
    for n in GRADS:
        if g1[n] is not None:
            assert np.array_equal(g1[n], g2[n]), n


def test_empty_batch_and_small_workspace(wt):
    inp = synth.make_inputs(2, 3, 16, 16, 2, 5, seed=3)
    d = to_dev(inp)
    e = {k: (v[:0] if k in ("x", "dy") else v) for k, v in d.items()}
    dx, g = wt.wtconv_bwd(e["x"], e["dy"], e["w_base"], e["b_base"], e["w_sub"], e["base_scale"],
                          e["wavelet_scale"], 2, 5)
    torch.cuda.synchronize()
    assert dx.numel() == 0
    for n in GRADS:
        assert torch.count_nonzero(g[n]) == 0, n
    with pytest.raises(wt.WtconvError) as err:
        wt.wtconv_bwd(d["x"], d["dy"], d["w_base"], d["b_base"], d["w_sub"], d["base_scale"], d["wavelet_scale"],
                      2, 5, workspace=torch.empty(256, dtype=torch.uint8, device="cuda"))
    assert err.value.status == wt.WTCONV_ERR_WORKSPACE
    check(wt, inp, d)  # the refusal launched nothing and left the context usable


def test_step_replays_from_a_cuda_graph(wt):
    # No call synchronises the host or allocates, so a whole step (forward +
    # fused backward) can be captured once and replayed, which is how small,
    # launch-bound layers are best run.  The replay must reproduce the eager
    # results bit for bit, on new inputs copied into the captured buffers.
    inp = synth.make_inputs(2, 32, 32, 32, 2, 5, seed=41)
    d = to_dev(inp)
    ps = [d[n] for n in ("w_base", "b_base", "w_sub", "base_scale", "wavelet_scale")]
    x, dy = d["x"].clone(), d["dy"].clone()
    y, dx = torch.empty_like(x), torch.empty_like(x)
    g = {n: torch.empty_like(p) for n, p in zip(GRADS, ps)}
    ws = torch.empty(max(wt.wtconv_workspace_size(wt.desc_for(x, 2, 5), wt.OP_BWD), 256), dtype=torch.uint8,
                     device="cuda")

    def step():
        wt.wtconv_fwd(x, *ps, 2, 5, y=y)
        wt.wtconv_bwd(x, dy, *ps, 2, 5, dx=dx, grads=g, workspace=ws)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    x.copy_(torch.flip(d["x"], dims=[3]))
    dy.copy_(torch.flip(d["dy"], dims=[2]))
    graph.replay()
    torch.cuda.synchronize()
    got = (y.clone(), dx.clone(), {n: t.clone() for n, t in g.items()})
    step()
    torch.cuda.synchronize()
    assert wt.wtconv_device_faults() == 0
    assert torch.equal(got[0], y) and torch.equal(got[1], dx)
    for n in GRADS:
        assert torch.equal(got[2][n], g[n]), n
