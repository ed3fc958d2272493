"""GPU parity of layers computed as a fine pass plus a coarse layer, against
the float64 oracle.

A layer whose tile window does not fit one CTA (a large plane with a deep
pyramid and a wide kernel: a halo of 2^L * (k/2) pixels) runs levels 1..s and
the base convolution on the full planes, and levels s+1..L as a layer of
their own on the level-s low-pass planes (block sums over 2^s x 2^s), whose
output is added back replicated over each block.  In the collapsed synthesis
a pixel takes level l's coefficient at (i >> l, j >> l) with the sign bits of
(i >> (l-1), j >> (l-1)); for l > s those are bits of (i >> s, j >> s), which
is what makes the split exact up to rounding.

Each case is checked three ways:
  - every output of every pass against the oracle (tolerances of the
    whole-plane tests), and each level of dw_sub and dwavelet_scale on its own,
    so that a wrong coarse level cannot hide behind the larger fine ones;
  - the coarse part alone: the base kernels and the fine levels' kernels set
    to zero, so y and dx are the coarse layer's contribution only;
  - the one-call backward (wtconv_bwd) against the two separate calls.
"""
import numpy as np
import pytest
import torch

import oracle
from memory_bound_cnn_wtconv2d_gb300 import synth

from test_parity_gpu import GRADS, compare, to_dev, wt  # noqa: F401  (wt is a fixture)

pytestmark = pytest.mark.gpu

# (N, C, H, W, L, k, dtype).  The fine pass takes the deepest level count
# whose tile window fits one CTA: 4 at k = 5..9, 5 at k = 3, 3 for 16-bit
# k = 9 (the comments give the split each case exercises).
CASES = [
    (1, 2, 128, 128, 5, 5, "f32"),    # the 64-pixel halo case: split at 4
    (2, 1, 130, 136, 5, 7, "f32"),    # ragged: odd block counts at the coarse levels
    (1, 2, 160, 152, 6, 3, "f16"),    # k = 3: split at 5
    (1, 2, 96, 100, 5, 9, "bf16"),    # whole-plane forward, split parameter gradient
    (1, 1, 224, 224, 8, 5, "f32"),    # deepest pyramid: a 4-level coarse layer on 14 x 14 planes
    (1, 1, 1024, 1024, 8, 9, "f16"),  # the coarse layer splits again
]


def ids(case):
    return "x".join(map(str, case))


def run_all(wt, inp, d):
    L, k = inp.levels, inp.k
    y = wt.wtconv_fwd(d["x"], d["w_base"], d["b_base"], d["w_sub"], d["base_scale"], d["wavelet_scale"], L, k)
    dx = wt.wtconv_bwd_data(d["dy"], d["w_base"], d["w_sub"], d["base_scale"], d["wavelet_scale"], L, k)
    g = wt.wtconv_bwd_weight(d["x"], d["dy"], d["w_base"], d["b_base"], d["w_sub"], d["base_scale"],
                             d["wavelet_scale"], L, k)
    dx2, g2 = wt.wtconv_bwd(d["x"], d["dy"], d["w_base"], d["b_base"], d["w_sub"], d["base_scale"],
                            d["wavelet_scale"], L, k)
    torch.cuda.synchronize()
    assert wt.wtconv_device_faults() == 0, "an in-kernel bounded wait gave up"
    return y, dx, g, dx2, g2


@pytest.mark.parametrize("case", CASES, ids=ids)
def test_split_layer_matches_oracle(wt, case):
    N, C, H, W, L, k, dtype = case
    inp = synth.make_inputs(N, C, H, W, L, k, dtype=dtype, seed=H + 3 * W + 5 * L + k)
    d = to_dev(inp)
    y, dx, g, dx2, g2 = run_all(wt, inp, d)
    y_ref = oracle.fwd(inp)
    ref = oracle.bwd(inp)
    compare("y", y.float().cpu().numpy(), y_ref, dtype, False)
    compare("dx", dx.float().cpu().numpy(), ref["dx"], dtype, False)
    for name in GRADS:
        compare(name, g[name].cpu().numpy(), ref[name], dtype, True)
    # every level of the wavelet-kernel and wavelet-scale gradients on its own
    for l in range(L):
        compare(f"dw_sub[{l}]", g["dw_sub"][l].cpu().numpy(), ref["dw_sub"][l], dtype, True)
        compare(f"dwavelet_scale[{l}]", g["dwavelet_scale"][l].cpu().numpy(), ref["dwavelet_scale"][l], dtype, True)
    # the one-call backward runs the same two passes
    assert torch.equal(dx2, dx)
    for name in GRADS:
        assert torch.equal(g2[name], g[name]), name


@pytest.mark.parametrize("case", CASES[:4], ids=ids)
def test_coarse_part_alone(wt, case):
    # base kernels and levels 1..L-1 zeroed: y and dx come from the deepest
    # level only, which every split above computes in its coarse layer
    N, C, H, W, L, k, dtype = case
    inp = synth.make_inputs(N, C, H, W, L, k, dtype=dtype, seed=7 * H + W + L, bias=False)
    inp.w_base[:] = 0
    inp.w_sub[:L - 1] = 0
    d = to_dev(inp)
    y = wt.wtconv_fwd(d["x"], d["w_base"], None, d["w_sub"], d["base_scale"], d["wavelet_scale"], L, k)
    dx = wt.wtconv_bwd_data(d["dy"], d["w_base"], d["w_sub"], d["base_scale"], d["wavelet_scale"], L, k)
    torch.cuda.synchronize()
    y_ref = oracle.fwd(inp)
    assert np.abs(y_ref).max() > 0
    compare("y", y.float().cpu().numpy(), y_ref, dtype, False)
    compare("dx", dx.float().cpu().numpy(), oracle.bwd(inp)["dx"], dtype, False)


def test_split_layer_empty_batch(wt):
    inp = synth.make_inputs(0, 2, 128, 128, 5, 5, seed=3)
    d = to_dev(inp)
    y = wt.wtconv_fwd(d["x"], d["w_base"], d["b_base"], d["w_sub"], d["base_scale"], d["wavelet_scale"], 5, 5)
    dx = wt.wtconv_bwd_data(d["dy"], d["w_base"], d["w_sub"], d["base_scale"], d["wavelet_scale"], 5, 5)
    g = wt.wtconv_bwd_weight(d["x"], d["dy"], d["w_base"], d["b_base"], d["w_sub"], d["base_scale"],
                             d["wavelet_scale"], 5, 5)
    torch.cuda.synchronize()
    assert y.numel() == 0 and dx.numel() == 0
    for name in GRADS:
        assert torch.count_nonzero(g[name]) == 0, name


def test_split_needs_its_workspace(wt):
    # the forward of a split layer takes a workspace; a caller's that is too
    # small is refused before anything is launched
    inp = synth.make_inputs(1, 2, 128, 128, 5, 5, seed=5)
    d = to_dev(inp)
    desc = wt.desc_for(d["x"], 5, 5)
    need = wt.wtconv_workspace_size(desc, wt.OP_FWD)
    assert need > 0
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(wt.WtconvError) as e:
        wt.wtconv_fwd(d["x"], d["w_base"], d["b_base"], d["w_sub"], d["base_scale"], d["wavelet_scale"], 5, 5,
                      workspace=small)
    assert e.value.status == wt.WTCONV_ERR_WORKSPACE
    enough = torch.empty(need, dtype=torch.uint8, device="cuda")
    y = wt.wtconv_fwd(d["x"], d["w_base"], d["b_base"], d["w_sub"], d["base_scale"], d["wavelet_scale"], 5, 5,
                      workspace=enough)
    torch.cuda.synchronize()
    compare("y", y.cpu().numpy(), oracle.fwd(inp), "f32", False)


def test_split_step_replays_from_a_cuda_graph(wt):
    # The split calls enqueue a memset, small element-wise kernels and the
    # fine and coarse layers' kernels on the caller's stream, nothing else:
    # a whole step on caller-owned workspaces captures into a CUDA graph and
    # replays bit for bit (new inputs copied into the captured buffers).
    inp = synth.make_inputs(1, 2, 128, 128, 5, 5, seed=43)
    d = to_dev(inp)
    ps = [d[n] for n in ("w_base", "b_base", "w_sub", "base_scale", "wavelet_scale")]
    x, dy = d["x"].clone(), d["dy"].clone()
    y, dx = torch.empty_like(x), torch.empty_like(x)
    g = {n: torch.empty_like(p) for n, p in zip(GRADS, ps)}
    desc = wt.desc_for(x, 5, 5)
    wsf = torch.empty(wt.wtconv_workspace_size(desc, wt.OP_FWD), dtype=torch.uint8, device="cuda")
    wsb = torch.empty(wt.wtconv_workspace_size(desc, wt.OP_BWD), dtype=torch.uint8, device="cuda")

    def step():
        wt.wtconv_fwd(x, *ps, 5, 5, y=y, workspace=wsf)
        wt.wtconv_bwd(x, dy, *ps, 5, 5, dx=dx, grads=g, workspace=wsb)

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


def test_split_layer_through_the_no_alloc_entry_point(wt):
    # the no-alloc entry point takes split layers whose scratch fits its
    # 4 MiB array, with the same results bit for bit
    inp = synth.make_inputs(1, 2, 128, 128, 5, 5, seed=47)
    d = to_dev(inp)
    ps = [d[n] for n in ("w_base", "b_base", "w_sub", "base_scale", "wavelet_scale")]
    assert wt.wtconv_workspace_size(wt.desc_for(d["x"], 5, 5), wt.OP_BWD_WEIGHT) <= 4 << 20
    ref = wt.wtconv_bwd_weight(d["x"], d["dy"], *ps, 5, 5)
    got = wt.wtconv_bwd_weight_noalloc(d["x"], d["dy"], *ps, 5, 5)
    torch.cuda.synchronize()
    assert wt.wtconv_device_faults() == 0
    for n in GRADS:
        assert torch.equal(got[n], ref[n]), n


@pytest.mark.parametrize("which", ["both", "input_only", "params_only"])
def test_split_layer_through_the_autograd_module(wt, which):
    # the module's forward and each of its backward paths (one fused call, or
    # the input / parameter gradient alone) size their workspaces for a split
    from memory_bound_cnn_wtconv2d_gb300.layer import WTConv2d
    torch.manual_seed(1)
    m = WTConv2d(2, kernel_size=5, levels=5, device="cuda")
    x = torch.randn(1, 2, 136, 128, device="cuda", requires_grad=which != "params_only")
    if which == "input_only":
        for p in m.parameters():
            p.requires_grad_(False)
    y = m(x)
    dy = torch.randn_like(y)
    y.backward(dy)
    torch.cuda.synchronize()
    assert wt.wtconv_device_faults() == 0
    inp = synth.make_inputs(1, 2, 136, 128, 5, 5)
    inp.x = x.detach().cpu().numpy()
    inp.dy = dy.cpu().numpy()
    inp.w_base = m.weight.detach().cpu().numpy()
    inp.b_base = m.bias.detach().cpu().numpy()
    inp.w_sub = m.wavelet_weight.detach().cpu().numpy()
    inp.base_scale = m.base_scale.detach().cpu().numpy()
    inp.wavelet_scale = m.wavelet_scale.detach().cpu().numpy()
    compare("y", y.detach().cpu().numpy(), oracle.fwd(inp), "f32", False)
    g = oracle.bwd(inp)
    if which != "params_only":
        compare("dx", x.grad.cpu().numpy(), g["dx"], "f32", False)
    if which != "input_only":
        compare("dw_base", m.weight.grad.cpu().numpy(), g["dw_base"], "f32", True)
        compare("dw_sub", m.wavelet_weight.grad.cpu().numpy(), g["dw_sub"], "f32", True)
        compare("dwavelet_scale", m.wavelet_scale.grad.cpu().numpy(), g["dwavelet_scale"], "f32", True)
