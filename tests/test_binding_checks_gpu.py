"""The Python binding's buffer checks.

The library receives plain pointers, so the binding checks every size the
kernels rely on: outputs must match x in shape, dtype and device; parameters
and gradient buffers must be float32 with the element counts the layer
implies; the workspace must be a CUDA tensor.  Each mismatch below raises
before anything is launched, and a valid call afterwards still matches the
oracle.  Parameters may use any shape with the right element count (the
depthwise [C,1,k,k] layout gives the same result as [C,k,k]).
"""
import pytest
import torch

import oracle
from memory_bound_cnn_wtconv2d_gb300 import synth

from test_parity_gpu import GRADS, compare, to_dev, wt  # noqa: F401  (wt is a fixture)

PARAMS = ("w_base", "b_base", "w_sub", "base_scale", "wavelet_scale")


def _setup():
    inp = synth.make_inputs(2, 3, 16, 16, 2, 5, seed=77)
    d = to_dev(inp)
    return inp, d, [d[n] for n in PARAMS]


@pytest.mark.gpu
def test_mismatched_buffers_are_refused_before_launch(wt):
    inp, d, ps = _setup()
    x, dy = d["x"], d["dy"]
    L, k = inp.levels, inp.k

    def refused(fn, *a, **kw):
        with pytest.raises(ValueError):
            fn(*a, **kw)

    # outputs of the wrong shape, dtype or device
    refused(wt.wtconv_fwd, x, *ps, L, k, y=torch.empty(2, 3, 16, 15, device="cuda"))
    refused(wt.wtconv_fwd, x, *ps, L, k, y=torch.empty_like(x, dtype=torch.float16))
    refused(wt.wtconv_fwd, x, *ps, L, k, y=torch.empty_like(x, device="cpu"))
    refused(wt.wtconv_bwd_data, dy, ps[0], ps[2], ps[3], ps[4], L, k, dx=torch.empty(1, 3, 16, 16, device="cuda"))
    refused(wt.wtconv_bwd, x, dy, *ps, L, k, dx=torch.empty(2, 3, 16, 17, device="cuda"))
    # dy unlike x
    refused(wt.wtconv_bwd_weight, x, dy[:1], *ps, L, k)
    refused(wt.wtconv_bwd, x, dy.half(), *ps, L, k)
    # parameters with the wrong element count (levels or k unlike the tensors), dtype or device
    refused(wt.wtconv_fwd, x, *ps, L + 1, k)
    refused(wt.wtconv_fwd, x, *ps, L, k + 2)
    for i in range(5):
        bad = list(ps)
        bad[i] = ps[i][..., :-1].contiguous() if ps[i].dim() > 1 else ps[i][:-1].contiguous()
        refused(wt.wtconv_fwd, x, *bad, L, k)
        refused(wt.wtconv_bwd, x, dy, *bad, L, k)
        bad[i] = ps[i].double()
        refused(wt.wtconv_bwd_weight, x, dy, *bad, L, k)
        bad[i] = ps[i].cpu()
        refused(wt.wtconv_fwd, x, *bad, L, k)
    # gradient buffers: missing, short, wrong dtype
    g = {n: torch.empty_like(p) for n, p in zip(GRADS, ps)}
    for n in GRADS:
        refused(wt.wtconv_bwd, x, dy, *ps, L, k, grads={m: t for m, t in g.items() if m != n})
        refused(wt.wtconv_bwd_weight, x, dy, *ps, L, k, grads=dict(g, **{n: g[n].flatten()[:-1]}))
        refused(wt.wtconv_bwd_weight_noalloc, x, dy, *ps, L, k, grads=dict(g, **{n: g[n].half()}))
    # a workspace that is not device memory
    need = wt.wtconv_workspace_size(wt.desc_for(x, L, k), wt.OP_BWD)
    refused(wt.wtconv_bwd, x, dy, *ps, L, k, workspace=torch.empty(need, dtype=torch.uint8))
    refused(wt.wtconv_bwd_weight, x, dy, *ps, L, k, workspace=torch.empty(need, dtype=torch.uint8))

    # nothing was launched; a valid call still matches the oracle
    torch.cuda.synchronize()
    assert wt.wtconv_device_faults() == 0
    y = wt.wtconv_fwd(x, *ps, L, k)
    dx, gr = wt.wtconv_bwd(x, dy, *ps, L, k, grads=g)
    torch.cuda.synchronize()
    assert gr is g
    compare("y", y.cpu().numpy(), oracle.fwd(inp), "f32", False)
    ref = oracle.bwd(inp)
    compare("dx", dx.cpu().numpy(), ref["dx"], "f32", False)
    for n in GRADS:
        compare(n, g[n].cpu().numpy(), ref[n], "f32", True)


@pytest.mark.gpu
def test_depthwise_weight_layout_and_bias_free_gradient(wt):
    inp, d, ps = _setup()
    x, dy = d["x"], d["dy"]
    L, k = inp.levels, inp.k
    C = x.shape[1]
    w4 = ps[0].view(C, 1, k, k)  # the layout of a depthwise nn.Conv2d weight
    assert torch.equal(wt.wtconv_fwd(x, w4, *ps[1:], L, k), wt.wtconv_fwd(x, *ps, L, k))
    # without a bias, a db_base buffer that is given receives s_base * sum(dy)
    g = {n: torch.full_like(p, float("nan")) for n, p in zip(GRADS, ps)}
    wt.wtconv_bwd_weight(x, dy, ps[0], None, *ps[2:], L, k, grads=g)
    g2 = wt.wtconv_bwd_weight(x, dy, ps[0], None, *ps[2:], L, k)
    torch.cuda.synchronize()
    assert g2["db_base"] is None
    expect = ps[3] * dy.double().sum(dim=(0, 2, 3)).float()
    torch.testing.assert_close(g["db_base"], expect, rtol=1e-5, atol=1e-5)
    for n in ("dw_base", "dw_sub", "dbase_scale", "dwavelet_scale"):
        assert torch.equal(g[n], g2[n]), n


def test_host_tensors_are_refused_without_a_device():
    # runs anywhere: host tensors never reach the library
    from memory_bound_cnn_wtconv2d_gb300 import wtconv
    inp = synth.make_inputs(1, 2, 8, 8, 1, 3, seed=5)
    t = {n: None if a is None else torch.tensor(a) for n, a in
         (("x", inp.x), ("dy", inp.dy), *((n, getattr(inp, n)) for n in PARAMS))}
    ps = [t[n] for n in PARAMS]
    for call in (lambda: wtconv.wtconv_fwd(t["x"], *ps, 1, 3),
                 lambda: wtconv.wtconv_bwd_data(t["dy"], ps[0], ps[2], ps[3], ps[4], 1, 3),
                 lambda: wtconv.wtconv_bwd_weight(t["x"], t["dy"], *ps, 1, 3),
                 lambda: wtconv.wtconv_bwd(t["x"], t["dy"], *ps, 1, 3)):
        with pytest.raises(ValueError, match="CUDA"):
            call()
