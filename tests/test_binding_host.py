"""The Python binding's marshalling, checked on the host (CPU only).

A fake library stands in for libwtconv.so and records each call, and host
tensors stand in for device memory, so every entry point of the binding runs
without a GPU.  The tests check that the pointers, sizes and descriptor reach
the C calls in the order include/wtconv.h declares them (the prototypes are
parsed from the header), and that the binding's refusals -- sizes the layer
does not imply, outputs overlapping inputs or one another -- happen before
anything reaches the library.
"""
import ctypes
import os
import re

import pytest
import torch

from memory_bound_cnn_wtconv2d_gb300 import synth, wtconv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_params():
    """Parameter names of each wtconv_* prototype in include/wtconv.h."""
    with open(os.path.join(ROOT, "include", "wtconv.h")) as f:
        text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    out = {}
    for m in re.finditer(r"\b(wtconv_\w+)\s*\(([^;{]*?)\)\s*;", text):
        args = [a.strip() for a in m.group(2).split(",") if a.strip() and a.strip() != "void"]
        out[m.group(1)] = [re.findall(r"\w+", a)[-1] for a in args]
    return out


class FakeLib:
    def __init__(self):
        self.calls = []
        self.current = None  # the device the binding made current, as the library would see it

    def _record(name):
        def call(self, *args):
            self.calls.append((name, args))
            self.devices.append(self.current)
            return 0
        return call

    devices = None

    wtconv_fwd = _record("wtconv_fwd")
    wtconv_bwd_data = _record("wtconv_bwd_data")
    wtconv_bwd_weight = _record("wtconv_bwd_weight")
    wtconv_bwd = _record("wtconv_bwd")
    wtconv_bwd_weight_noalloc = _record("wtconv_bwd_weight_noalloc")

    fwd_ws = 0  # forward / input-gradient workspace: none, as for every layer that needs no split

    def wtconv_workspace_size(self, desc, op):
        return self.fwd_ws if op in (wtconv.OP_FWD, wtconv.OP_BWD_DATA) else 4096


@pytest.fixture
def fake(monkeypatch):
    import contextlib
    lib = FakeLib()
    lib.devices = []

    @contextlib.contextmanager
    def device_ctx(device):  # records the device made current around each call
        prev, lib.current = lib.current, device
        try:
            yield
        finally:
            lib.current = prev

    monkeypatch.setattr(wtconv, "_LIB", lib)
    monkeypatch.setattr(wtconv, "_FWD_WS", {})
    monkeypatch.setattr(wtconv, "_on_cuda", lambda t: True)
    monkeypatch.setattr(wtconv, "_device_ctx", device_ctx)
    return lib


def layer(bias=True):
    inp = synth.make_inputs(2, 3, 10, 12, 2, 5, seed=4, bias=bias)
    t = lambda a: None if a is None else torch.tensor(a)
    return inp, t(inp.x), t(inp.dy), [t(getattr(inp, n)) for n in wtconv.PARAM_NAMES]


def ptr(a):
    v = a.value if isinstance(a, ctypes.c_void_p) else a
    return v or None


def address(t):
    return None if t is None else t.data_ptr()


def check_call(call, name, expect):
    """expect: parameter name -> tensor / int / None, for every parameter but desc and stream."""
    got_name, args = call
    assert got_name == name
    params = header_params()[name]
    assert len(args) == len(params), (name, len(args), params)
    desc = args[0]._obj
    assert params[0] == "desc" and params[-1] == "stream"
    for pname, a in zip(params[1:-1], args[1:-1]):
        want = expect[pname]
        if isinstance(want, int) and not isinstance(want, bool):
            assert a == want, (name, pname)
        else:
            assert ptr(a) == address(want), (name, pname)
    return desc


def test_header_prototypes_match_the_binding():
    p = header_params()
    for name in ("wtconv_fwd", "wtconv_bwd_data", "wtconv_bwd_weight", "wtconv_bwd", "wtconv_bwd_weight_noalloc"):
        assert name in p and name in wtconv.EXPORTS


def test_arguments_reach_the_library_in_header_order(fake):
    inp, x, dy, ps = layer()
    wb, bb, wsub, sb, sw = ps
    y = torch.empty_like(x)
    wtconv.wtconv_fwd(x, *ps, 2, 5, y=y, stream=0)
    desc = check_call(fake.calls[-1], "wtconv_fwd",
                      dict(x=x, w_base=wb, b_base=bb, w_sub=wsub, base_scale=sb, wavelet_scale=sw, y=y, ws=None,
                           ws_bytes=0))
    assert (desc.N, desc.C, desc.H, desc.W, desc.levels, desc.k, desc.dtype) == (2, 3, 10, 12, 2, 5, 0)
    dx = torch.empty_like(x)
    wtconv.wtconv_bwd_data(dy, wb, wsub, sb, sw, 2, 5, dx=dx, stream=0)
    check_call(fake.calls[-1], "wtconv_bwd_data",
               dict(dy=dy, w_base=wb, w_sub=wsub, base_scale=sb, wavelet_scale=sw, dx=dx, ws=None, ws_bytes=0))
    g = {n: torch.empty_like(p) for n, p in zip(wtconv.GRAD_NAMES, ps)}
    ws = torch.empty(1000, dtype=torch.float32)  # bytes = numel * element size
    wtconv.wtconv_bwd_weight(x, dy, *ps, 2, 5, grads=g, workspace=ws, stream=0)
    grads = dict(dw_base=g["dw_base"], db_base=g["db_base"], dw_sub=g["dw_sub"], dbase_scale=g["dbase_scale"],
                 dwavelet_scale=g["dwavelet_scale"])
    common = dict(x=x, dy=dy, w_base=wb, b_base=bb, w_sub=wsub, base_scale=sb, wavelet_scale=sw, **grads)
    check_call(fake.calls[-1], "wtconv_bwd_weight", dict(common, ws=ws, ws_bytes=4000))
    dx2, g2 = wtconv.wtconv_bwd(x, dy, *ps, 2, 5, dx=dx, grads=g, workspace=ws, stream=0)
    assert dx2 is dx and g2 is g
    check_call(fake.calls[-1], "wtconv_bwd", dict(common, dx=dx, ws=ws, ws_bytes=4000))
    wtconv.wtconv_bwd_weight_noalloc(x, dy, *ps, 2, 5, grads=g, stream=0)
    check_call(fake.calls[-1], "wtconv_bwd_weight_noalloc", common)
    # a workspace the binding allocates has the size the library asked for
    wtconv.wtconv_bwd(x, dy, *ps, 2, 5, stream=0)
    assert fake.calls[-1][1][-2] == 4096


def test_every_call_runs_with_the_tensors_device_current(fake):
    # the library launches on the current device, so the binding makes the
    # activations' device current around every call (and the workspace query)
    inp, x, dy, ps = layer()
    wtconv.wtconv_fwd(x, *ps, 2, 5, stream=0)
    wtconv.wtconv_bwd_data(dy, ps[0], ps[2], ps[3], ps[4], 2, 5, stream=0)
    wtconv.wtconv_bwd_weight(x, dy, *ps, 2, 5, stream=0)
    wtconv.wtconv_bwd(x, dy, *ps, 2, 5, stream=0)
    wtconv.wtconv_bwd_weight_noalloc(x, dy, *ps, 2, 5, stream=0)
    assert len(fake.devices) == 5 and all(d == x.device for d in fake.devices)
    assert fake.current is None  # restored after each call


def test_no_bias_and_depthwise_weight_layout(fake):
    inp, x, dy, ps = layer(bias=False)
    wb, bb, wsub, sb, sw = ps
    assert bb is None
    wtconv.wtconv_fwd(x, wb.view(3, 1, 5, 5), None, wsub, sb, sw, 2, 5, stream=0)
    assert ptr(fake.calls[-1][1][3]) is None  # b_base
    g = wtconv.wtconv_bwd_weight(x, dy, *ps, 2, 5, stream=0)
    assert g["db_base"] is None and ptr(fake.calls[-1][1][9]) is None


def test_refusals_reach_nothing(fake):
    inp, x, dy, ps = layer()
    wb, bb, wsub, sb, sw = ps
    g = {n: torch.empty_like(p) for n, p in zip(wtconv.GRAD_NAMES, ps)}
    ws = torch.empty(4096, dtype=torch.uint8)
    n = x.numel()
    big = torch.empty(2 * n)  # views of one buffer: overlapping, or adjacent
    cases = [
        # outputs overlapping inputs
        lambda: wtconv.wtconv_fwd(x, *ps, 2, 5, y=x, stream=0),
        lambda: wtconv.wtconv_fwd(big[:n].view_as(x), *ps, 2, 5, y=big[n - 7:2 * n - 7].view_as(x), stream=0),
        lambda: wtconv.wtconv_bwd_data(dy, wb, wsub, sb, sw, 2, 5, dx=dy, stream=0),
        lambda: wtconv.wtconv_bwd(x, dy, *ps, 2, 5, dx=dy, grads=g, workspace=ws, stream=0),
        lambda: wtconv.wtconv_bwd(x, dy, *ps, 2, 5, grads=dict(g, dw_base=wb), workspace=ws, stream=0),
        lambda: wtconv.wtconv_bwd_weight(x, dy, *ps, 2, 5, grads=g, workspace=x.view(torch.uint8), stream=0),
        lambda: wtconv.wtconv_bwd_weight_noalloc(x, dy, *ps, 2, 5, grads=dict(g, dwavelet_scale=sw), stream=0),
        # outputs overlapping one another
        lambda: wtconv.wtconv_bwd(x, dy, *ps, 2, 5, grads=g, workspace=g["dw_sub"].view(torch.uint8), stream=0),
        lambda: wtconv.wtconv_bwd(x, dy, *ps, 2, 5, dx=torch.empty_like(x),
                                  grads=dict(g, dbase_scale=g["db_base"]), workspace=ws, stream=0),
        # sizes the layer does not imply
        lambda: wtconv.wtconv_fwd(x, *ps, 2, 5, y=torch.empty(2, 3, 10, 11), stream=0),
        lambda: wtconv.wtconv_fwd(x, *ps, 3, 5, stream=0),
        lambda: wtconv.wtconv_bwd(x, dy[:1], *ps, 2, 5, stream=0),
        lambda: wtconv.wtconv_bwd_weight(x, dy, *ps, 2, 5, grads=dict(g, dw_sub=g["dw_sub"][:1]), stream=0),
        lambda: wtconv.wtconv_bwd_weight(x, dy, wb.double(), *ps[1:], 2, 5, stream=0),
        # an activation type the library does not take
        lambda: wtconv.wtconv_fwd(x.double(), *ps, 2, 5, stream=0),
    ]
    for i, case in enumerate(cases):
        with pytest.raises(ValueError):
            case()
        assert fake.calls == [], f"case {i} reached the library"
    # adjacent, disjoint views of one buffer are accepted
    wtconv.wtconv_fwd(big[:n].view_as(x), *ps, 2, 5, y=big[n:].view_as(x), stream=0)
    assert len(fake.calls) == 1


def test_layer_workspace_cache_is_reused_and_bounded(monkeypatch):
    from memory_bound_cnn_wtconv2d_gb300 import layer as layer_mod

    class Stream:
        cuda_stream = 7

    monkeypatch.setattr(torch.cuda, "current_stream", lambda device=None: Stream())
    import contextlib
    monkeypatch.setattr(wtconv, "_device_ctx", lambda device: contextlib.nullcontext())
    monkeypatch.setattr(wtconv, "wtconv_workspace_size", lambda desc, op: 1000 + desc.N)
    monkeypatch.setattr(layer_mod, "_WORKSPACES", type(layer_mod._WORKSPACES)())
    first = torch.empty(1, 3, 8, 8)
    ws = layer_mod._workspace(first, 2, 5, wtconv.OP_BWD)
    assert ws.numel() == 1001 and ws.dtype == torch.uint8
    assert layer_mod._workspace(first, 2, 5, wtconv.OP_BWD) is ws  # reused, not reallocated
    assert layer_mod._workspace(first, 2, 5, wtconv.OP_BWD_WEIGHT) is not ws  # one per call kind
    for n in range(2, 2 + 3 * layer_mod.MAX_WORKSPACES):  # many batch sizes
        layer_mod._workspace(torch.empty(n, 3, 8, 8), 2, 5, wtconv.OP_BWD)
        assert layer_mod._workspace(first, 2, 5, wtconv.OP_BWD) is ws  # kept while in use
    assert len(layer_mod._WORKSPACES) == layer_mod.MAX_WORKSPACES


def test_module_checks_its_hyperparameters_at_construction():
    from memory_bound_cnn_wtconv2d_gb300.layer import WTConv2d
    m = WTConv2d(4, kernel_size=5, levels=3)
    assert m.weight.shape == (4, 5, 5) and m.wavelet_weight.shape == (3, 16, 5, 5)
    assert m.wavelet_scale.shape == (3, 16) and m.bias.shape == (4,)
    assert "kernel_size=5" in repr(m) and "levels=3" in repr(m)
    assert WTConv2d(2, kernel_size=9, levels=8, bias=False).bias is None
    for kw in (dict(kernel_size=4), dict(kernel_size=11), dict(kernel_size=1), dict(levels=0), dict(levels=9)):
        with pytest.raises(ValueError):
            WTConv2d(4, **kw)
    with pytest.raises(ValueError):
        WTConv2d(0)


def test_split_layers_get_a_forward_workspace(fake):
    # a layer computed as a fine pass plus a coarse layer needs a workspace in
    # the forward and input-gradient calls too: the binding sizes it from the
    # library and passes it (or the caller's) with its byte count
    fake.fwd_ws = 5000
    inp, x, dy, ps = layer()
    wb, bb, wsub, sb, sw = ps
    wtconv.wtconv_fwd(x, *ps, 2, 5, stream=0)
    args = fake.calls[-1][1]
    assert ptr(args[8]) is not None and args[9] == 5000
    wtconv.wtconv_bwd_data(dy, wb, wsub, sb, sw, 2, 5, stream=0)
    args = fake.calls[-1][1]
    assert ptr(args[7]) is not None and args[8] == 5000
    own = torch.empty(6000, dtype=torch.uint8)
    wtconv.wtconv_fwd(x, *ps, 2, 5, stream=0, workspace=own)
    args = fake.calls[-1][1]
    assert ptr(args[8]) == own.data_ptr() and args[9] == 6000
    with pytest.raises(ValueError):  # a workspace may not overlap an input
        wtconv.wtconv_bwd_data(dy, wb, wsub, sb, sw, 2, 5, stream=0, workspace=dy.view(torch.uint8))
