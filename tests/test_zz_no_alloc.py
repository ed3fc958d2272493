"""The parameter-gradient entry point that allocates nothing.

wtconv_bwd_weight_noalloc serves callers that cannot allocate device memory
(a plugin inside an application that owns the device-memory budget, or a
caller that must not risk cudaMalloc's device synchronisation): it uses the
library's built-in 4 MiB device scratch instead of a caller workspace.
These tests call it through the C ABI and check it against the regular
wtconv_bwd_weight on calls in a row with different layers (so each later
call runs on the scratch contents left by the one before).  Both calls run
the same kernels and add the partial sums in the same fixed order, so the
results must agree bit for bit; a stale partial sum left in the scratch
would show up as a difference.  This file is named to be collected last.
"""
import ctypes

import pytest
import torch

from memory_bound_cnn_wtconv2d_gb300 import build, synth, wtconv

GRADS = ("dw_base", "db_base", "dw_sub", "dbase_scale", "dwavelet_scale")


def test_rejects_layers_beyond_the_static_scratch():
    # validated on the host before any device work: a layer whose partial
    # sums exceed 4 MiB is refused with a message naming the sizes
    build.build()
    L = wtconv.lib()
    d = wtconv.make_desc(4, 65536, 8, 8, 3, 9, 0)
    assert L.wtconv_workspace_size(ctypes.byref(d), wtconv.OP_BWD_WEIGHT) > (4 << 20)
    p = ctypes.c_void_p(0x10000)
    rc = L.wtconv_bwd_weight_noalloc(ctypes.byref(d), p, p, p, None, p, p, p, p, None, p, p, p, None)
    assert rc == wtconv.WTCONV_ERR_UNSUPPORTED
    assert "static scratch" in L.wtconv_last_error().decode()


def _dev(inp):
    dt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[inp.dtype]
    t = lambda a, d=torch.float32: None if a is None else torch.tensor(a, dtype=d, device="cuda")
    return dict(x=t(inp.x, dt), dy=t(inp.dy, dt), w_base=t(inp.w_base), b_base=t(inp.b_base),
                w_sub=t(inp.w_sub), base_scale=t(inp.base_scale), wavelet_scale=t(inp.wavelet_scale))


@pytest.mark.gpu
def test_noalloc_matches_workspace_call_twice_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    layers = [synth.make_inputs(16, 24, 28, 28, 3, 5, dtype="f32", seed=71),   # larger record set first
              synth.make_inputs(5, 6, 13, 11, 2, 3, dtype="f16", seed=72, bias=False),
              synth.make_inputs(32, 24, 28, 28, 3, 5, dtype="f32", seed=74),
              # planes beyond one CTA: the windowed planner, right after a larger record set
              synth.make_inputs(1, 4, 128, 128, 3, 5, dtype="f32", seed=73)]
    for inp in layers:
        d = _dev(inp)
        args = (d["x"], d["dy"], d["w_base"], d["b_base"], d["w_sub"], d["base_scale"], d["wavelet_scale"],
                inp.levels, inp.k)
        ref = wtconv.wtconv_bwd_weight(*args)
        got = wtconv.wtconv_bwd_weight_noalloc(*args)
        torch.cuda.synchronize()
        assert wtconv.wtconv_device_faults() == 0
        for name in GRADS:
            if ref[name] is None:
                assert got[name] is None
                continue
            assert torch.isfinite(got[name]).all(), name
            assert torch.equal(got[name], ref[name]), f"{name}: differs from the workspace call"
