"""The give-up path of the kernels' bounded waits, exercised on the GPU
without a fault.

Every kernel that copies its planes asynchronously (box copies of float32
planes, bulk copies of 16-bit planes) waits for them on an mbarrier with a
time limit; a wait that runs out records itself in a device counter
(wtconv_device_faults), lets the copy land and makes the CTA leave.  The test
hook wtconv_test_copy_timeout arms each copy barrier with 16 bytes more than
the copy delivers and shortens the limit, so every such wait runs out: the
call must then complete, leave the context usable, and report the faults.
With the hook off, the same call on the same context must be correct again.
"""
import numpy as np
import pytest
import torch

import oracle
from memory_bound_cnn_wtconv2d_gb300 import synth

pytestmark = pytest.mark.gpu

TORCH_DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module")
def wt():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from memory_bound_cnn_wtconv2d_gb300 import build
    build.build()
    from memory_bound_cnn_wtconv2d_gb300 import wtconv
    return wtconv


def rel(a, b):
    a = np.asarray(a, np.float64)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


# (call, layer): whole-plane box copies (float32), bulk copies (16-bit), the
# fused backward, the separate parameter-gradient pass, and the windowed
# passes of planes beyond one CTA (box copies of the windows)
CASES = [
    ("fwd", (2, 4, 28, 28, 2, 5, "f32")),
    ("fwd", (2, 4, 28, 28, 2, 5, "f16")),
    ("bwd", (2, 4, 28, 28, 2, 5, "f32")),
    ("bwd_weight", (2, 4, 28, 28, 2, 5, "f32")),
    ("bwd_weight", (2, 4, 28, 28, 2, 5, "bf16")),
    ("fwd", (1, 2, 128, 128, 3, 5, "f32")),
    ("bwd_weight", (1, 2, 128, 128, 3, 5, "f32")),
]


def run(wt, call, inp):
    dt = TORCH_DT[inp.dtype]
    t = lambda a, d=torch.float32: None if a is None else torch.tensor(a, dtype=d, device="cuda")
    x, dy = t(inp.x, dt), t(inp.dy, dt)
    ps = [t(inp.w_base), t(inp.b_base), t(inp.w_sub), t(inp.base_scale), t(inp.wavelet_scale)]
    L, k = inp.levels, inp.k
    if call == "fwd":
        out = wt.wtconv_fwd(x, *ps, L, k)
    elif call == "bwd":
        out = wt.wtconv_bwd(x, dy, *ps, L, k)[0]
    else:
        out = wt.wtconv_bwd_weight(x, dy, *ps, L, k)["dw_sub"]
    return out


@pytest.mark.parametrize("call,layer", CASES, ids=lambda v: str(v))
def test_copy_wait_runs_out_and_the_context_stays_usable(wt, call, layer):
    inp = synth.make_inputs(*layer[:6], dtype=layer[6], seed=sum(layer[:6]))
    assert wt.wtconv_device_faults() == 0
    wt.wtconv_test_copy_timeout(True)
    try:
        run(wt, call, inp)
        torch.cuda.synchronize()  # the kernels returned: nothing hung, nothing faulted
    finally:
        wt.wtconv_test_copy_timeout(False)
    assert wt.wtconv_device_faults() > 0, "the waits that ran out were not reported"
    # the same call, normal limits, on the same context: correct again
    out = run(wt, call, inp)
    torch.cuda.synchronize()
    assert wt.wtconv_device_faults() == 0
    got = out.float().cpu().numpy()
    if call == "fwd":
        ref = oracle.fwd(inp)
    elif call == "bwd":
        ref = oracle.bwd(inp)["dx"]
    else:
        ref = oracle.bwd(inp)["dw_sub"]
    tol = {"f32": 1e-4, "f16": 2e-2, "bf16": 4e-2}[inp.dtype]
    assert rel(got, ref) <= tol
