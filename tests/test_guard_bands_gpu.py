"""Guard-band checks of every GPU entry point (the memory check this pool
allows in place of a sanitizer).

Every output, gradient and workspace buffer is placed inside a larger
allocation whose margins before and after it hold a canary bit pattern; the
inputs are snapshotted.  After each call the margins must still hold the
canary (no write outside a buffer) and the inputs must be unchanged (no write
to a read-only argument).  The layers cover whole planes, windowed planes,
the fused backward and its fallback, float32 and 16-bit activations, and
buffers one element off a 16-byte boundary (the scalar paths).
"""
import pytest
import torch

from memory_bound_cnn_wtconv2d_gb300 import synth

from test_parity_gpu import GRADS, to_dev, wt  # noqa: F401  (wt is a fixture)

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes of canary before and after each buffer


class Guarded:
    """A tensor view inside a canary-filled allocation."""

    def __init__(self, shape, dtype, misalign=0):
        es = torch.empty((), dtype=dtype).element_size()
        n = 1
        for s in shape:
            n *= s
        self.lead = GUARD + misalign * es
        total = self.lead + n * es + GUARD
        self.raw = torch.empty(total, dtype=torch.uint8, device="cuda")
        self.raw.fill_(0xA5)
        self.view = self.raw[self.lead:self.lead + n * es].view(dtype).view(shape)
        self.n_bytes = n * es

    def intact(self):
        head = self.raw[:self.lead]
        tail = self.raw[self.lead + self.n_bytes:]
        return bool((head == 0xA5).all()) and bool((tail == 0xA5).all())


def guarded_like(t, misalign=0):
    return Guarded(tuple(t.shape), t.dtype, misalign)


CASES = [  # (N, C, H, W, L, k, dtype, misalign)
    (2, 3, 13, 17, 3, 5, "f32", 0), (2, 4, 56, 56, 3, 5, "f32", 0), (3, 4, 28, 28, 2, 5, "f16", 0),
    (9, 6, 7, 7, 2, 5, "bf16", 0), (2, 2, 40, 40, 1, 7, "f32", 1), (2, 3, 16, 16, 2, 5, "f16", 1),
    (1, 2, 130, 124, 2, 5, "f32", 0), (1, 2, 120, 120, 3, 5, "bf16", 0), (1, 2, 113, 129, 3, 5, "f32", 1),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_no_write_outside_outputs_and_inputs_untouched(wt, case):
    N, C, H, W, L, k, dtype, mis = case
    inp = synth.make_inputs(N, C, H, W, L, k, dtype=dtype, seed=N + C + H + W + L + k)
    d = to_dev(inp)
    ps = [d[n] for n in ("w_base", "b_base", "w_sub", "base_scale", "wavelet_scale")]
    snap = {n: t.clone() for n, t in d.items() if t is not None}
    desc = wt.desc_for(d["x"], L, k)
    ws_bytes = max(wt.wtconv_workspace_size(desc, wt.OP_BWD), wt.wtconv_workspace_size(desc, wt.OP_BWD_WEIGHT), 256)
    y, dx, dx2 = guarded_like(d["x"], mis), guarded_like(d["x"], mis), guarded_like(d["x"], mis)
    g1 = {n: guarded_like(p) for n, p in zip(GRADS, ps)}
    g2 = {n: guarded_like(p) for n, p in zip(GRADS, ps)}
    ws1, ws2 = Guarded((ws_bytes,), torch.uint8), Guarded((ws_bytes,), torch.uint8)
    wt.wtconv_fwd(d["x"], *ps, L, k, y=y.view)
    wt.wtconv_bwd_data(d["dy"], ps[0], ps[2], ps[3], ps[4], L, k, dx=dx.view)
    wt.wtconv_bwd_weight(d["x"], d["dy"], *ps, L, k, grads={n: g.view for n, g in g1.items()}, workspace=ws1.view)
    wt.wtconv_bwd(d["x"], d["dy"], *ps, L, k, dx=dx2.view, grads={n: g.view for n, g in g2.items()},
                  workspace=ws2.view)
    torch.cuda.synchronize()
    assert wt.wtconv_device_faults() == 0
    for name, buf in [("y", y), ("dx", dx), ("dx (fused)", dx2), ("workspace", ws1), ("workspace (fused)", ws2)] + \
            [(n, g) for n, g in g1.items()] + [(n + " (fused)", g) for n, g in g2.items()]:
        assert buf.intact(), f"write outside {name}"
    for n, t in snap.items():
        assert torch.equal(t, d[n]), f"input {n} was modified"
