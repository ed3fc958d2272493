"""Seeded random layers through every entry point, against the float64 oracle.

The hand-picked cases elsewhere pin the planner's known corners; this sweep
draws layers at random within the documented limits (planes up to 56 px
at every level count; larger planes, which run in windowed tiles, with
levels <= 4, or 5 at k = 3; and larger planes with deeper pyramids, which
run as a fine pass plus a coarse layer), so that plane grouping, final-tile heights,
input-set counts, load modes and the fused-or-separate backward choice meet
combinations nobody picked.  Batch, channels, odd and even sizes, k, dtype
and bias are drawn too.  Every call must accept its layer, and y, dx (from
both backward entry points) and every parameter gradient must match the
oracle within the parity tolerances.
"""
import numpy as np
import pytest
import torch

import oracle
from memory_bound_cnn_wtconv2d_gb300 import synth

from test_parity_gpu import GRADS, compare, to_dev, wt  # noqa: F401  (wt is a fixture)

DTYPES = ("f32", "f16", "bf16")


def random_cases(n=96, seed=2026):
    """(N, C, H, W, L, k, dtype, bias) drawn within the documented limits."""
    rng = np.random.Generator(np.random.PCG64(seed))
    cases = []
    for i in range(n):
        k = int(rng.choice([3, 5, 7, 9]))
        if i % 3 == 2:  # a plane beyond one CTA: windowed tiles
            H, W = (int(v) for v in rng.integers(57, 161, size=2))
            L = int(rng.integers(1, 6 if k == 3 else 5))
        else:
            H, W = (int(v) for v in rng.integers(1, 57, size=2))
            L = int(rng.integers(1, 9))
        N, C = int(rng.integers(1, 5)), int(rng.integers(1, 6))
        cases.append((N, C, H, W, L, k, DTYPES[int(rng.integers(0, 3))], bool(rng.random() < 0.8)))
    return cases


CASES = random_cases()


def random_split_cases(n=12, seed=2027):
    """Larger planes with deep pyramids, whose tile window does not fit one CTA:
    they run as a fine pass plus a coarse layer on the low-pass planes."""
    rng = np.random.Generator(np.random.PCG64(seed))
    cases = []
    for _ in range(n):
        k = int(rng.choice([3, 5, 7, 9]))
        H, W = (int(v) for v in rng.integers(113, 261, size=2))
        L = int(rng.integers(6 if k == 3 else 5, 9))
        N, C = int(rng.integers(1, 3)), int(rng.integers(1, 4))
        cases.append((N, C, H, W, L, k, DTYPES[int(rng.integers(0, 3))], bool(rng.random() < 0.8)))
    return cases


SPLIT_CASES = random_split_cases()


def case_seed(case):
    return 7 + sum((i + 1) * v for i, v in enumerate(case[:6])) + 1000 * DTYPES.index(case[6])


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES + SPLIT_CASES, ids=lambda c: "x".join(map(str, c)))
def test_random_layer_all_entry_points(wt, case):
    N, C, H, W, L, k, dtype, bias = case
    inp = synth.make_inputs(N, C, H, W, L, k, dtype=dtype, seed=case_seed(case), bias=bias)
    d = to_dev(inp)
    ps = [d[n] for n in ("w_base", "b_base", "w_sub", "base_scale", "wavelet_scale")]
    y = wt.wtconv_fwd(d["x"], *ps, L, k)
    dx = wt.wtconv_bwd_data(d["dy"], ps[0], ps[2], ps[3], ps[4], L, k)
    g = wt.wtconv_bwd_weight(d["x"], d["dy"], *ps, L, k)
    dx2, g2 = wt.wtconv_bwd(d["x"], d["dy"], *ps, L, k)
    torch.cuda.synchronize()
    assert wt.wtconv_device_faults() == 0
    compare("y", y.float().cpu().numpy(), oracle.fwd(inp), dtype, False)
    ref = oracle.bwd(inp)
    compare("dx", dx.float().cpu().numpy(), ref["dx"], dtype, False)
    compare("dx (wtconv_bwd)", dx2.float().cpu().numpy(), ref["dx"], dtype, False)
    for n in GRADS:
        if ref[n] is None:
            assert g[n] is None and g2[n] is None
            continue
        compare(n, g[n].cpu().numpy(), ref[n], dtype, True)
        compare(n + " (wtconv_bwd)", g2[n].cpu().numpy(), ref[n], dtype, True)


def test_cases_stay_within_the_documented_limits():
    for N, C, H, W, L, k, dtype, bias in CASES:
        assert 1 <= L <= 8 and k in (3, 5, 7, 9) and dtype in DTYPES
        if max(H, W) > 56:
            assert L <= 4 or (L == 5 and k == 3)
    # the draw covers windowed planes, deep pyramids, every k and dtype, and both bias settings
    assert any(max(c[2], c[3]) > 56 for c in CASES) and any(c[4] >= 6 for c in CASES)
    assert {c[5] for c in CASES} == {3, 5, 7, 9} and {c[6] for c in CASES} == set(DTYPES)
    assert {c[7] for c in CASES} == {True, False}
    # the split draws: beyond one CTA, and deeper than one tile window reaches
    for N, C, H, W, L, k, dtype, bias in SPLIT_CASES:
        assert min(H, W) > 112 and L <= 8 and (L >= 5 if k > 3 else L >= 6)
    assert {c[5] for c in SPLIT_CASES} == {3, 5, 7, 9} and {c[6] for c in SPLIT_CASES} == set(DTYPES)
