"""The batch-split oracle helpers (test infrastructure) agree with the plain
oracle: the slices run the same code, dx is concatenated, and the parameter
gradients (sums over the shared parameters) are added in float64."""
import numpy as np
import pytest

import oracle
from memory_bound_cnn_wtconv2d_gb300 import synth


@pytest.mark.parametrize("workers", [1, 3, 7])
def test_parallel_oracle_equals_plain_oracle(workers):
    inp = synth.make_inputs(5, 3, 13, 10, 3, 5, seed=9)
    y = oracle.fwd(inp)
    yp = oracle.fwd_parallel(inp, workers)
    assert np.array_equal(y, yp)  # per-image results are computed independently
    g = oracle.bwd(inp)
    gp = oracle.bwd_parallel(inp, workers)
    assert np.array_equal(g["dx"], gp["dx"])
    for name in ("dw_base", "db_base", "dw_sub", "dbase_scale", "dwavelet_scale"):
        np.testing.assert_allclose(gp[name], g[name], rtol=1e-12, atol=1e-13)


def test_parallel_oracle_without_bias_and_empty_batch():
    inp = synth.make_inputs(4, 2, 9, 9, 2, 3, seed=3, bias=False)
    gp = oracle.bwd_parallel(inp, 2)
    assert gp["db_base"] is None
    np.testing.assert_allclose(gp["dw_sub"], oracle.bwd(inp)["dw_sub"], rtol=1e-12, atol=1e-13)
    empty = synth.make_inputs(0, 2, 9, 9, 2, 3, seed=3)
    assert oracle.fwd_parallel(empty).shape == (0, 2, 9, 9)
