"""Minimal filtering (Winograd-style, Lavin & Gray 2016) for the layer's
5 x 5 depthwise convolution tiles: the transforms, and the probe that
measures them against the direct form.

The library keeps the direct form (25 FMAs per output): a depthwise kernel
has one input plane, so a transformed input serves one kernel, and the
transform additions run on the same FP32 pipe as the products.  The probe in
``minimal_filtering/`` times both on identical shared-memory tiles; these
tests pin its transforms (CPU) and its numerics (GPU).
"""
import importlib.util
import os
import shutil
import subprocess
import sys

import pytest

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "minimal_filtering")


def _generator():
    pytest.importorskip("sympy")
    spec = importlib.util.spec_from_file_location("gen_transforms", os.path.join(HERE, "gen_transforms.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("m", [2, 4])
def test_transforms_compute_the_correlation(m):
    """A^T [(G g) * (B^T d)] equals sum_k d[i + k] g[k] symbolically, and the
    row and column pairings the probe's factored transforms rely on hold."""
    gen = _generator()
    AT, G, BT = gen.transforms(m)
    gen.check(m, AT, G, BT)
    gen.check_pairs(m, AT, BT)
    n = m + gen.R - 1
    assert AT.shape == (m, n) and G.shape == (n, gen.R) and BT.shape == (n, n)


def test_transforms_at_random_integers():
    """Exact rational evaluation on random integer data (independent of the
    symbolic check): each F(m, 5) reproduces the direct correlation."""
    import random

    import sympy as sp
    gen = _generator()
    rng = random.Random(5)
    for m in (2, 4):
        AT, G, BT = gen.transforms(m)
        n = m + gen.R - 1
        for _ in range(20):
            g = [rng.randint(-9, 9) for _ in range(gen.R)]
            d = [rng.randint(-9, 9) for _ in range(n)]
            u = G * sp.Matrix(g)
            v = BT * sp.Matrix(d)
            y = AT * sp.Matrix([u[i] * v[i] for i in range(n)])
            assert [y[i] for i in range(m)] == [sum(d[i + k] * g[k] for k in range(gen.R)) for i in range(m)]


def test_header_matches_generator(tmp_path):
    """The committed header is what the generator writes."""
    _generator()  # (skips without sympy)
    src = os.path.join(HERE, "winograd_transforms.h")
    with open(src) as f:
        committed = f.read()
    work = tmp_path / "gen"
    work.mkdir()
    shutil.copy(os.path.join(HERE, "gen_transforms.py"), work / "gen_transforms.py")
    subprocess.run([sys.executable, str(work / "gen_transforms.py")], check=True, capture_output=True)
    assert (work / "winograd_transforms.h").read_text() == committed


@pytest.mark.gpu
def test_probe_numerics(tmp_path):
    """Every form of the probe's tile (direct, F(2, 5), F(4, 5); 4- and 8-row
    tiles) against a double direct sum: rel-L2 within 1e-6 (direct), 1e-5
    (F(2, 5)) and 1e-4 (F(4, 5))."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    exe = str(tmp_path / "minimal_filtering_probe")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    os.path.join(HERE, "minimal_filtering_probe.cu"), "-o", exe], check=True, capture_output=True)
    r = subprocess.run([exe, "check"], capture_output=True, text=True, timeout=300)
    print(r.stdout)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "all forms within bounds" in r.stdout
