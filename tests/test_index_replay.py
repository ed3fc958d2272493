"""CPU replay of every kernel's memory accesses for the planner's launch plans
(CPU only; needs nvcc to compile host code, no GPU).

``index_replay/replay_indices.cu`` compiles the library's planner with the
launch functions stubbed out, then, for each plan, walks the kernels' phases
and recomputes every shared- and global-memory index they form: accesses
must stay inside their buffers, zero margins must never be written, and every
interior read must follow the write that fills it.  It covers small planes
exhaustively (every size up to 40 x 40, every level count and k, float32 and
16-bit), windowed plans on planes up to 1023 px, the fused backward up to
64 x 64, the benchmark's layers, and the random layers of the GPU sweep.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "index_replay", "replay_indices.cu")


@pytest.fixture(scope="module")
def replay(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path_factory.mktemp("replay") / "replay_indices")
    subprocess.run([nvcc, "-std=c++17", "-O2", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(ROOT, "memory_bound_cnn_wtconv2d_gb300", "csrc"), SRC, "-o", exe],
                   check=True, capture_output=True)
    return exe


def run(args):
    r = subprocess.run(args, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0 and "errors: 0" in r.stdout, r.stdout[-4000:]
    return r.stdout


def test_plans_of_every_small_plane_windowed_and_fused_layer(replay):
    out = run([replay])
    assert "window plans checked" in out and "fused backward plans checked" in out


def test_plans_of_the_random_gpu_sweep(replay, tmp_path):
    from test_random_shapes_gpu import CASES, DTYPES
    cases = tmp_path / "cases.txt"
    cases.write_text("".join(" ".join(map(str, c[:6])) + f" {DTYPES.index(c[6])}\n" for c in CASES))
    out = run([replay, "file", str(cases)])
    assert f"layers: {len(CASES)}, refused: 0" in out

