"""The multi-process (N > 1) host path of bench.py on CPU with gloo ranks.

bench.py runs one process per GPU: N independent replicas of the layer step,
a barrier on both sides of the timed region and the maximum over ranks, and
a single JSON line from rank 0.  These tests exercise that host logic with
world size 2 on the CPU (the rendezvous on 127.0.0.1).
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    out[rank] = bench.max_over_ranks(world, float(10 * (rank + 1)))
    bench.barrier(world)
    dist.destroy_process_group()


def test_barrier_and_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(2, free_port(), out), nprocs=2, join=True, start_method="spawn")
        assert dict(out) == {0: 20.0, 1: 20.0}


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    env = dict(os.environ, OMP_NUM_THREADS="1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()),
           "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    res = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["unit"] == "ms/layer" and line["higher_is_better"] is False
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
    # every key of the bench line's contract, with the reference arm's own values
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["steps"] == 1 and line["warmup"] == 0 and line["ms_per_step"] == line["value"]
    assert "workload" in line["config"] and line["dtype"] == "f64" and line["vs_baseline"] is None
    assert {"value", "unit", "cores", "sample", "kind"} <= set(line["cpu_baseline"])
    assert line["cpu_baseline"]["value"] == line["value"] and line["e2e"]["value"] == line["value"]


def test_bench_algorithmic_counts():
    # The roofline's algorithmic figures: 181,300 FMAs per 56x56 plane at 3
    # levels and k = 5 (25 per base output and per coefficient of the 4 bands
    # at 28x28, 14x14, 7x7), i.e. 1.114 G per pass over the stage-1 layer's
    # 6144 planes; odd sizes are padded to even at every level.
    import bench
    assert bench.fma_per_plane(56, 56, 3, 5) == 25 * (56 * 56 + 4 * (28 * 28 + 14 * 14 + 7 * 7)) == 181300
    assert bench.fma_per_plane(56, 56, 3, 5) * 64 * 96 == 1113907200
    assert bench.level_sizes(7, 5, 3) == ([7, 4, 2, 1], [5, 3, 2, 1])
    assert bench.fma_per_plane(1, 1, 2, 3) == 9 * (1 + 4 * 2)
