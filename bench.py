"""WTConv2d forward + backward benchmark on GB300.

One step = one full training pass of one WTConv2d layer: wtconv_fwd,
wtconv_bwd_data and wtconv_bwd_weight through the C ABI, on the WTConvNeXt-T
stage-1 layer shape x[64,96,56,56] float32, L=3, k=5 (synthetic seeded
inputs and random-init weights).  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 (under torch.distributed.run) runs N independent replicas, one per
GPU: every rank processes its own layer, the path has no data exchange.
``--impl reference`` times the float64 CPU oracle on a bounded sample of the
same workload instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from memory_bound_cnn_wtconv2d_gb300 import synth  # noqa: E402

METRIC = "WTConv2d fwd+bwd ms/layer and achieved HBM TB/s vs ~8 TB/s peak (1 GB300)"
WORKLOAD = "stage1"
ROTATE = 4          # input buffer sets cycled through (4 x 154 MB > 129 MB L2)
NUM_SMS = 152
FP32_LANES = 128    # FP32 FMA lanes per SM (measured: 128 FMA/clk/SM)
SM_MAX_MHZ = 2070.0
ESIZE = {"f32": 4, "f16": 2, "bf16": 2}


def level_sizes(H, W, L):
    Hs, Ws = [H], [W]
    for _ in range(L):
        Hs.append((Hs[-1] + 1) // 2)
        Ws.append((Ws[-1] + 1) // 2)
    return Hs, Ws


def fma_per_plane(H, W, L, k):
    """Algorithmic FMAs of one pass over one plane: k^2 per base output and per
    subband coefficient of every level (identical for fwd, bwd_data, bwd_weight)."""
    Hs, Ws = level_sizes(H, W, L)
    return k * k * (H * W + 4 * sum(Hs[l] * Ws[l] for l in range(1, L + 1)))


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch of each
# kernel, from one ncu capture of the stage-1 layer (profiles/ncu_full_stage1_f32.md),
# valid only for the kernel sources they were taken on (hash below).
MEASURED_TRAFFIC = {
    "csrc_sha256": "8e13c6a1d3194ec875e038bdce258726c891f8dc80ce663fbbba9a3f3ad842d9",
    "workload": "stage1",
    "bytes": {"fwd": 108_307_456, "bwd_data": 108_124_416, "bwd_weight": 157_428_736},
}


def csrc_sha256():
    import hashlib
    h = hashlib.sha256()
    d = os.path.join(ROOT, "memory_bound_cnn_wtconv2d_gb300", "csrc")
    for name in sorted(os.listdir(d)):
        if name.endswith((".cu", ".cuh", ".h")):
            h.update(name.encode())
            with open(os.path.join(d, name), "rb") as f:
                h.update(f.read())
    return h.hexdigest()


def measured_traffic(kernel):
    t = MEASURED_TRAFFIC
    if WORKLOAD != t["workload"] or csrc_sha256() != t["csrc_sha256"]:
        return None  # the kernels changed since the counters were taken
    return t["bytes"].get(kernel)


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [v.strip() for v in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def setup_dist(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if (args.impl == "ours" and not args.cpu_dist) else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, value, device=None):
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def workload_config(inp, rotate=ROTATE):
    return {"workload": f"WTConvNeXt-T stage-1 WTConv2d layer x[{inp.N},{inp.C},{inp.H},{inp.W}] "
                        f"{inp.dtype} L={inp.levels} k={inp.k}",
            "N": inp.N, "C": inp.C, "H": inp.H, "W": inp.W, "levels": inp.levels, "k": inp.k,
            "l2": f"inputs larger than L2: {rotate} rotating (x, dy) sets of "
                  f"{2 * inp.numel * ESIZE[inp.dtype] / 1e6:.0f} MB each"}


def time_oracle(inp, n_images):
    """fwd+bwd of the float64 oracle on the first n_images of the batch; seconds."""
    import oracle
    sample = synth.LayerInputs(N=n_images, C=inp.C, H=inp.H, W=inp.W, levels=inp.levels, k=inp.k,
                               dtype=inp.dtype, x=inp.x[:n_images], dy=inp.dy[:n_images],
                               w_base=inp.w_base, b_base=inp.b_base, w_sub=inp.w_sub,
                               base_scale=inp.base_scale, wavelet_scale=inp.wavelet_scale)
    t0 = time.perf_counter()
    oracle.fwd(sample)
    oracle.bwd(sample)
    return time.perf_counter() - t0


def run_reference(args, world, rank):
    """The oracle on the host cores, each step a bounded sample of the workload."""
    if rank != 0:
        return None
    import oracle
    oracle.build()
    inp = synth.workload(WORKLOAD)
    n_img = 1
    for _ in range(args.warmup):
        time_oracle(inp, n_img)
    times = [time_oracle(inp, n_img) for _ in range(args.steps)]
    ms_layer = 1e3 * sum(times) / len(times) * (inp.N / n_img)
    sample = f"{n_img} of {inp.N} images per step ({n_img * inp.C} planes), scaled to the full batch"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(ms_layer, 3), "unit": "ms/layer",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_layer, 3),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) activations, random-init weights)",
        "config": workload_config(inp),
        "cpu_baseline": {"value": round(ms_layer, 3), "unit": "ms/layer", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(ms_layer, 3), "unit": "ms/layer", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return line


def run_ours(args, world, rank, local):
    import torch

    from memory_bound_cnn_wtconv2d_gb300 import build, wtconv

    build.build()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    inp = synth.workload(WORKLOAD)
    dt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[inp.dtype]
    L, k = inp.levels, inp.k
    P = lambda a: None if a is None else torch.tensor(a, dtype=torch.float32, device=dev)
    wb, bb, wsub, sb, sw = P(inp.w_base), P(inp.b_base), P(inp.w_sub), P(inp.base_scale), P(inp.wavelet_scale)
    x0 = torch.tensor(inp.x, dtype=dt, device=dev)
    dy0 = torch.tensor(inp.dy, dtype=dt, device=dev)
    xs = [x0] + [x0.clone() for _ in range(ROTATE - 1)]
    dys = [dy0] + [dy0.clone() for _ in range(ROTATE - 1)]
    y = torch.empty_like(x0)
    dx = torch.empty_like(x0)
    grads = dict(dw_base=torch.empty_like(wb), db_base=torch.empty_like(bb), dw_sub=torch.empty_like(wsub),
                 dbase_scale=torch.empty_like(sb), dwavelet_scale=torch.empty_like(sw))
    desc = wtconv.desc_for(x0, L, k)
    ws = torch.empty(max(wtconv.wtconv_workspace_size(desc, wtconv.OP_BWD_WEIGHT), 256), dtype=torch.uint8,
                     device=dev)
    launches_per_step = 4  # fwd, bwd_data, bwd_weight correlation + its finalize

    def step(i, ev=None):
        x, dy_ = xs[i % ROTATE], dys[i % ROTATE]
        if ev is not None:
            ev[0].record(stream)
        wtconv.wtconv_fwd(x, wb, bb, wsub, sb, sw, L, k, y=y, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        wtconv.wtconv_bwd_data(dy_, wb, wsub, sb, sw, L, k, dx=dx, stream=stream)
        if ev is not None:
            ev[2].record(stream)
        wtconv.wtconv_bwd_weight(x, dy_, wb, bb, wsub, sb, sw, L, k, grads=grads, workspace=ws, stream=stream)
        if ev is not None:
            ev[3].record(stream)

    warmup = max(args.warmup, 3)
    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        start.record(stream)
        for i in range(args.steps):
            step(i, evs[i])
        end.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    elapsed_ms = start.elapsed_time(end)
    elapsed_ms = max_over_ranks(world, elapsed_ms, dev)
    per = {"fwd": [], "bwd_data": [], "bwd_weight": []}
    for e in evs:
        per["fwd"].append(e[0].elapsed_time(e[1]))
        per["bwd_data"].append(e[1].elapsed_time(e[2]))
        per["bwd_weight"].append(e[2].elapsed_time(e[3]))
    avg = {kname: sum(v) / len(v) for kname, v in per.items()}

    # end to end through the public API with host buffers (pinned)
    e2e = None
    if not args.no_e2e:
        xh = torch.tensor(inp.x, dtype=dt).pin_memory()
        dyh = torch.tensor(inp.dy, dtype=dt).pin_memory()
        yh = torch.empty_like(xh).pin_memory()
        dxh = torch.empty_like(xh).pin_memory()
        gh = {n: torch.empty(t.shape, dtype=t.dtype).pin_memory() for n, t in grads.items()}

        def e2e_step():
            xs[0].copy_(xh, non_blocking=True)
            dys[0].copy_(dyh, non_blocking=True)
            step(0)
            yh.copy_(y, non_blocking=True)
            dxh.copy_(dx, non_blocking=True)
            for n, t in grads.items():
                gh[n].copy_(t, non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        barrier(world)
        s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s2.record(stream)
        for _ in range(args.steps):
            e2e_step()
        e2.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        e2e_ms = max_over_ranks(world, s2.elapsed_time(e2), dev)
        h2d = 2 * xh.numel() * xh.element_size()
        d2h = 2 * yh.numel() * yh.element_size() + sum(t.numel() * 4 for t in gh.values())
        e2e = {"value": round(e2e_ms / (args.steps * world), 4), "unit": "ms/layer",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    if rank != 0:
        return None
    peaks, peak_kind = measured_peaks()
    e = ESIZE[inp.dtype]
    ne = inp.numel
    alg_bytes = {"fwd": 2 * ne * e, "bwd_data": 2 * ne * e, "bwd_weight": 2 * ne * e}
    fma = fma_per_plane(inp.H, inp.W, L, k) * inp.N * inp.C
    ms_step = elapsed_ms / args.steps
    step_bytes = sum(alg_bytes.values())
    hbm_tbs = step_bytes / (ms_step * 1e-3) / 1e12
    dom = max(avg, key=avg.get)
    clocks = clk.summary()
    alu_peak = NUM_SMS * FP32_LANES * 2 * SM_MAX_MHZ * 1e6 / 1e12  # TFLOP/s at the maximum SM clock
    achieved_alu = 2 * fma / (avg[dom] * 1e-3) / 1e12
    roofline = {"bound": "alu", "kernel": dom, "achieved": round(achieved_alu, 2), "peak": round(alu_peak, 2),
                "unit": "TFLOP/s", "frac": round(achieved_alu / alu_peak, 4), "traffic": measured_traffic(dom),
                "traffic_unit": "bytes per launch (ncu dram read+write)",
                "peak_source": f"{NUM_SMS} SMs x {FP32_LANES} FP32 FMA/clk x 2 x {SM_MAX_MHZ:.0f} MHz",
                "algorithmic_fma_per_launch": fma}
    hbm = {"achieved_step_tbs": round(hbm_tbs, 3), "peak_gbs": peaks.get("hbm_gbs"), "peak_kind": peak_kind,
           "frac_of_measured": round(hbm_tbs * 1e3 / peaks["hbm_gbs"], 4), "frac_of_8tbs": round(hbm_tbs / 8.0, 4),
           "algorithmic_bytes_per_step": step_bytes,
           "per_kernel_gbs": {kn: round(alg_bytes[kn] / (avg[kn] * 1e-3) / 1e9, 1) for kn in avg}}
    line = {
        "metric": METRIC, "value": round(elapsed_ms / (args.steps * world), 4), "unit": "ms/layer",
        "n_gpus": world, "steps": args.steps, "warmup": warmup,
        "ms_per_step": round(ms_step, 4), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": inp.dtype,
        "data": "synthetic (seeded N(0,1) activations, random-init weights)",
        "config": workload_config(inp) | {"parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "kernel_ms": {kn: round(v, 4) for kn, v in avg.items()},
        "roofline": roofline, "hbm": hbm, "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks, "e2e": e2e,
    }
    if world == 1 and not args.no_cpu_baseline:
        n_img = inp.N
        t = time_oracle(inp, n_img)
        line["cpu_baseline"] = {"value": round(1e3 * t * inp.N / n_img, 1), "unit": "ms/layer", "cores": 1,
                                "kind": "oracle",
                                "sample": f"one fwd+bwd of the float64 oracle over {n_img} of {inp.N} images "
                                          f"(single thread)"}
    print(json.dumps(line), flush=True)
    return line


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-dist", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args(argv)
    world, rank, local = setup_dist(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
