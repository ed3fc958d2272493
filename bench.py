"""WTConv2d forward + backward benchmark on GB300.

One step = one full training pass of one WTConv2d layer through the C ABI:
wtconv_fwd, then wtconv_bwd (the input gradient and every parameter gradient
in one call, one fused kernel over x and dy), on the WTConvNeXt-T stage-1
layer shape x[64,96,56,56] float32, L=3, k=5 (synthetic seeded inputs and
random-init weights).  The same backward as the two separate calls
(wtconv_bwd_data + wtconv_bwd_weight) is timed beside it for context.
Prints one JSON line.

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
# kernel of the step, from one ncu capture of the stage-1 layer, valid only
# for the kernel sources they were taken on (hash below).
MEASURED_TRAFFIC = {
    "csrc_sha256": "697b577392655455cc5738c8deca8ffda2025c90136ede2c8414a4cbba4c2ebf",
    "workload": "stage1",
    # fwd: fwd_kernel; bwd: the fused backward kernel (its finalize reads < 1 MB)
    "bytes": {"fwd": 108_246_528, "bwd": 202_700_032},
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


def time_oracle_parallel(inp, workers):
    """fwd+bwd of the float64 oracle over the whole batch, the images split into
    `workers` slices run by that many threads (the oracle's C calls release the
    interpreter lock); seconds.  The same work as time_oracle over all images."""
    import concurrent.futures
    import oracle
    oracle.fwd(synth.LayerInputs(N=1, C=inp.C, H=inp.H, W=inp.W, levels=inp.levels, k=inp.k, dtype=inp.dtype,
                                 x=inp.x[:1], dy=inp.dy[:1], w_base=inp.w_base, b_base=inp.b_base,
                                 w_sub=inp.w_sub, base_scale=inp.base_scale,
                                 wavelet_scale=inp.wavelet_scale))  # load the library first
    bounds = [inp.N * i // workers for i in range(workers + 1)]

    def run(i):
        a, b = bounds[i], bounds[i + 1]
        if b <= a:
            return
        part = synth.LayerInputs(N=b - a, C=inp.C, H=inp.H, W=inp.W, levels=inp.levels, k=inp.k,
                                 dtype=inp.dtype, x=inp.x[a:b], dy=inp.dy[a:b], w_base=inp.w_base,
                                 b_base=inp.b_base, w_sub=inp.w_sub, base_scale=inp.base_scale,
                                 wavelet_scale=inp.wavelet_scale)
        oracle.fwd(part)
        oracle.bwd(part)

    t0 = time.perf_counter()
    with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as ex:
        list(ex.map(run, range(workers)))
    return time.perf_counter() - t0


def unfused_torch_layer(x, w_base, b_base, w_sub, base_scale, wavelet_scale, levels, k):
    """WTConv2d with one PyTorch library op per stage, the way the pages describe
    the reference implementation (technical summary, "Problem statement"): a
    grouped stride-2 convolution with the four Haar filters writes the
    subbands of each level, a depthwise convolution per subband, the wavelet
    scale as its own elementwise pass, a grouped transposed convolution per
    level for the synthesis (the previous reconstruction added to the
    low-pass band first), and the scaled base depthwise convolution.  Autograd
    differentiates it.  A comparison arm only: nothing calls it on the path.
    """
    import torch
    import torch.nn.functional as F

    N, C = x.shape[:2]
    r = k // 2
    haar = 0.5 * torch.tensor([[[1, 1], [1, 1]], [[1, 1], [-1, -1]], [[1, -1], [1, -1]], [[1, -1], [-1, 1]]],
                              dtype=x.dtype, device=x.device)
    filt = haar.unsqueeze(1).repeat(C, 1, 1, 1)  # [4C, 1, 2, 2]: subband channel 4c+b
    cur, zs, sizes = x, [], []
    for lev in range(levels):
        h, w = cur.shape[-2:]
        sizes.append((h, w))
        Y = F.conv2d(F.pad(cur, (0, w % 2, 0, h % 2)), filt, stride=2, groups=C)
        Z = F.conv2d(Y, w_sub[lev].unsqueeze(1), padding=r, groups=4 * C)
        zs.append(Z * wavelet_scale[lev].view(1, -1, 1, 1))
        cur = Y.view(N, C, 4, *Y.shape[-2:])[:, :, 0]
    nxt = None
    for lev in reversed(range(levels)):
        Z = zs[lev]
        if nxt is not None:
            Zv = Z.view(N, C, 4, *Z.shape[-2:])
            Z = torch.cat([Zv[:, :, :1] + nxt.unsqueeze(2), Zv[:, :, 1:]], dim=2).view(Z.shape)
        h, w = sizes[lev]
        nxt = F.conv_transpose2d(Z, filt, stride=2, groups=C)[..., :h, :w]
    base = F.conv2d(x, w_base.unsqueeze(1), b_base, padding=r, groups=C) * base_scale.view(1, -1, 1, 1)
    return base + nxt


def compare_arms(inp, dev, reps=10):
    """Training step (fwd + autograd bwd) and inference (fwd) of the fused
    layer, the unfused PyTorch composition and a cuDNN depthwise 7x7
    convolution on the same x, plus the peak extra device memory of one
    training step.  Comparison figures only."""
    import torch
    import torch.nn.functional as F

    from memory_bound_cnn_wtconv2d_gb300 import layer, wtconv

    dt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[inp.dtype]
    L, k, C = inp.levels, inp.k, inp.C
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)  # > L2
    f32 = lambda a: None if a is None else torch.tensor(a, dtype=torch.float32, device=dev)
    p32 = [f32(a) for a in (inp.w_base, inp.b_base, inp.w_sub, inp.base_scale, inp.wavelet_scale)]
    pdt = [a.to(dt) for a in p32]
    w7 = (0.05 * torch.randn(C, 1, 7, 7, generator=torch.Generator().manual_seed(7))).to(dev, dt)
    x = torch.tensor(inp.x, dtype=dt, device=dev)
    dy = torch.tensor(inp.dy, dtype=dt, device=dev)

    def leaves(ps):
        return [p.detach().clone().requires_grad_(True) for p in ps]

    def train_fused():
        xg = x.detach().requires_grad_(True)
        y = layer.WTConv2dFunction.apply(xg, *leaves(p32), L, k)
        y.backward(dy)

    def train_unfused():
        xg = x.detach().requires_grad_(True)
        y = unfused_torch_layer(xg, *leaves(pdt), L, k)
        y.backward(dy)

    def train_dw7():
        xg = x.detach().requires_grad_(True)
        wg = w7.detach().requires_grad_(True)
        F.conv2d(xg, wg, padding=3, groups=C).backward(dy)

    def infer_fused():
        wtconv.wtconv_fwd(x, *p32, L, k)

    def infer_unfused():
        with torch.no_grad():
            unfused_torch_layer(x, *pdt, L, k)

    def infer_dw7():
        with torch.no_grad():
            F.conv2d(x, w7, padding=3, groups=C)

    def timed(fn):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(reps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        return round(statistics.median(ts), 4)

    def peak(fn):
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        base = torch.cuda.memory_allocated(dev)
        torch.cuda.reset_peak_memory_stats(dev)
        fn()
        torch.cuda.synchronize()
        return int(torch.cuda.max_memory_allocated(dev) - base)

    def steady(fn, steps=10):
        # back-to-back steps, as in training: the host enqueues ahead of the
        # GPU, so per-call host latency is hidden (a step's tensors, >= 300 MB
        # at the bench workload, exceed the L2 anyway)
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(steps):
            fn()
        b.record()
        torch.cuda.synchronize()
        return round(a.elapsed_time(b) / steps, 4)

    train = {"fused": timed(train_fused), "unfused_torch": timed(train_unfused), "dw7x7_cudnn": timed(train_dw7)}
    train_steady = {"fused": steady(train_fused), "unfused_torch": steady(train_unfused),
                    "dw7x7_cudnn": steady(train_dw7)}
    infer = {"fused": timed(infer_fused), "unfused_torch": timed(infer_unfused), "dw7x7_cudnn": timed(infer_dw7)}
    mem = {"fused": peak(train_fused), "unfused_torch": peak(train_unfused), "dw7x7_cudnn": peak(train_dw7)}
    del flush
    return {
        "workload": workload_config(inp)["workload"], "dtype": inp.dtype,
        "train_ms": train, "train_steady_ms": train_steady, "infer_ms": infer, "train_peak_extra_bytes": mem,
        "train_speedup_vs_unfused": round(train["unfused_torch"] / train["fused"], 3),
        "train_speedup_vs_dw7x7": round(train["dw7x7_cudnn"] / train["fused"], 3),
        "train_steady_speedup_vs_unfused": round(train_steady["unfused_torch"] / train_steady["fused"], 3),
        "train_steady_speedup_vs_dw7x7": round(train_steady["dw7x7_cudnn"] / train_steady["fused"], 3),
        "infer_speedup_vs_unfused": round(infer["unfused_torch"] / infer["fused"], 3),
        "infer_speedup_vs_dw7x7": round(infer["dw7x7_cudnn"] / infer["fused"], 3),
        "train_peak_mem_reduction_vs_unfused": round(mem["unfused_torch"] / max(mem["fused"], 1), 3),
    }


def run_arm_only(args):
    """One arm's training step on the bench workload, for a profiler's launch
    list (its per-kernel DRAM bytes give the bytes moved per element)."""
    import torch
    import torch.nn.functional as F

    from memory_bound_cnn_wtconv2d_gb300 import build, layer

    build.build()
    dev = torch.device("cuda:0")
    inp = synth.workload(WORKLOAD)
    dt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[inp.dtype]
    f32 = lambda a: None if a is None else torch.tensor(a, dtype=torch.float32, device=dev, requires_grad=True)
    ps = [f32(a) for a in (inp.w_base, inp.b_base, inp.w_sub, inp.base_scale, inp.wavelet_scale)]
    x = torch.tensor(inp.x, dtype=dt, device=dev, requires_grad=True)
    dy = torch.tensor(inp.dy, dtype=dt, device=dev)
    w7 = torch.zeros(inp.C, 1, 7, 7, dtype=dt, device=dev, requires_grad=True)
    arm = args.arm_only.replace("_infer", "")
    train = not args.arm_only.endswith("_infer")
    for _ in range(args.warmup + args.steps):
        with torch.set_grad_enabled(train):
            if arm == "fused":
                y = layer.WTConv2dFunction.apply(x, *ps, inp.levels, inp.k)
            elif arm == "unfused":
                y = unfused_torch_layer(x, *ps, inp.levels, inp.k)
            else:
                y = F.conv2d(x, w7, padding=3, groups=inp.C)
        if train:
            y.backward(dy)
    torch.cuda.synchronize()


def time_events(fn, flush, reps):
    """Median CUDA-event time (ms) of fn over reps runs, L2 flushed before each."""
    import torch
    for _ in range(3):
        fn()
    ts = []
    for _ in range(reps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.median(ts)


def run_suite(args):
    """The shape/level sweep (WTConvNeXt-T stage shapes x levels 1-5, N=128, fp32
    and fp16, a cuDNN depthwise 7x7 timed on the same x), the 18 WTConv layers
    of WTConvNeXt-T at batch 128 in fp16 (summed fwd+bwd time and peak device
    memory, fused vs the unfused PyTorch composition), every workload (tiny,
    stage 1, stage 2 in fp16 and bf16, one layer of each network stage) with
    the float64 oracle timed on one and on all host cores, or the planes
    larger than one CTA (forward and input gradient, tiled with a halo).
    One JSON line."""
    import torch
    import torch.nn.functional as F

    from memory_bound_cnn_wtconv2d_gb300 import build, layer, wtconv

    build.build()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
    reps = max(args.steps, 5)

    def fused_step(x, dy, ps, L, k, out):
        def run():
            wtconv.wtconv_fwd(x, *ps, L, k, y=out["y"])
            wtconv.wtconv_bwd(x, dy, *ps, L, k, dx=out["dx"], grads=out["g"], workspace=out["ws"])
        return run

    def buffers(x, ps, L, k):
        desc = wtconv.desc_for(x, L, k)
        return {"y": torch.empty_like(x), "dx": torch.empty_like(x),
                "g": dict(dw_base=torch.empty_like(ps[0]), db_base=torch.empty_like(ps[1]),
                          dw_sub=torch.empty_like(ps[2]), dbase_scale=torch.empty_like(ps[3]),
                          dwavelet_scale=torch.empty_like(ps[4])),
                "ws": torch.empty(max(wtconv.wtconv_workspace_size(desc, wtconv.OP_BWD),
                                      wtconv.wtconv_workspace_size(desc, wtconv.OP_BWD_WEIGHT), 256),
                                  dtype=torch.uint8, device=dev)}

    rows = []
    if args.suite == "sweep":
        N = 128
        for dtype in ("f32", "f16"):
            for C, H in synth.SWEEP_SHAPES:
                base = synth.make_inputs(N, C, H, H, 1, 5, dtype=dtype, seed=3000 + C)
                x = torch.tensor(base.x, dtype=tdt[dtype], device=dev)
                dy = torch.tensor(base.dy, dtype=tdt[dtype], device=dev)
                w7 = torch.zeros(C, 1, 7, 7, dtype=tdt[dtype], device=dev, requires_grad=True)

                def dw7():
                    xg = x.detach().requires_grad_(True)
                    F.conv2d(xg, w7, padding=3, groups=C).backward(dy)
                t7 = time_events(dw7, flush, reps)
                for L in synth.SWEEP_LEVELS:
                    pin = synth.make_inputs(1, C, 1, 1, L, 5, dtype=dtype, seed=3000 + 10 * C + L)
                    ps = [torch.tensor(a, dtype=torch.float32, device=dev) for a in
                          (pin.w_base, pin.b_base, pin.w_sub, pin.base_scale, pin.wavelet_scale)]
                    t = time_events(fused_step(x, dy, ps, L, 5, buffers(x, ps, L, 5)), flush, reps)
                    ne = x.numel()
                    rows.append({"C": C, "H": H, "L": L, "dtype": dtype, "fused_fwd_bwd_ms": round(t, 4),
                                 "dw7x7_cudnn_fwd_bwd_ms": round(t7, 4), "speedup_vs_dw7x7": round(t7 / t, 3),
                                 "hbm_tbs": round(6 * ne * x.element_size() / (t * 1e-3) / 1e12, 3)})
                del x, dy
        line = {"suite": "sweep", "metric": "fwd+bwd ms per layer", "n": N, "rows": rows}
    elif args.suite == "configs":
        cases = [("tiny", synth.workload("tiny")), ("stage1", synth.workload("stage1")),
                 ("stage2_f16", synth.workload("stage2_f16")), ("stage2_bf16", synth.workload("stage2_bf16"))]
        cases += [(f"network C{C} H{H} L{L}", synth.make_inputs(128, C, H, H, L, 5, dtype="f16", seed=4000 + C))
                  for C, H, _, L in synth.NETWORK_STAGES]
        workers = os.cpu_count() or 1
        for name, inp in cases:
            x = torch.tensor(inp.x, dtype=tdt[inp.dtype], device=dev)
            dy = torch.tensor(inp.dy, dtype=tdt[inp.dtype], device=dev)
            ps = [torch.tensor(a, dtype=torch.float32, device=dev) for a in
                  (inp.w_base, inp.b_base, inp.w_sub, inp.base_scale, inp.wavelet_scale)]
            t = time_events(fused_step(x, dy, ps, inp.levels, inp.k, buffers(x, ps, inp.levels, inp.k)), flush, reps)
            t1 = time_oracle(inp, inp.N)
            tn = time_oracle_parallel(inp, max(1, min(workers, inp.N)))
            rows.append({"config": name, "shape": [inp.N, inp.C, inp.H, inp.W], "levels": inp.levels,
                         "dtype": inp.dtype, "fused_fwd_bwd_ms": round(t, 4),
                         "hbm_tbs": round(6 * x.numel() * x.element_size() / (t * 1e-3) / 1e12, 3),
                         "oracle_1core_s": round(t1, 3), "oracle_all_cores_s": round(tn, 3),
                         "oracle_cores": max(1, min(workers, inp.N))})
            del x, dy
        line = {"suite": "configs", "metric": "fwd+bwd ms per layer; oracle seconds per layer", "rows": rows}
    elif args.suite == "large":
        # Planes beyond one CTA (tiled with a halo): each call of the fused
        # layer, and the training step (wtconv_fwd + wtconv_bwd, which runs the
        # two windowed backward passes for such planes) against the unfused
        # PyTorch composition with autograd and a cuDNN depthwise 7x7, forward
        # alone and forward + backward, on the same x.
        cases = synth.LARGE_PLANES if args.large_case is None else [synth.LARGE_PLANES[args.large_case]]
        for N, C, H, W, L, k, dtype in cases:
            pin = synth.make_inputs(1, C, 1, 1, L, k, dtype=dtype, seed=5000 + C + L)
            ps = [torch.tensor(a, dtype=torch.float32, device=dev) for a in
                  (pin.w_base, pin.b_base, pin.w_sub, pin.base_scale, pin.wavelet_scale)]
            pdt = [p.to(tdt[dtype]) for p in ps]
            g = torch.Generator(device=dev).manual_seed(5000 + H + L)
            x = torch.randn(N, C, H, W, generator=g, device=dev).to(tdt[dtype])
            dy = torch.randn(N, C, H, W, generator=g, device=dev).to(tdt[dtype])
            out = buffers(x, ps, L, k)
            w7 = torch.zeros(C, 1, 7, 7, dtype=tdt[dtype], device=dev, requires_grad=True)
            tf = time_events(lambda: wtconv.wtconv_fwd(x, *ps, L, k, y=out["y"]), flush, reps)
            tb = time_events(lambda: wtconv.wtconv_bwd_data(dy, ps[0], ps[2], ps[3], ps[4], L, k, dx=out["dx"]),
                             flush, reps)
            tw = time_events(lambda: wtconv.wtconv_bwd_weight(x, dy, *ps, L, k, grads=out["g"], workspace=out["ws"]),
                             flush, reps)
            tt = time_events(fused_step(x, dy, ps, L, k, out), flush, reps)
            with torch.no_grad():
                tu = time_events(lambda: unfused_torch_layer(x, *pdt, L, k), flush, reps)
                t7 = time_events(lambda: F.conv2d(x, w7, padding=3, groups=C), flush, reps)

            def unf_train():
                xg = x.detach().requires_grad_(True)
                leaves = [p.detach().clone().requires_grad_(True) for p in pdt]
                unfused_torch_layer(xg, *leaves, L, k).backward(dy)

            def dw7_train():
                xg = x.detach().requires_grad_(True)
                F.conv2d(xg, w7, padding=3, groups=C).backward(dy)
            tut = time_events(unf_train, flush, reps)
            t7t = time_events(dw7_train, flush, reps)
            assert wtconv.wtconv_device_faults() == 0
            ne = x.numel()
            rows.append({"shape": [N, C, H, W], "levels": L, "k": k, "dtype": dtype,
                         "fwd_ms": round(tf, 4), "bwd_data_ms": round(tb, 4), "bwd_weight_ms": round(tw, 4),
                         "fused_fwd_bwd_ms": round(tt, 4),
                         "ps_per_element_fwd": round(tf * 1e9 / ne, 3),
                         "hbm_tbs_fwd_bwd": round(6 * ne * x.element_size() / (tt * 1e-3) / 1e12, 3),
                         "unfused_torch_fwd_ms": round(tu, 4), "unfused_torch_fwd_bwd_ms": round(tut, 4),
                         "dw7x7_cudnn_fwd_ms": round(t7, 4), "dw7x7_cudnn_fwd_bwd_ms": round(t7t, 4),
                         "speedup_fwd_vs_unfused": round(tu / tf, 3),
                         "speedup_fwd_bwd_vs_unfused": round(tut / tt, 3),
                         "speedup_fwd_vs_dw7x7": round(t7 / tf, 3),
                         "speedup_fwd_bwd_vs_dw7x7": round(t7t / tt, 3)})
            del x, dy, out
        line = {"suite": "large", "metric": "ms per call and per fwd+bwd step on planes beyond one CTA (tiled with a "
                "halo; the deepest reaches as a fine pass plus a coarse layer)",
                "rows": rows}
    else:
        N, dtype = 128, "f16"
        tot_fused = tot_unf = 0.0
        peak = {"fused": 0, "unfused_torch": 0}
        for C, H, depth, L in synth.NETWORK_STAGES:
            inp = synth.make_inputs(N, C, H, H, L, 5, dtype=dtype, seed=4000 + C)
            x = torch.tensor(inp.x, dtype=tdt[dtype], device=dev)
            dy = torch.tensor(inp.dy, dtype=tdt[dtype], device=dev)
            ps = [torch.tensor(a, dtype=torch.float32, device=dev) for a in
                  (inp.w_base, inp.b_base, inp.w_sub, inp.base_scale, inp.wavelet_scale)]
            pdt = [p.to(tdt[dtype]) for p in ps]
            t = time_events(fused_step(x, dy, ps, L, 5, buffers(x, ps, L, 5)), flush, reps)

            def unf():
                xg = x.detach().requires_grad_(True)
                leaves = [p.detach().clone().requires_grad_(True) for p in pdt]
                unfused_torch_layer(xg, *leaves, L, 5).backward(dy)

            def fus():
                xg = x.detach().requires_grad_(True)
                leaves = [p.detach().clone().requires_grad_(True) for p in ps]
                layer.WTConv2dFunction.apply(xg, *leaves, L, 5).backward(dy)
            tu = time_events(unf, flush, reps)
            for name, fn in (("fused", fus), ("unfused_torch", unf)):
                torch.cuda.synchronize()
                torch.cuda.empty_cache()
                torch.cuda.reset_peak_memory_stats(dev)
                fn()
                torch.cuda.synchronize()
                peak[name] = max(peak[name], int(torch.cuda.max_memory_allocated(dev)))
            rows.append({"C": C, "H": H, "depth": depth, "L": L, "fused_fwd_bwd_ms": round(t, 4),
                         "unfused_torch_fwd_bwd_ms": round(tu, 4)})
            tot_fused += depth * t
            tot_unf += depth * tu
            del x, dy
        line = {"suite": "network", "metric": "summed fwd+bwd ms of the 18 WTConv layers (batch 128, fp16)",
                "fused_ms": round(tot_fused, 3), "unfused_torch_ms": round(tot_unf, 3),
                "speedup": round(tot_unf / tot_fused, 3), "peak_device_bytes": peak,
                "peak_mem_reduction": round(peak["unfused_torch"] / max(peak["fused"], 1), 3), "rows": rows}
    print(json.dumps(line), flush=True)


PAGES_CONTEXT = ("pages (RTX A6000, context only): training 3.71-4.35x fp32 / 2.68-3.09x fp16 faster than "
                 "the reference, 1.83-2.31x less peak memory, 1.27-1.50x (fp32) / 1.40-1.76x (fp16) faster "
                 "than a depthwise 7x7; inference 3.67-4.37x fp32 / 3.38-3.60x fp16 vs the reference")


def run_reference(args, world, rank):
    """The oracle on the host cores: every step is one fwd+bwd of the float64
    oracle over the whole workload (all images), split over all host cores."""
    if rank != 0:
        return None
    import platform

    import oracle
    oracle.build()
    inp = synth.workload(WORKLOAD)
    workers = max(1, min(os.cpu_count() or 1, inp.N))
    for _ in range(args.warmup):
        time_oracle_parallel(inp, workers)
    times = [time_oracle_parallel(inp, workers) for _ in range(args.steps)]
    ms_layer = 1e3 * sum(times) / len(times)
    cpu = platform.processor() or platform.machine()
    sample = (f"the whole workload every step: fwd+bwd over all {inp.N} images ({inp.N * inp.C} planes), "
              f"split over {workers} threads on {cpu}")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(ms_layer, 3), "unit": "ms/layer",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_layer, 3),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) activations, random-init weights)",
        "config": workload_config(inp) | {"parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "cpu_baseline": {"value": round(ms_layer, 3), "unit": "ms/layer", "cores": workers, "kind": "oracle",
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
    ws = torch.empty(max(wtconv.wtconv_workspace_size(desc, wtconv.OP_BWD),
                         wtconv.wtconv_workspace_size(desc, wtconv.OP_BWD_WEIGHT), 256), dtype=torch.uint8,
                     device=dev)
    launches_per_step = 3  # fwd, the fused backward kernel + its dW finalize

    # One step: the forward, then the whole backward in one call (the fused
    # backward kernel: dx and every parameter gradient from one read of x, dy).
    def step(i, ev=None):
        x, dy_ = xs[i % ROTATE], dys[i % ROTATE]
        if ev is not None:
            ev[0].record(stream)
        wtconv.wtconv_fwd(x, wb, bb, wsub, sb, sw, L, k, y=y, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        wtconv.wtconv_bwd(x, dy_, wb, bb, wsub, sb, sw, L, k, dx=dx, grads=grads, workspace=ws, stream=stream)
        if ev is not None:
            ev[2].record(stream)

    # The same backward as the two separate calls, timed after the step (not
    # part of the value): context for the fused call.
    def step_separate(i, ev):
        x, dy_ = xs[i % ROTATE], dys[i % ROTATE]
        ev[0].record(stream)
        wtconv.wtconv_bwd_data(dy_, wb, wsub, sb, sw, L, k, dx=dx, stream=stream)
        ev[1].record(stream)
        wtconv.wtconv_bwd_weight(x, dy_, wb, bb, wsub, sb, sw, L, k, grads=grads, workspace=ws, stream=stream)
        ev[2].record(stream)

    warmup = max(args.warmup, 3)
    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
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
    per = {"fwd": [], "bwd": []}
    for e in evs:
        per["fwd"].append(e[0].elapsed_time(e[1]))
        per["bwd"].append(e[1].elapsed_time(e[2]))
    avg = {kname: sum(v) / len(v) for kname, v in per.items()}
    sep_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    for i in range(args.steps):
        step_separate(i, sep_ev[i])
    torch.cuda.synchronize()
    separate = {"bwd_data": sum(e[0].elapsed_time(e[1]) for e in sep_ev) / args.steps,
                "bwd_weight": sum(e[1].elapsed_time(e[2]) for e in sep_ev) / args.steps}

    # End to end through the public API with host buffers (pinned): every step
    # copies its inputs in, runs the three calls and copies y, dx and the
    # parameter gradients out.  Copies in, layer and copies out are pipelined on
    # three streams over two device buffer sets (step i+1's inputs arrive while
    # step i computes and step i-1's results leave).
    e2e = None
    if not args.no_e2e:
        xh = torch.tensor(inp.x, dtype=dt).pin_memory()
        dyh = torch.tensor(inp.dy, dtype=dt).pin_memory()
        yh = [torch.empty_like(xh).pin_memory() for _ in range(2)]
        dxh = [torch.empty_like(xh).pin_memory() for _ in range(2)]
        gh = [{n: torch.empty(t.shape, dtype=t.dtype).pin_memory() for n, t in grads.items()} for _ in range(2)]
        yd = [y, torch.empty_like(x0)]
        dxd = [dx, torch.empty_like(x0)]
        gd = [grads, {n: torch.empty_like(t) for n, t in grads.items()}]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

        def e2e_run(nsteps, start=None, end=None):
            ev_in = [torch.cuda.Event() for _ in range(nsteps)]
            ev_cp = [torch.cuda.Event() for _ in range(nsteps)]
            ev_out = [torch.cuda.Event() for _ in range(nsteps)]
            if start is not None:
                start.record(s_in)
            for i in range(nsteps):
                b = i % 2
                with torch.cuda.stream(s_in):
                    if i >= 2:
                        s_in.wait_event(ev_cp[i - 2])  # step i-2 is done reading input set b
                    xs[b].copy_(xh, non_blocking=True)
                    dys[b].copy_(dyh, non_blocking=True)
                    ev_in[i].record(s_in)
                stream.wait_event(ev_in[i])
                if i >= 2:
                    stream.wait_event(ev_out[i - 2])  # step i-2's results have left output set b
                wtconv.wtconv_fwd(xs[b], wb, bb, wsub, sb, sw, L, k, y=yd[b], stream=stream)
                wtconv.wtconv_bwd(xs[b], dys[b], wb, bb, wsub, sb, sw, L, k, dx=dxd[b], grads=gd[b], workspace=ws,
                                  stream=stream)
                ev_cp[i].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_cp[i])
                    yh[b].copy_(yd[b], non_blocking=True)
                    dxh[b].copy_(dxd[b], non_blocking=True)
                    for n, t in gd[b].items():
                        gh[b][n].copy_(t, non_blocking=True)
                    ev_out[i].record(s_out)
            if end is not None:
                s_out.wait_event(ev_out[nsteps - 1])
                end.record(s_out)

        e2e_run(3)
        torch.cuda.synchronize()
        barrier(world)
        s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e2e_run(args.steps, s2, e2)
        torch.cuda.synchronize()
        barrier(world)
        e2e_ms = max_over_ranks(world, s2.elapsed_time(e2), dev)
        h2d = 2 * xh.numel() * xh.element_size()
        d2h = 2 * yh[0].numel() * yh[0].element_size() + sum(t.numel() * 4 for t in gh[0].values())
        e2e = {"value": round(e2e_ms / (args.steps * world), 4), "unit": "ms/layer",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "pipelined": "copies in / layer / copies out on three streams, two buffer sets"}

    if rank != 0:
        return None
    peaks, peak_kind = measured_peaks()
    e = ESIZE[inp.dtype]
    ne = inp.numel
    # algorithmic bytes: fwd reads x, writes y; the fused backward reads x and
    # dy once and writes dx (5 element transfers per element per step)
    alg_bytes = {"fwd": 2 * ne * e, "bwd": 3 * ne * e}
    fma = fma_per_plane(inp.H, inp.W, L, k) * inp.N * inp.C  # one pass: fwd, dx, or the dW correlations
    fma_kernel = {"fwd": fma, "bwd": 2 * fma}
    ms_step = elapsed_ms / args.steps
    step_bytes = sum(alg_bytes.values())
    hbm_tbs = step_bytes / (ms_step * 1e-3) / 1e12
    dom = max(avg, key=avg.get)
    clocks = clk.summary()
    num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    alu_peak = num_sms * FP32_LANES * 2 * SM_MAX_MHZ * 1e6 / 1e12  # TFLOP/s at the maximum SM clock
    achieved_alu = 2 * fma_kernel[dom] / (avg[dom] * 1e-3) / 1e12
    roofline = {"bound": "alu", "kernel": dom, "achieved": round(achieved_alu, 2), "peak": round(alu_peak, 2),
                "unit": "TFLOP/s", "frac": round(achieved_alu / alu_peak, 4), "traffic": measured_traffic(dom),
                "traffic_unit": "bytes per launch (ncu dram read+write)",
                "peak_source": f"{num_sms} SMs x {FP32_LANES} FP32 FMA/clk x 2 x {SM_MAX_MHZ:.0f} MHz",
                "algorithmic_fma_per_launch": fma_kernel[dom],
                "timed_span": "bwd = the fused backward kernel and its dW finalize (one C call)" if dom == "bwd"
                else "the forward kernel"}
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
        "separate_bwd_ms": {kn: round(v, 4) for kn, v in separate.items()} | {
            "note": "the backward as wtconv_bwd_data + wtconv_bwd_weight, timed after the step; not in the value"},
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
        workers = max(1, min(os.cpu_count() or 1, inp.N))
        tp = time_oracle_parallel(inp, workers)
        line["cpu_baseline_all_cores"] = {"value": round(1e3 * tp, 1), "unit": "ms/layer", "cores": workers,
                                          "kind": "oracle",
                                          "sample": f"the same fwd+bwd over all {inp.N} images, split over "
                                                    f"{workers} threads"}
    if world == 1 and not args.no_compare:
        comps = []
        for name, dtype in ((WORKLOAD, None), (WORKLOAD, "f16")):
            try:
                w_inp = synth.workload(name, **({"dtype": dtype} if dtype else {}))
                comps.append(compare_arms(w_inp, dev))
            except Exception as exc:  # a comparison arm must not sink the bench line
                comps.append({"workload": name, "dtype": dtype, "error": repr(exc)[:200]})
        line["comparisons"] = {"arms": comps, "context": PAGES_CONTEXT}
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
    ap.add_argument("--no-compare", action="store_true",
                    help="skip the unfused-PyTorch and depthwise-7x7 comparison arms")
    ap.add_argument("--suite", choices=["sweep", "network", "configs", "large"], default=None,
                    help="time the shape/level sweep, the 18-layer network, every workload with the "
                         "oracle beside it, or the planes larger than one CTA, instead of the bench step")
    ap.add_argument("--large-case", type=int, default=None,
                    help="with --suite large: time only this entry of synth.LARGE_PLANES")
    ap.add_argument("--arm-only", default=None,
                    choices=["fused", "unfused", "dw7x7", "fused_infer", "unfused_infer", "dw7x7_infer"],
                    help="run only this arm's training step or forward (steps + warmup times, no JSON); "
                         "for profilers")
    ap.add_argument("--cpu-dist", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args(argv)
    world, rank, local = setup_dist(args)
    if args.suite:
        run_suite(args)
    elif args.arm_only:
        run_arm_only(args)
    elif args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
