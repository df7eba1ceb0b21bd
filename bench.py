"""Benchmark of the PTB forward pass (y = x + MLP(LN(x)) + Attn(LN(x)), causal
sliding-window attention) on GB300.

One step = one full layer forward (LayerNorm, [QKV | up] GEMM + GELU,
banded SWA, [out | down] GEMM + residual) over one micro-batch of the
175B-shaped layer of MegaScale's Table 1 (hidden 12288, 128 heads x 96,
MLP 4H, seq 2048, window 1024) with synthetic seeded bf16 inputs resident
in HBM.  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload 175b|13b|530b|tiny|swa]

--impl reference times the fp64 CPU oracle (the only other implementation
there is) on a bounded sample of the same workload on the host's cores.
Under torchrun each rank runs an independent replica of the layer (weak
scaling, no collective in the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from block_sliding_window_gb300 import workloads  # noqa: E402

METRIC = "PTB-layer fwd tokens/s and TFLOP/s (bf16) on 1 GB300; % of tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
GEMM_SRC = os.path.join(ROOT, "block_sliding_window_gb300", "csrc", "gemm_tcgen05.cu")
SWA_SRC = os.path.join(ROOT, "block_sliding_window_gb300", "csrc", "swa_tcgen05.cu")


def event_steps(steps: int) -> list:
    """The timed steps that record per-kernel CUDA events: every tenth one
    (every one in runs under 30 steps).  Five event records per step held
    back the launch-bound tiny layer by 38% and the 13B-class layer by 1.3%
    (the 175B-class one not measurably), so they go on a sample of the timed
    steps, which still gives each kernel's average from live launches."""
    stride = 10 if steps >= 30 else 1
    return list(range(0, steps, stride))
TRAIN_METRIC = ("PTB-layer training step (forward + backward) tokens/s and TFLOP/s (bf16) on "
                "1 GB300; % of tensor peak")


def layer_flops(cfg) -> dict:
    """Algorithmic forward FLOPs: exact GEMMs plus in-band attention only."""
    t, h, f, w, s = cfg.tokens, cfg.hidden, cfg.ffn, cfg.window, cfg.seq
    band = sum(min(i + 1, w) for i in range(s))
    gemm1 = 2 * t * h * (3 * h + f)
    gemm2 = 2 * t * (h + f) * h
    attn = 4 * cfg.batch * h * band
    return {"gemm1": gemm1, "gemm2": gemm2, "attn": attn, "total": gemm1 + gemm2 + attn,
            "band_keys": band * cfg.batch * cfg.heads}


def swa_flops(cfg) -> int:
    """Algorithmic FLOPs of the SWA operator: Q K^T and P V over the in-band
    (query, key) pairs only, 4 d per pair and head."""
    band = sum(min(i + 1, cfg.window) for i in range(cfg.seq))
    return 4 * cfg.batch * cfg.heads * cfg.head_dim * band


def backward_flops(cfg) -> dict:
    """Algorithmic backward FLOPs: an input-gradient and a weight-gradient
    GEMM per forward GEMM, and dV, dP, dQ, dK over the in-band pairs."""
    fl = layer_flops(cfg)
    band = fl["band_keys"] // cfg.heads
    attn = 8 * cfg.hidden * band
    gemm = 2 * (fl["gemm1"] + fl["gemm2"])
    return {"dgrad_out": fl["gemm2"], "wgrad_out": fl["gemm2"], "dgrad_in": fl["gemm1"],
            "wgrad_in": fl["gemm1"], "attn": attn, "total": gemm + attn}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def sha_of(path: str):
    try:
        with open(path, "rb") as fh:
            return hashlib.sha256(fh.read()).hexdigest()[:16]
    except OSError:
        return None


def traffic_for(kernel: str, workload: str, src: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current source of the kernel; else None."""
    try:
        with open(TRAFFIC_FILE) as fh:
            entries = json.load(fh)
    except (OSError, ValueError):
        return None
    for e in entries:
        if e.get("kernel") == kernel and e.get("workload") == workload:
            if e.get("source_sha") == sha_of(src):
                return e.get("dram_bytes_per_launch")
    return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,utilization.gpu,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(index), "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, mx, busy_sm, reasons = [], [], [], set()
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 8:
                continue
            try:
                cur, top, util = float(parts[0]), float(parts[1]), float(parts[3])
            except ValueError:
                continue
            sm.append(cur)
            mx.append(top)
            if util > 0:
                busy_sm.append(cur)
                for n, v in zip(names, parts[4:]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        if not sm:
            return None
        pool = busy_sm or sm
        return {"sm_mhz": statistics.median(pool), "sm_max_mhz": max(mx), "samples": len(sm),
                "samples_under_load": len(busy_sm), "reasons": sorted(reasons)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def workload_config(name: str):
    if name == "swa":
        return workloads.SWA_CONFIGS["swa"]
    return workloads.PTB_CONFIGS[name]


def config_json(name: str, cfg, world: int) -> dict:
    if name == "swa":
        return {"workload": (f"SWA operator alone: batch {cfg.batch}, {cfg.heads} heads x "
                             f"{cfg.head_dim}, seq {cfg.seq}, causal window {cfg.window}"),
                "batch": cfg.batch, "seq_len": cfg.seq, "heads": cfg.heads,
                "head_dim": cfg.head_dim, "window": cfg.window,
                "l2": "L2 flushed between steps (256 MB buffer written)",
                "parallelism": f"replicas x{world}"}
    return {"workload": (f"PTB layer forward, {cfg.name} shape: micro-batch {cfg.batch}, seq "
                         f"{cfg.seq}, hidden {cfg.hidden}, {cfg.heads} heads x {cfg.head_dim}, "
                         f"MLP {cfg.hidden}->{cfg.ffn}->{cfg.hidden} tanh-GELU, causal SWA window "
                         f"{cfg.window}"),
            "batch": cfg.batch, "seq_len": cfg.seq, "hidden": cfg.hidden, "heads": cfg.heads,
            "ffn": cfg.ffn, "window": cfg.window, "tokens_per_step_per_gpu": cfg.tokens,
            "l2": (f"inputs larger than L2: {2 * (4 * cfg.hidden ** 2 + 2 * cfg.hidden * cfg.ffn) / 1e9:.2f}"
                   " GB of weights streamed every step"),
            "parallelism": f"replicas x{world} (independent layers, no collective)"}


# ---------------------------------------------------------------- oracle leg --

def oracle_sample(cfg, rows: int, seed_device="cpu"):
    """Host fp64 copies of the layer's inputs for the oracle (not timed)."""
    import numpy as np
    host = workloads.ptb_inputs(cfg, device=seed_device)
    f64 = {k: v.detach().to("cpu").double().numpy() for k, v in host.items()}
    f64["x"] = np.ascontiguousarray(f64["x"][:, :rows])
    return f64


def time_oracle(cfg, f64, rows: int, repeats: int):
    import oracle
    times = []
    for _ in range(repeats):
        t0 = time.perf_counter()
        oracle.ptb_forward(f64["x"], f64["ln_gamma"], f64["ln_beta"], f64["w_qkv"], f64["w_o"],
                           f64["w_up"], f64["w_down"], cfg.heads, cfg.window,
                           rows=list(range(rows)))
        times.append(time.perf_counter() - t0)
    return times


def cpu_threads() -> int:
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        v = os.environ.get(var)
        if v and v.isdigit():
            return int(v)
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def sample_desc(cfg, rows):
    return (f"rows 0..{rows - 1} of batch 0 of the {cfg.name} layer (LN, Q/K/V, banded softmax over"
            f" the keys those rows see, out/up/down projections, all weights), fp64, numpy BLAS")


def run_reference(args, world, rank):
    """The oracle, as it stands, timed on the host cores."""
    if rank != 0:
        return
    name = args.workload if args.workload != "swa" else "175b"
    cfg = workload_config(name)
    rows = args.ref_rows
    f64 = oracle_sample(cfg, rows, seed_device="cuda" if torch.cuda.is_available() else "cpu")
    time_oracle(cfg, f64, rows, max(0, min(args.warmup, 1)))
    times = time_oracle(cfg, f64, rows, args.steps)
    per_step = sum(times) / len(times)
    value = rows / per_step
    fl = layer_flops(cfg)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": per_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "tflops": value * fl["total"] / cfg.tokens / 1e12,
        "config": config_json(name, cfg, 1),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_threads(),
                         "kind": "oracle", "sample": sample_desc(cfg, rows)},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# -------------------------------------------------------------- CUDA path --

def run_swa(args, world, rank, local):
    import block_sliding_window_gb300 as bsw
    cfg = workload_config("swa")
    q, k, v = workloads.swa_inputs(cfg.batch, cfg.heads, cfg.seq, cfg.head_dim, cfg.seed,
                                   device="cuda")
    o = torch.empty_like(q)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        bsw.swa_attention(q, k, v, cfg.window, o=o)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        evs[i][0].record(stream)
        bsw.swa_attention(q, k, v, cfg.window, o=o)
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    per_step = [a.elapsed_time(b) for a, b in evs]
    kern_ms = sum(per_step) / args.steps
    ms = max_over_ranks(kern_ms, world)

    # End to end: q, k and v in from pinned host memory and o out, every
    # step.  Step i's copies run on copy stream i % 2 into and out of device
    # buffers of their own, so one step's copies overlap the neighbouring
    # steps' kernels.
    hosts = [t.cpu().pin_memory() for t in (q, k, v)]
    o_hosts = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for _ in range(2)]
    bufs = [[torch.empty_like(q) for _ in range(4)] for _ in range(2)]  # q, k, v, o
    copy_streams = [torch.cuda.Stream(), torch.cuda.Stream()]

    def copied_step(i):
        cs, b = copy_streams[i % 2], bufs[i % 2]
        with torch.cuda.stream(cs):
            for dst, src in zip(b[:3], hosts):
                dst.copy_(src, non_blocking=True)
            ready = torch.cuda.Event()
            ready.record(cs)
        stream.wait_event(ready)
        bsw.swa_attention(b[0], b[1], b[2], cfg.window, o=b[3])
        done = torch.cuda.Event()
        done.record(stream)
        cs.wait_event(done)
        with torch.cuda.stream(cs):
            o_hosts[i % 2].copy_(b[3], non_blocking=True)

    for i in range(max(2, args.warmup)):
        copied_step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    e0.record(stream)
    for cs in copy_streams:
        cs.wait_event(e0)
    for i in range(args.steps):
        copied_step(i)
    for cs in copy_streams:
        fin = torch.cuda.Event()
        fin.record(cs)
        stream.wait_event(fin)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)
    band = sum(min(i + 1, cfg.window) for i in range(cfg.seq))
    tokens = cfg.batch * cfg.seq
    flops = swa_flops(cfg)
    bytes_ = 4 * q.numel() * 2
    peaks, peak_src = load_peaks()
    ach = bytes_ / (kern_ms * 1e-3) / 1e9
    if rank == 0:
        print(json.dumps({
            "metric": "SWA operator tokens/s (bf16) on 1 GB300", "value": tokens * world / (ms * 1e-3),
            "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic", "config": config_json("swa", cfg, world),
            "tflops": flops / (ms * 1e-3) / 1e12,
            "step_ms": {"mean": kern_ms, "median": statistics.median(per_step),
                        "min": min(per_step)},
            "tensor_frac_of_burst": flops / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
            "exp_per_s": cfg.batch * cfg.heads * band / (ms * 1e-3),
            "roofline": {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": ach / peaks["hbm_gbs"], "peak_source": peak_src,
                         "traffic": traffic_for("swa_kernel", "swa", SWA_SRC)},
            "e2e": {"value": tokens * world / (e2e_ms * 1e-3), "unit": "tokens/s",
                    "h2d_bytes_per_step": 3 * q.numel() * 2, "d2h_bytes_per_step": o.numel() * 2},
            "clocks": clk, "gpu_launches": args.steps}), flush=True)


def run_train(args, world, rank, local):
    """One training step of the layer: ptb_forward_train + ptb_backward."""
    import block_sliding_window_gb300 as bsw
    cfg = workload_config(args.workload)
    d = workloads.ptb_inputs(cfg, device="cuda")
    dy = workloads.normal_bf16(tuple(d["x"].shape), seed=cfg.seed + 1000, device="cuda")
    b, s, h, f = cfg.batch, cfg.seq, cfg.hidden, cfg.ffn
    saved = torch.empty(bsw.train_saved_size(b, s, h, f, cfg.heads), dtype=torch.uint8,
                        device="cuda")
    ws_f = torch.empty(bsw.workspace_size(b, s, h, f), dtype=torch.uint8, device="cuda")
    ws_b = torch.empty(bsw.backward_workspace_size(b, s, h, f, cfg.heads), dtype=torch.uint8,
                       device="cuda")
    y = torch.empty_like(d["x"])
    dev, f32 = "cuda", torch.float32
    grads = dict(dx=torch.empty_like(d["x"]), dln_gamma=torch.empty(h, dtype=f32, device=dev),
                 dln_beta=torch.empty(h, dtype=f32, device=dev),
                 dw_qkv=torch.empty(3 * h, h, dtype=f32, device=dev),
                 dw_o=torch.empty(h, h, dtype=f32, device=dev),
                 dw_up=torch.empty(f, h, dtype=f32, device=dev),
                 dw_down=torch.empty(h, f, dtype=f32, device=dev))
    w = (d["w_qkv"], d["w_o"], d["w_up"], d["w_down"])
    stream = torch.cuda.current_stream()

    def step(x_in, dy_in, marks=None, g=None):
        g = grads if g is None else g
        if marks is not None:
            marks[0].record(stream)
        bsw.ptb_forward_train(x_in, d["ln_gamma"], d["ln_beta"], *w, cfg.heads, cfg.window, y=y,
                              saved=saved, workspace=ws_f)
        if marks is not None:
            return bsw.ptb_backward_events(dy_in, x_in, d["ln_gamma"], *w, saved, cfg.heads,
                                           cfg.window, marks[1:], grads=g, workspace=ws_b)
        return bsw.ptb_backward(dy_in, x_in, d["ln_gamma"], *w, saved, cfg.heads, cfg.window,
                                grads=g, workspace=ws_b)

    for _ in range(args.warmup):
        step(d["x"], dy)
    torch.cuda.synchronize()
    if bsw.last_device_error() != 0:
        raise RuntimeError("device status set during warm-up")
    sampled = event_steps(args.steps)
    marks = {i: [torch.cuda.Event(enable_timing=True) for _ in range(8)] for i in sampled}
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(args.steps):
        step(d["x"], dy, marks.get(i))
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    if bsw.last_device_error() != 0:
        raise RuntimeError("device status set in the timed region")
    ms = max_over_ranks(t0.elapsed_time(t1) / args.steps, world)
    names = ["forward_train", "dgrad_out", "wgrad_out", "swa_backward", "dgrad_in", "wgrad_in",
             "layernorm_backward"]
    per_kernel = {n: sum(m[j].elapsed_time(m[j + 1]) for m in marks.values()) / len(marks)
                  for j, n in enumerate(names)}
    per_step = [m[0].elapsed_time(m[-1]) for m in marks.values()]

    # End to end through the public calls: x and dy in from pinned host
    # memory, dx out, every step (the weight gradients stay on the device
    # for the optimizer).
    # The steps run in order on the launching stream; step i's copies run on
    # copy stream i % 2 into and out of buffers of their own, so one step's
    # copies overlap the neighbouring steps' kernels.
    x_host, dy_host = d["x"].cpu().pin_memory(), dy.cpu().pin_memory()
    dx_host = torch.empty(d["x"].shape, dtype=torch.bfloat16, pin_memory=True)
    dx_hosts = [dx_host, torch.empty(d["x"].shape, dtype=torch.bfloat16, pin_memory=True)]
    x_devs = [torch.empty_like(d["x"]) for _ in range(2)]
    dy_devs = [torch.empty_like(dy) for _ in range(2)]
    g_bufs = [grads, dict(grads, dx=torch.empty_like(d["x"]))]
    copy_streams = [torch.cuda.Stream(), torch.cuda.Stream()]

    def copied_step(i):
        cs = copy_streams[i % 2]
        with torch.cuda.stream(cs):
            x_devs[i % 2].copy_(x_host, non_blocking=True)
            dy_devs[i % 2].copy_(dy_host, non_blocking=True)
            ready = torch.cuda.Event()
            ready.record(cs)
        stream.wait_event(ready)
        step(x_devs[i % 2], dy_devs[i % 2], g=g_bufs[i % 2])
        done = torch.cuda.Event()
        done.record(stream)
        cs.wait_event(done)
        with torch.cuda.stream(cs):
            dx_hosts[i % 2].copy_(g_bufs[i % 2]["dx"], non_blocking=True)

    for i in range(max(2, args.warmup)):
        copied_step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    e0.record(stream)
    for cs in copy_streams:
        cs.wait_event(e0)
    for i in range(args.steps):
        copied_step(i)
    for cs in copy_streams:
        fin = torch.cuda.Event()
        fin.record(cs)
        stream.wait_event(fin)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)

    fwd, bwd = layer_flops(cfg), backward_flops(cfg)
    total = fwd["total"] + bwd["total"]
    peaks, peak_src = load_peaks()
    peak_sus = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
    tokens = cfg.tokens * world
    tflops = total * world / (ms * 1e-3) / 1e12
    # Dominant kernel: the slowest backward GEMM of the step.
    gemms = ["dgrad_out", "wgrad_out", "dgrad_in", "wgrad_in"]
    top = max(gemms, key=lambda n: per_kernel[n])
    top_tf = bwd[top] / (per_kernel[top] * 1e-3) / 1e12
    line = {
        "metric": TRAIN_METRIC, "value": tokens / (ms * 1e-3), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": config_json(args.workload, cfg, world),
        "tflops": tflops,
        "pct_of_peak": {"burst": 100 * tflops / world / peaks["bf16_tflops"],
                        "sustained": 100 * tflops / world / peak_sus, "source": peak_src},
        "kernels_ms": per_kernel, "kernels_ms_sampled_steps": len(marks),
        "step_ms": {"mean": sum(per_step) / len(per_step),
                    "median": statistics.median(per_step), "min": min(per_step)},
        "flops": {"forward": fwd["total"], "backward": bwd["total"]},
        "roofline": {"bound": "tensor", "kernel": f"{top} (tcgen05 GEMM, backward)",
                     "achieved": top_tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": top_tf / peaks["bf16_tflops"],
                     "peak_source": f"{peak_src} bf16 dense (burst)",
                     "frac_of_sustained": top_tf / peak_sus,
                     "traffic": traffic_for(top, args.workload + "_train", GEMM_SRC),
                     "algorithmic_flops_per_launch": bwd[top]},
        "e2e": {"value": tokens / (e2e_ms * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": 2 * x_host.numel() * 2,
                "d2h_bytes_per_step": dx_host.numel() * 2},
        "clocks": clk,
        "gpu_launches": 14 * args.steps,
        "cpu_baseline": None,
        "cpu_baseline_note": "the fp64 backward oracle has no row-sampled form; see --pass forward",
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_ours(args, world, rank, local):
    import block_sliding_window_gb300 as bsw
    from block_sliding_window_gb300 import build as _build
    _build.build()
    bsw.load()
    if args.workload == "swa":
        return run_swa(args, world, rank, local)
    if args.pass_ == "train":
        return run_train(args, world, rank, local)
    cfg = workload_config(args.workload)
    d = workloads.ptb_inputs(cfg, device="cuda")
    serial = args.block == "serial"
    fp8 = args.precision == "fp8"
    w8 = None
    if fp8:  # weights quantized once, outside the timed region
        w8 = bsw.prepare_fp8_weights(d["w_qkv"], d["w_o"], d["w_up"], d["w_down"])
        ws = torch.empty(bsw.fp8_workspace_size(cfg.batch, cfg.seq, cfg.hidden, cfg.ffn),
                         dtype=torch.uint8, device="cuda")
    elif serial:
        ws = torch.empty(bsw.serial_workspace_size(cfg.batch, cfg.seq, cfg.hidden, cfg.ffn),
                         dtype=torch.uint8, device="cuda")
    else:
        ws = torch.empty(bsw.workspace_size(cfg.batch, cfg.seq, cfg.hidden, cfg.ffn),
                         dtype=torch.uint8, device="cuda")
    y = torch.empty_like(d["x"])
    fwd_args = (d["x"], d["ln_gamma"], d["ln_beta"], d["w_qkv"], d["w_o"], d["w_up"],
                d["w_down"], cfg.heads, cfg.window)
    stream = torch.cuda.current_stream()

    def layer(x_in, marks=None, y_out=None):
        y_out = y if y_out is None else y_out
        if fp8:
            if marks is not None:
                return bsw.ptb_forward_fp8_events(x_in, d["ln_gamma"], d["ln_beta"], w8,
                                                  cfg.heads, cfg.window, marks, y=y_out,
                                                  workspace=ws)
            return bsw.ptb_forward_fp8(x_in, d["ln_gamma"], d["ln_beta"], w8, cfg.heads,
                                       cfg.window, y=y_out, workspace=ws)
        if serial:  # second LayerNorm: gamma = 1, beta = 0 like the first
            return bsw.serial_forward(x_in, d["ln_gamma"], d["ln_beta"], d["ln_gamma"],
                                      d["ln_beta"], *fwd_args[3:], y=y_out, workspace=ws)
        if marks is not None:
            return bsw.ptb_forward_events(x_in, *fwd_args[1:], marks, y=y_out, workspace=ws)
        return bsw.ptb_forward(x_in, *fwd_args[1:], y=y_out, workspace=ws)

    for _ in range(args.warmup):
        layer(d["x"])
    torch.cuda.synchronize()
    if bsw.last_device_error() != 0:
        raise RuntimeError("device status set during warm-up")

    # Timed region: K steps, per-kernel events recorded on the launching stream.
    n_marks = 6 if fp8 else 5
    sampled = [] if serial else event_steps(args.steps)
    marks = {i: [torch.cuda.Event(enable_timing=True) for _ in range(n_marks)] for i in sampled}
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)  # sampled over the timed and the e2e regions
    barrier(world)
    torch.cuda.synchronize()
    t_start.record(stream)
    for i in range(args.steps):
        layer(d["x"], marks.get(i))
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    status = bsw.last_device_error()
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")
    ms_local = t_start.elapsed_time(t_end) / args.steps
    ms = max_over_ranks(ms_local, world)
    names = (["layernorm_quantize", "gemm_qkv_up", "swa", "quantize_ctx_g", "gemm_out_down"]
             if fp8 else ["layernorm", "gemm_qkv_up", "swa", "gemm_out_down"])
    per_kernel = None if serial else {
        n: sum(m[j].elapsed_time(m[j + 1]) for m in marks.values()) / len(marks)
        for j, n in enumerate(names)}
    step_stats = None
    if not serial:  # one step = first to last boundary event of that step
        per_step = [m[0].elapsed_time(m[-1]) for m in marks.values()]
        step_stats = {"mean": sum(per_step) / len(per_step),
                      "median": statistics.median(per_step), "min": min(per_step)}

    # End to end with host buffers: every step copies x in and y out.  The
    # PTB layer goes through ptb_forward_host (the C-ABI call on host
    # memory) on two streams in turn, so one step's copies overlap the other
    # step's kernels; the other blocks copy with torch on the launching
    # stream.
    x_host = d["x"].cpu().pin_memory()
    y_host = torch.empty(d["x"].shape, dtype=torch.bfloat16, pin_memory=True)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if not serial and not fp8:
        y_hosts = [y_host, torch.empty(d["x"].shape, dtype=torch.bfloat16, pin_memory=True)]
        streams = [torch.cuda.Stream(), torch.cuda.Stream()]
        hws = [torch.empty(bsw.host_workspace_size(cfg.batch, cfg.seq, cfg.hidden, cfg.ffn),
                           dtype=torch.uint8, device="cuda") for _ in range(2)]

        def host_step(i):
            bsw.ptb_forward_host(x_host, d["ln_gamma"], d["ln_beta"], d["w_qkv"], d["w_o"],
                                 d["w_up"], d["w_down"], cfg.heads, cfg.window, y_hosts[i % 2],
                                 hws[i % 2], stream=streams[i % 2])

        for i in range(max(2, args.warmup)):
            host_step(i)
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        e0.record(stream)
        for st in streams:
            st.wait_event(e0)
        for i in range(args.steps):
            host_step(i)
        for st in streams:
            done = torch.cuda.Event()
            done.record(st)
            stream.wait_event(done)
        e1.record(stream)
    else:
        # The layers run in order on the launching stream; step i's copies
        # run on copy stream i % 2 into and out of buffers of their own, so
        # one step's copies overlap the neighbouring steps' layers.
        x_devs = [torch.empty_like(d["x"]) for _ in range(2)]
        y_devs = [torch.empty_like(d["x"]) for _ in range(2)]
        y_hosts = [y_host, torch.empty(d["x"].shape, dtype=torch.bfloat16, pin_memory=True)]
        copy_streams = [torch.cuda.Stream(), torch.cuda.Stream()]

        def copied_step(i):
            cs = copy_streams[i % 2]
            with torch.cuda.stream(cs):
                x_devs[i % 2].copy_(x_host, non_blocking=True)
                ready = torch.cuda.Event()
                ready.record(cs)
            stream.wait_event(ready)
            layer(x_devs[i % 2], y_out=y_devs[i % 2])
            done = torch.cuda.Event()
            done.record(stream)
            cs.wait_event(done)
            with torch.cuda.stream(cs):
                y_hosts[i % 2].copy_(y_devs[i % 2], non_blocking=True)

        for i in range(max(2, args.warmup)):
            copied_step(i)
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        e0.record(stream)
        for cs in copy_streams:
            cs.wait_event(e0)
        for i in range(args.steps):
            copied_step(i)
        for cs in copy_streams:
            fin = torch.cuda.Event()
            fin.record(cs)
            stream.wait_event(fin)
        e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)

    fl = layer_flops(cfg)
    peaks, peak_src = load_peaks()
    tokens = cfg.tokens * world
    value = tokens / (ms * 1e-3)
    tflops = fl["total"] * world / (ms * 1e-3) / 1e12
    peak_sus = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
    roofline = None
    if per_kernel:
        g1_tf = fl["gemm1"] / (per_kernel["gemm_qkv_up"] * 1e-3) / 1e12
        # The timed region is a fraction of a second, so the denominator is
        # the burst (dense) peak; the fraction of the seconds-long sustained
        # figure is reported beside it, labelled.
        roofline = {"bound": "tensor", "kernel": "gemm_qkv_up (tcgen05 [QKV|up] GEMM + GELU)",
                    "achieved": g1_tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                    "frac": g1_tf / peaks["bf16_tflops"],
                    "peak_source": f"{peak_src} bf16 dense (burst)",
                    "frac_of_sustained": g1_tf / peak_sus,
                    "traffic": traffic_for("gemm_qkv_up", args.workload, GEMM_SRC),
                    "algorithmic_flops_per_launch": fl["gemm1"]}
        if fp8:  # e4m3 peak = measured bf16 x the nominal 4.5 : 2.25 dense ratio
            fp8_burst = 2.0 * peaks["bf16_tflops"]
            roofline.update(kernel="gemm_qkv_up (tcgen05 e4m3 [QKV|up] GEMM + GELU)",
                            peak=fp8_burst, frac=g1_tf / fp8_burst,
                            peak_source=f"{peak_src} bf16 dense (burst) x 2 (nominal e4m3:bf16)",
                            frac_of_sustained=g1_tf / (2.0 * peak_sus),
                            traffic=traffic_for("fp8_gemm_qkv_up", args.workload, GEMM_SRC))
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_json(args.workload, cfg, world),
        "tflops": tflops,
        "pct_of_peak": {"burst": 100 * tflops / world / peaks["bf16_tflops"],
                        "sustained": 100 * tflops / world / peak_sus, "source": peak_src},
        "kernels_ms": per_kernel, "kernels_ms_sampled_steps": len(marks),
        "step_ms": step_stats,
        "roofline": roofline,
        "e2e": {"value": tokens / (e2e_ms * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": x_host.numel() * 2, "d2h_bytes_per_step": y_host.numel() * 2},
        "clocks": clk,
        "gpu_launches": (7 if serial else 4) * args.steps,
    }
    if serial:
        line["block"] = "serial (h = x + Attn(LN1(x)), y = h + MLP(LN2(h)))"
    if fp8:
        line["dtype"] = "e4m3 GEMM operands (per-row scales), bf16 activations and attention"
        line["gpu_launches"] = 5 * args.steps
        # nominal e4m3 / bf16 dense ratio 4.5 / 2.25
        line["pct_of_peak"] = {
            "fp8_burst_nominal_ratio": 100 * tflops / world / (2.0 * peaks["bf16_tflops"]),
            "fp8_sustained_nominal_ratio": 100 * tflops / world / (2.0 * peak_sus),
            "bf16_burst": 100 * tflops / world / peaks["bf16_tflops"],
            "source": f"{peak_src} bf16 x 2"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not serial and not fp8:
        f64 = oracle_sample(cfg, args.cpu_rows, seed_device="cuda")
        times = time_oracle(cfg, f64, args.cpu_rows, 1)
        cpu_v = args.cpu_rows / times[0]
        line["cpu_baseline"] = {"value": cpu_v, "unit": "tokens/s", "cores": cpu_threads(),
                                "kind": "oracle", "sample": sample_desc(cfg, args.cpu_rows),
                                "seconds": times[0]}
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["175b", "13b", "530b", "tiny", "swa"], default="175b")
    ap.add_argument("--block", choices=["ptb", "serial"], default="ptb",
                    help="the parallel block (default) or the serial block it replaces")
    ap.add_argument("--precision", choices=["bf16", "fp8"], default="bf16",
                    help="bf16 (default) or the variant with e4m3 GEMM operands")
    ap.add_argument("--pass", dest="pass_", choices=["forward", "train"], default="forward",
                    help="the layer forward (default) or a training step (forward + backward)")
    ap.add_argument("--cpu-rows", type=int, default=1024,
                    help="rows of the layer the CPU baseline computes (about 10 s of oracle work)")
    ap.add_argument("--ref-rows", type=int, default=64,
                    help="rows per step of the reference arm (the oracle)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    world, rank, local = dist_setup()
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
