"""Benchmark of the exact FlashAttention-2 forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload c4]

One step = one forward pass over each mask mode of the workload (default c4,
the largest: B=1, H=32, Lq=Lk=16384, D=128, bf16, causal), inputs resident in
HBM, L2 flushed (a 256 MiB write) before every launch.  Metric: attention
forward TFLOP/s with FLOPs = 4*B*H*Lq*Lk*D, halved for causal, plus the
fraction of the measured dense-bf16 tensor peak.  Prints one JSON line, which
also carries the other workloads (B2 H16 L4096 D128 both modes, B4 H16 L1024
D64 both modes, B2 H8 Lq2000 Lk3000 D256) timed the same way in `per_config`.

--impl reference times the fp64 CPU oracle (the parity reference) on the
host cores on a bounded sample of the same workload's rows.

With torchrun (WORLD_SIZE > 1) every rank runs the same per-GPU workload on
its own GPU (weak scaling, no data exchange); the timed region is bracketed by
barriers and the max over ranks is reported.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from io_aware_exact_fa2_gb300.workloads import WORKLOADS, workload_inputs  # noqa: E402

METRIC = "attention fwd TFLOP/s (1×GB300) and % of dense BF16 tensor peak"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20


# ---------------------------------------------------------------- helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def load_traffic(kernel_digest: str, workload: str):
    """DRAM bytes per launch of `workload` from the committed ncu summary, if it was
    taken on this kernel source (None otherwise)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as fh:
        d = json.load(fh)
    if d.get("kernel_source_digest") != kernel_digest:
        return None
    return d.get("workloads", {}).get(workload)


class ClockSampler:
    """nvidia-smi samples (every 100 ms) of SM clock and throttle reasons during a region."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)  # let the first sample land before the timed region

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=2)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        return self.summarize(self.lines, t0, t1)

    @staticmethod
    def summarize(lines, t0: float, t1: float):
        """Median SM clock, max clock, throttle reasons seen, from (time, csv line) samples
        taken within [t0, t1] (all samples if none fall inside)."""
        rows = []
        for ts, line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((ts, parts))
        inside = [r for ts, r in rows if t0 - 0.1 <= ts <= t1 + 0.1] or [r for _, r in rows]
        mhz = [float(r[1]) for r in inside if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in inside if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(mhz) if mhz else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside),
                "power_w_max": max((float(r[3]) for r in inside
                                    if r[3].replace(".", "").isdigit()), default=None)}


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
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- oracle timing
_INPUT_CACHE = {}


def oracle_sample_run(w, budget_s: float, seed: int = 0):
    """Time the fp64 oracle on random rows of both modes for about budget_s seconds.

    Returns (TFLOP/s in the metric's units, description, threads used, seconds)."""
    import oracle
    if w.name not in _INPUT_CACHE:
        _INPUT_CACHE[w.name] = workload_inputs(w)
    q, k, v = _INPUT_CACHE[w.name]
    rng = np.random.default_rng(seed)
    n_rows_total = w.B * w.H * w.Lq
    threads = oracle.max_threads()
    flops = 0.0
    elapsed = 0.0
    parts = []
    for mode in w.modes:
        causal = mode == "causal"
        per_row = w.flops(causal) / n_rows_total
        # calibrate on a small batch, then size the timed batch to the budget
        probe = rng.integers(0, n_rows_total, size=max(threads * 4, 64))
        t = time.perf_counter()
        oracle.attention_rows(q, k, v, causal, w.scale, probe)
        rate = probe.size / max(time.perf_counter() - t, 1e-6)
        n = int(min(n_rows_total, max(threads, rate * budget_s / len(w.modes))))
        rows = rng.integers(0, n_rows_total, size=n)
        t = time.perf_counter()
        oracle.attention_rows(q, k, v, causal, w.scale, rows)
        dt = time.perf_counter() - t
        flops += per_row * n
        elapsed += dt
        parts.append(f"{n} random {mode} rows")
    desc = (f"{w.name} B{w.B} H{w.H} Lq{w.Lq} Lk{w.Lk} D{w.D}: " + ", ".join(parts)
            + f" of {n_rows_total} per mode; fp64 oracle, FLOPs credited per row by the metric formula")
    return flops / elapsed / 1e12, desc, threads, elapsed


# ---------------------------------------------------------------- arms
def run_reference(args, world, rank):
    if rank != 0:
        return
    w = WORKLOADS[args.workload]
    per_step = min(4.0, 150.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample_run(w, per_step, seed=1)
    vals, times, desc, threads = [], [], "", 1
    for s in range(args.steps):
        v, desc, threads, dt = oracle_sample_run(w, per_step, seed=100 + s)
        vals.append(v)
        times.append(dt)
    value = float(np.mean(vals))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * float(np.mean(times)),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# tile configuration of the forward kernel per head dimension (fa2_fwd_d*.cu defaults)
FWD_KERNEL_LABEL = {64: "fa2::fwd_kernel<D=64,BN=128,NQ=2>", 128: "fa2::fwd_kernel<D=128,BN=128,NQ=2>",
                    256: "fa2::fwd_kernel<D=256,BN=64,NQ=1,Q in TMEM>"}
# the other workloads, timed beside the headline in the same run (context, not the headline)
PER_CONFIG = [("c3", "noncausal"), ("c3", "causal"), ("c2", "noncausal"), ("c2", "causal"),
              ("c5", "noncausal"), ("c4", "causal")]
BWD_DIMS = (64, 128, 256)
# the e4m3 forward (fa2_fwd_fp8) on the D = 128 workloads' shapes; its peak is the measured
# bf16 peak times the nominal fp8 / bf16 dense ratio (4.5 / 2.25 PFLOP/s)
FP8_CONFIG = [("c3", "noncausal"), ("c3", "causal"), ("c4", "causal")]
FP8_PEAK_RATIO = 2.0


def workload_config(w):
    return {"workload": f"{w.name}: B{w.B} H{w.H} Lq{w.Lq} Lk{w.Lk} D{w.D} bf16, "
                        + " + ".join(w.modes) + " per step",
            "B": w.B, "H": w.H, "Lq": w.Lq, "Lk": w.Lk, "D": w.D, "modes": list(w.modes),
            "scale": "1/sqrt(D)", "l2": "flushed (256 MiB write) before every timed launch"}


class Problem:
    """One workload's inputs and outputs resident on the device."""

    def __init__(self, w, dev):
        q, k, v = workload_inputs(w)
        self.w, self.dev = w, dev
        self.q_host, self.k_host, self.v_host = q, k, v
        self.q, self.k, self.v = q.to(dev), k.to(dev), v.to(dev)
        self.o = torch.empty(w.B, w.H, w.Lq, w.D, dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty(w.B, w.H, w.Lq, dtype=torch.float32, device=dev)


def time_launches(launch, flush, stream, steps: int, warmup: int):
    """CUDA-event duration (ms) of each of `steps` launches, L2 flushed before each."""
    for i in range(warmup):
        flush.fill_(float(i))
        launch()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        flush.fill_(float(i))
        ev[i][0].record(stream)
        launch()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def check_device_error(stream, what):
    from io_aware_exact_fa2_gb300 import fa2_get_device_error
    st, code = fa2_get_device_error(stream)
    if st != 0:
        raise RuntimeError(f"device error {st} code {code:#x} in {what}")


def time_backward(pb, causal, flush, stream, steps, warmup, window=None):
    """Mean CUDA-event ms of fa2_bwd (or fa2_bwd_window) on a resident problem."""
    from io_aware_exact_fa2_gb300 import (fa2_bwd, fa2_bwd_window, fa2_bwd_workspace_size, fa2_fwd,
                                          fa2_fwd_window)
    w, dev = pb.w, pb.dev
    g = torch.Generator(device="cpu").manual_seed(w.seed_base + 7)
    dout = torch.randn(w.B, w.H, w.Lq, w.D, generator=g).to(torch.bfloat16).to(dev)
    dq, dk, dv = torch.empty_like(pb.q), torch.empty_like(pb.k), torch.empty_like(pb.v)
    bws = torch.empty(max(fa2_bwd_workspace_size(w.B, w.H, w.Lq, w.Lk, w.D), 16), dtype=torch.uint8, device=dev)
    if window is None:
        fa2_fwd(pb.q, pb.k, pb.v, pb.o, pb.lse, causal, w.scale, stream=stream)

        def launch():
            fa2_bwd(pb.q, pb.k, pb.v, pb.o, pb.lse, dout, dq, dk, dv, causal, w.scale, stream=stream, workspace=bws)
    else:
        fa2_fwd_window(pb.q, pb.k, pb.v, pb.o, pb.lse, window, w.scale, stream=stream)

        def launch():
            fa2_bwd_window(pb.q, pb.k, pb.v, pb.o, pb.lse, dout, dq, dk, dv, window, w.scale, stream=stream,
                           workspace=bws)
    ms = time_launches(launch, flush, stream, steps, max(2, warmup))
    check_device_error(stream, "the backward pass")
    return float(np.mean(ms))


def run_ours(args, world, rank, local):
    from io_aware_exact_fa2_gb300 import build as fa2_build
    from io_aware_exact_fa2_gb300 import fa2_fwd, fa2_fwd_from_host, fa2_workspace

    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    w = WORKLOADS[args.workload]
    pb = Problem(w, dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    modes = [m == "causal" for m in w.modes]
    # per-mode workspace (allocated once, outside the timed region; None where the
    # library estimates that whole query tiles already balance the SMs)
    workspaces = [fa2_workspace(pb.q, pb.k, causal) for causal in modes]

    def step(events=None):
        for i, causal in enumerate(modes):
            flush.fill_(float(i))
            if events is not None:
                events[i][0].record(stream)
            fa2_fwd(pb.q, pb.k, pb.v, pb.o, pb.lse, causal, w.scale, stream=stream, workspace=workspaces[i])
            if events is not None:
                events[i][1].record(stream)

    for _ in range(args.warmup):
        step()
    check_device_error(stream, "the warm-up")

    evs = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
            for _ in modes] for _ in range(args.steps)]
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = time.time()
    for s in range(args.steps):
        step(evs[s])
    torch.cuda.synchronize(dev)
    barrier(world)
    t1 = time.time()
    clocks = sampler.stop(t0, t1) if sampler else None
    check_device_error(stream, "the timed region")

    per_mode_ms = [[evs[s][i][0].elapsed_time(evs[s][i][1]) for s in range(args.steps)]
                   for i in range(len(modes))]
    dev_ms_total = float(sum(sum(x) for x in per_mode_ms))
    dev_ms_total = max_over_ranks(dev_ms_total, world, dev)
    flops_step = sum(w.flops(c) for c in modes)
    value = world * flops_step * args.steps / (dev_ms_total * 1e-3) / 1e12
    ms_per_step = dev_ms_total / args.steps

    # ---- end to end through the host-buffer entry point (pinned host memory)
    qh, kh, vh = pb.q_host.pin_memory(), pb.k_host.pin_memory(), pb.v_host.pin_memory()
    oh = torch.empty(w.B, w.H, w.Lq, w.D, dtype=torch.bfloat16).pin_memory()
    lh = torch.empty(w.B, w.H, w.Lq, dtype=torch.float32).pin_memory()
    e2e_steps = max(3, min(args.steps, 20))

    def e2e_step():
        for causal in modes:
            fa2_fwd_from_host(qh, kh, vh, oh, lh, pb.q, pb.k, pb.v, pb.o, pb.lse, causal, w.scale, stream=stream)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    check_device_error(stream, "the end-to-end region")
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    e2e_value = world * flops_step * e2e_steps / (e2e_ms * 1e-3) / 1e12
    in_bytes = (pb.q.numel() + pb.k.numel() + pb.v.numel()) * 2
    out_bytes = pb.o.numel() * 2 + pb.lse.numel() * 4

    # the host link itself (what bounds the end-to-end number): plain pinned copies of
    # Q in and O out, three of each, CUDA events on the same stream
    def link_gbs(dst, src):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        dst.copy_(src, non_blocking=True)
        ev[0].record(stream)
        for _ in range(3):
            dst.copy_(src, non_blocking=True)
        ev[1].record(stream)
        torch.cuda.synchronize(dev)
        return 3 * src.numel() * src.element_size() / (ev[0].elapsed_time(ev[1]) * 1e-3) / 1e9
    link = {"h2d_gbs": link_gbs(pb.q, qh), "d2h_gbs": link_gbs(oh, pb.o)}
    del qh, kh, vh, oh, lh

    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops"])

    # ---- backward pass of the headline workload (context, not the headline metric)
    backward = {}
    if not args.no_backward and w.D in BWD_DIMS:
        for causal in modes:
            ms = max_over_ranks(time_backward(pb, causal, flush, stream, args.steps, args.warmup), world, dev)
            tf = 2.5 * w.flops(causal) / (ms * 1e-3) / 1e12
            backward["causal" if causal else "noncausal"] = {"ms": ms, "tflops": tf, "frac_of_peak": tf / peak}

    # ---- sliding-window pass (context): causal with keys i - window <= j <= i
    window = None
    if args.window is not None and w.Lq <= w.Lk:
        from io_aware_exact_fa2_gb300 import fa2_fwd_window
        fwd_ms = time_launches(lambda: fa2_fwd_window(pb.q, pb.k, pb.v, pb.o, pb.lse, args.window, w.scale,
                                                      stream=stream), flush, stream, args.steps, max(3, args.warmup))
        check_device_error(stream, "the windowed pass")
        fwd_w_ms = max_over_ranks(float(np.mean(fwd_ms)), world, dev)
        bwd_w_ms = None
        if not args.no_backward and w.D in BWD_DIMS:
            bwd_w_ms = max_over_ranks(time_backward(pb, True, flush, stream, args.steps, args.warmup,
                                                    window=args.window), world, dev)
        window = (args.window, fwd_w_ms, bwd_w_ms)
    del pb

    # ---- the other workloads, each timed the same way (after the headline's region)
    per_config = {}
    if not args.no_per_config:
        for name, mode in PER_CONFIG:
            wc = WORKLOADS[name]
            causal = mode == "causal"
            pc = Problem(wc, dev)
            ws = fa2_workspace(pc.q, pc.k, causal)
            ms = time_launches(lambda: fa2_fwd(pc.q, pc.k, pc.v, pc.o, pc.lse, causal, wc.scale, stream=stream,
                                               workspace=ws), flush, stream, args.steps, args.warmup)
            check_device_error(stream, f"{name} {mode}")
            ms = max_over_ranks(float(np.mean(ms)), world, dev)
            tf = wc.flops(causal) / (ms * 1e-3) / 1e12
            ent = {"ms": ms, "tflops": tf, "frac_of_peak": tf / peak,
                   "shape": f"B{wc.B} H{wc.H} Lq{wc.Lq} Lk{wc.Lk} D{wc.D}",
                   "schedule": ("cost-balanced key-tile ranges per SM (workspace %d B)" % ws.numel()
                                if ws is not None else "whole query tiles")}
            if not args.no_backward and wc.D in BWD_DIMS:
                bms = max_over_ranks(time_backward(pc, causal, flush, stream, args.steps, args.warmup), world, dev)
                btf = 2.5 * wc.flops(causal) / (bms * 1e-3) / 1e12
                ent["backward"] = {"ms": bms, "tflops": btf, "frac_of_peak": btf / peak}
            per_config[f"{name}_{mode}"] = ent
            del pc, ws
        from io_aware_exact_fa2_gb300 import fa2_fwd_fp8
        from io_aware_exact_fa2_gb300.workloads import make_qkv_fp8
        for name, mode in FP8_CONFIG:
            wc = WORKLOADS[name]
            causal = mode == "causal"
            q8, k8, v8, dq, dk, dv = make_qkv_fp8(wc.B, wc.H, wc.Lq, wc.Lk, wc.D, wc.seed_base)
            q8, k8, v8 = q8.to(dev), k8.to(dev), v8.to(dev)
            dq, dk, dv = (torch.from_numpy(d).to(dev) for d in (dq, dk, dv))
            o = torch.empty(wc.B, wc.H, wc.Lq, wc.D, dtype=torch.bfloat16, device=dev)
            lse = torch.empty(wc.B, wc.H, wc.Lq, dtype=torch.float32, device=dev)
            ws = fa2_workspace(o, k8, causal)   # sized as the bf16 problem of the same shape
            ms = time_launches(lambda: fa2_fwd_fp8(q8, k8, v8, dq, dk, dv, o, lse, causal, wc.scale, stream=stream,
                                                   workspace=ws), flush, stream, args.steps, args.warmup)
            check_device_error(stream, f"{name} {mode} fp8")
            ms = max_over_ranks(float(np.mean(ms)), world, dev)
            tf = wc.flops(causal) / (ms * 1e-3) / 1e12
            per_config[f"{name}_{mode}_fp8"] = {
                "ms": ms, "tflops": tf, "frac_of_peak": tf / (peak * FP8_PEAK_RATIO),
                "peak": peak * FP8_PEAK_RATIO, "dtype": "e4m3 in (per-head descales), fp32 accumulate, bf16 out",
                "shape": f"B{wc.B} H{wc.H} Lq{wc.Lq} Lk{wc.Lk} D{wc.D}",
                "schedule": ("cost-balanced key-tile ranges per SM (workspace %d B)" % ws.numel()
                             if ws is not None else "whole query tiles")}
            del q8, k8, v8, o, lse, ws

    if rank != 0:
        return
    avg_launch_ms = dev_ms_total / (args.steps * len(modes))
    achieved = flops_step / len(modes) / (avg_launch_ms * 1e-3) / 1e12
    traffic = load_traffic(fa2_build.kernel_digest(), w.name)
    per_mode = {}
    for i, c in enumerate(modes):
        ms = float(np.mean(per_mode_ms[i]))
        per_mode["causal" if c else "noncausal"] = {
            "ms": ms, "tflops": w.flops(c) / (ms * 1e-3) / 1e12,
            "frac_of_peak": w.flops(c) / (ms * 1e-3) / 1e12 / peak,
            "schedule": ("cost-balanced key-tile ranges per SM (fa2_fwd_ws, workspace %d B)" % workspaces[i].numel()
                         if workspaces[i] is not None else "whole query tiles (fa2_fwd)")}
    cpu_val, cpu_desc, cpu_threads, _ = (oracle_sample_run(w, args.cpu_budget)
                                        if (world == 1 and not args.no_cpu_baseline) else (None, "", 0, 0))
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(w),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                     "frac": achieved / peak,
                     "peak_source": f"{peak_src} bf16_tflops (burst: each launch is timed alone)",
                     "traffic": (traffic["dram_bytes_per_launch"] if traffic else None),
                     "algorithmic_bytes_per_launch": w.algorithmic_bytes(),
                     "kernel": FWD_KERNEL_LABEL[w.D]},
        "per_mode": per_mode,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": in_bytes * len(modes),
                "d2h_bytes_per_step": out_bytes * len(modes),
                "how": "fa2_fwd_from_host per mode: pinned host -> device copies, kernels "
                       "(whole-query-tile schedule) and device -> host copies of O and LSE, "
                       "overlapped over chunks of heads, all inside the CUDA-event region",
                "host_link_gbs": link},
        "gpu_launches": args.steps * len(modes),
        "clocks": clocks,
    }
    if cpu_val is not None:
        line["cpu_baseline"] = {"value": cpu_val, "unit": UNIT, "cores": cpu_threads, "kind": "oracle",
                                "sample": cpu_desc}
    if backward:
        line["backward"] = {
            "metric": "attention bwd TFLOP/s (FLOPs = 2.5 x the forward's: the five matmuls of dS, dP, dV, "
                      "dK, dQ; the kernels also recompute S and dP for dQ)",
            "unit": UNIT, "per_mode": backward,
            "kernels": "Delta, dQ (query tiles resident), dK/dV (key tiles resident) per call (fa2_bwd)",
            "l2": "flushed (256 MiB write) before every timed call"}
    if per_config:
        line["per_config"] = dict(
            per_config, note="each workload and mode timed like the headline (CUDA events per launch, L2 "
                             "flushed before each, mean of --steps launches after --warmup); frac_of_peak "
                             "against the same measured bf16 peak (the *_fp8 lines: that peak x 2, the "
                             "nominal fp8/bf16 dense ratio); backward FLOPs = 2.5 x the forward's")
    if window is not None:
        wv, ms, bms = window
        tf = window_flops(w, wv) / (ms * 1e-3) / 1e12
        line["window"] = {
            "metric": "sliding-window attention fwd TFLOP/s, FLOPs = 4 D per visible (query, key) pair",
            "window": wv, "ms": ms, "tflops": tf, "frac_of_peak": tf / peak, "unit": UNIT,
            "l2": "flushed (256 MiB write) before every timed launch"}
        if bms is not None:
            btf = 2.5 * window_flops(w, wv) / (bms * 1e-3) / 1e12
            line["window"]["backward"] = {"ms": bms, "tflops": btf, "frac_of_peak": btf / peak,
                                          "flops": "2.5 x the windowed forward's (fa2_bwd_window)"}
    print(json.dumps(line), flush=True)


def window_flops(w, window: int) -> float:
    """4 * D FLOPs per visible pair: query i sees keys max(0, i - window) .. i (Lq <= Lk)."""
    lq, n = w.Lq, window + 1
    pairs = lq * (lq + 1) // 2 if lq <= n else n * (n + 1) // 2 + (lq - n) * n
    return 4.0 * w.B * w.H * w.D * pairs


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="c4")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle work for the cpu_baseline field")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-backward", action="store_true", help="skip the backward-pass timing")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip timing the other workloads beside the headline")
    ap.add_argument("--window", type=int, default=None,
                    help="also time the sliding-window pass with this window (keys i - window .. i)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
