#!/usr/bin/env python3
"""Benchmark of the attention backward (preprocess + main + dQ finalise) on
GB300, printing one JSON line.

Workload: bf16, B=4, H=32, H_kv=8 (GQA 4:1), S_q=S_k=2048, d=128, causal,
scale=1/sqrt(d); Q, K, V ~ N(0,1), dO ~ N(0, 0.1^2) (seeded, synthetic), O and
LSE from the library forward.  Metric: attention-backward TFLOP/s counting
10*B*H*S_q*S_k*d flops, halved for causal.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

`value` times K fa_bwd calls with inputs resident in HBM (CUDA events on the
launching stream, L2 flushed by a 256 MiB write between steps, outside the
events).  `e2e` times fa_bwd_host: pinned host inputs copied in, the backward,
dQ / dK / dV copied out, every step.  `roofline` reports the main kernel's
own event-timed duration against the measured bf16 tensor peak.
`cpu_baseline` times the fp64 oracle on the host cores on a bounded sample.
`--impl reference` times that oracle alone (the slow reference arm).
With N > 1 (torchrun) every rank runs its own replica of the workload
(replicas only: the backward of one problem is not split across GPUs).
"""
from __future__ import annotations

import argparse
import json
import math
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

from flashattention_backward_preprocess_gb300.inputs import BENCH_WORKLOAD, WORKLOADS, make_inputs  # noqa: E402

METRIC = "attn-backward TFLOP/s (causal-adjusted)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.proc = None
        self.gpu_index = gpu_index
        self.window = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        rows = []
        for ts, line in self.samples:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((ts, parts))
        if not rows:
            return None
        inside = [r for r in rows if t0 <= r[0] <= t1] or rows
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for _, p in inside if num(p[1]) is not None]
        smax = [num(p[2]) for _, p in inside if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for _, p in inside for k in range(4) if p[5 + k].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(inside),
                "samples_in_timed_region": sum(1 for r in rows if t0 <= r[0] <= t1)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
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


# Sources each main kernel is built from: ncu traffic counters are only valid for this exact code.
KERNEL_SOURCES = {
    "bwd_sm103_kernel": ("bwd_sm103.cu", "sm103_ptx.cuh", "bounded_wait.cuh", "fa_internal.cuh"),
    "bwd_d256_kernel": ("bwd_d256.cu", "sm103_ptx.cuh", "bounded_wait.cuh", "fa_internal.cuh", "tma_map.cuh"),
    "bwd_simt_kernel": ("bwd_simt.cu", "sm103_ptx.cuh", "fa_internal.cuh"),
}


def kernel_source_hash(kernel: str = "bwd_sm103_kernel") -> str:
    """Hash of a main kernel's sources (see KERNEL_SOURCES)."""
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "flashattention_backward_preprocess_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def main_kernel_traffic(workload: str, deterministic: bool = False, kernel: str = "bwd_sm103_kernel"):
    """DRAM bytes (read + write) per main-kernel launch from the committed ncu summary, or None
    when the kernel's sources changed since the counters were taken.  The counters are those of
    the default (non-deterministic) kernel instance: a deterministic run gets None."""
    if deterministic:
        return None
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:
        return None
    k = d.get("kernels", {}).get(kernel)
    if not k or k.get("sha") != kernel_source_hash(kernel):
        return None
    return k.get("bytes_per_launch", {}).get(workload)


FP32_SMS = 152  # GB300 streaming multiprocessors (each 128 fp32 FMA lanes)


def main_kernel_family(w) -> str:
    """The main backward kernel fa_bwd runs for a workload (the library's dispatch)."""
    if w.dtype == "f32":
        return "bwd_simt_kernel"
    return "bwd_d256_kernel" if w.d == 256 else "bwd_sm103_kernel"


def main_kernel_name(w, det: bool) -> str:
    fam = main_kernel_family(w)
    if fam == "bwd_simt_kernel":
        return f"bwd_simt_kernel<f32,{w.d}>"
    if fam == "bwd_d256_kernel":
        return f"bwd_d256_kernel<{w.dtype}>"
    return f"bwd_sm103_kernel<{w.dtype},{128 if w.d > 64 else 64},{'det' if det else 'default'}>"


def workload_config(w, extra=None):
    cfg = {"workload": w.name, "B": w.B, "H": w.H, "H_kv": w.H_kv, "S_q": w.S_q, "S_k": w.S_k,
           "d": w.d, "causal": w.causal, "window": w.window, "scale": "1/sqrt(d)", "dtype": w.dtype,
           "inputs": f"Q,K,V~N(0,1), dO~N(0,{w.do_std}^2), seed {w.seed}; O, LSE from the library forward"}
    if extra:
        cfg.update(extra)
    return cfg


def cpu_oracle_time(w, Q, K, V, dO, O, LSE, batches: int):
    """fp64 oracle backward on the first `batches` batch entries (all heads, full sequences)."""
    import oracle
    batches = min(batches, w.B)
    args = [x[:batches].detach().to("cpu", torch.float64).numpy() for x in (dO, Q, K, V, O, LSE)]
    t0 = time.perf_counter()
    oracle.ref_bwd(*args, w.scale, w.causal, w.window)
    dt = time.perf_counter() - t0
    flops = w.with_(B=batches).flops()
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"fp64 oracle ref_bwd on batch entries 0..{batches - 1} of {w.B} "
                      f"(all {w.H} heads, S={w.S_q}), {dt:.2f} s wall, {flops:.3g} flops"}


def run_reference(args, world, rank):
    """Reference arm: the fp64 CPU oracle as it stands, on the host cores."""
    if rank != 0:
        return 0
    import oracle
    w = WORKLOADS[args.workload]
    sample_b = 1
    ws = w.with_(B=sample_b)
    if args.ref_seq:  # a shorter sample of the same heads and head dim (quick checks)
        ws = ws.with_(S_q=min(args.ref_seq, w.S_q), S_k=min(args.ref_seq, w.S_k))
    Q, K, V, dO = make_inputs(ws)
    args64 = [x.to(torch.float64).numpy() for x in (Q, K, V, dO)]
    O, LSE = oracle.ref_fwd(args64[0], args64[1], args64[2], w.scale, w.causal, w.window)
    bwd_args = (args64[3], args64[0], args64[1], args64[2], O, LSE)
    for _ in range(args.warmup):
        oracle.ref_bwd(*bwd_args, w.scale, w.causal, w.window)
    times = []
    t_all = time.perf_counter()
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.ref_bwd(*bwd_args, w.scale, w.causal, w.window)
        times.append(time.perf_counter() - t0)
    total = time.perf_counter() - t_all
    ms = 1e3 * statistics.mean(times)
    value = ws.flops() / (ms / 1e3) / 1e12
    sample = (f"each step: fp64 oracle ref_bwd on batch entry 0 of {w.B} (all {w.H} heads, "
              f"S={ws.S_q}, d={w.d}, causal), {ws.flops():.3g} flops")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(w, {"sample_batch_entries": sample_b}),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "timed_region_s": total}
    print(json.dumps(line), flush=True)
    return 0


def run_forward(args, fa, w, Q, K, V, O, LSE, flush, stream, world, rank, device):
    """The forward (O and LSE the backward consumes) on the bench workload: CUDA events per
    call, L2 flushed between calls; 4·B·H·S_q·S_k·d flops, halved for causal (the band's
    pairs with a sliding window)."""
    for _ in range(args.warmup):
        fa.fa_fwd(Q, K, V, scale=w.scale, causal=w.causal, O=O, LSE=LSE, window_size=w.window)
    torch.cuda.synchronize(device)
    fa.fa_check_device()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        fa.fa_fwd(Q, K, V, scale=w.scale, causal=w.causal, O=O, LSE=LSE, window_size=w.window)
        ends[i].record(stream)
    torch.cuda.synchronize(device)
    fa.fa_check_device()
    ms = max_over_ranks(statistics.mean(s.elapsed_time(e) for s, e in zip(starts, ends)), world, device)
    flops = w.fwd_flops()
    peaks, peak_src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    value = world * flops / (ms / 1e3) / 1e12
    if rank == 0:
        print(json.dumps({"metric": "attn-forward TFLOP/s (causal-adjusted)", "value": value, "unit": "TFLOP/s",
                          "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
                          "higher_is_better": True, "dtype": w.dtype, "data": "synthetic",
                          "roofline": {"bound": "tensor", "achieved": value / world, "peak": peak,
                                       "unit": "TFLOP/s", "frac": value / world / peak,
                                       "peak_source": f"{peak_src} bf16_tflops (burst)"},
                          "config": workload_config(w, {"l2": "flushed between calls (256 MiB write)"})}),
              flush=True)


def run_e2e(args, fa, w, dO, Q, K, V, O, LSE, flops, world, device):
    """The same backward through fa_bwd_host: pinned host inputs in, host results out,
    every copy inside the timed region."""
    host_in = [x.detach().cpu().pin_memory() for x in (dO, Q, K, V, O, LSE)]
    host_out = [torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in (Q, K, V)]
    fa.fa_bwd_host(*host_in, scale=w.scale, causal=w.causal, dQ=host_out[0], dK=host_out[1], dV=host_out[2])
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        fa.fa_bwd_host(*host_in, scale=w.scale, causal=w.causal, dQ=host_out[0], dK=host_out[1],
                       dV=host_out[2])
    e2e_s = max_over_ranks((time.perf_counter() - t0) / args.e2e_steps, world, device)
    h2d = sum(x.numel() * x.element_size() for x in host_in)
    d2h = sum(x.numel() * x.element_size() for x in host_out)
    return {"value": world * flops / e2e_s / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3, "steps": args.e2e_steps}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=600)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-batches", type=int, default=2,
                    help="batch entries of the workload the CPU oracle baseline runs")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-seq", type=int, default=0,
                    help="reference arm: limit the sampled sequence length (0 = the workload's)")
    ap.add_argument("--forward", action="store_true",
                    help="time the forward (fa_fwd) on the same workload instead of the backward")
    ap.add_argument("--workload", default=BENCH_WORKLOAD, choices=sorted(WORKLOADS),
                    help="workload to time (default: the headline one)")
    ap.add_argument("--deterministic", action="store_true",
                    help="time the backward with bitwise-reproducible dQ (fa_bwd_ex deterministic = 1)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, world, rank)

    import flashattention_backward_preprocess_gb300 as fa

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    w = WORKLOADS[args.workload]
    Qh, Kh, Vh, dOh = make_inputs(w)
    Q, K, V, dO = (x.to(device) for x in (Qh, Kh, Vh, dOh))
    O, LSE = fa.fa_fwd(Q, K, V, scale=w.scale, causal=w.causal, window_size=w.window)
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    if args.forward:
        return run_forward(args, fa, w, Q, K, V, O, LSE, flush, stream, world, rank, device)

    det = bool(args.deterministic)
    for _ in range(args.warmup):
        fa.fa_bwd(dO, Q, K, V, O, LSE, scale=w.scale, causal=w.causal, dQ=dQ, dK=dK, dV=dV,
                  window_size=w.window, deterministic=det)
    torch.cuda.synchronize(device)
    fa.fa_check_device()

    sampler = ClockSampler(device.index if device.index is not None else 0)
    sampler.start()
    time.sleep(0.3)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(device)
    fa.fa_profile(True)
    t_wall0 = time.time()
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        fa.fa_bwd(dO, Q, K, V, O, LSE, scale=w.scale, causal=w.causal, dQ=dQ, dK=dK, dV=dV,
                  window_size=w.window, deterministic=det)
        ends[i].record(stream)
    torch.cuda.synchronize(device)
    barrier(world)
    t_wall1 = time.time()
    ms_pre, ms_main, ms_fin, calls = fa.fa_profile_read()
    fa.fa_profile(False)
    fa.fa_check_device()
    time.sleep(0.2)
    sampler.stop()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = max_over_ranks(statistics.mean(step_ms), world, device)
    flops = w.flops()
    value = world * flops / (ms / 1e3) / 1e12

    # ---- roofline of the dominant kernel (the main kernel of the workload's path)
    peaks, peak_src = load_peaks()
    main_ms = ms_main / max(calls, 1)
    achieved = flops / (main_ms / 1e3) / 1e12
    kernel = main_kernel_name(w, det)
    if w.dtype == "f32":
        # CUDA-core path: FFMA peak = SMs x 128 fp32 lanes x 2 flops x the maximum SM clock
        sm_mhz = float(peaks.get("sm_max_mhz", 2070.0))
        peak = FP32_SMS * 128 * 2 * sm_mhz * 1e6 / 1e12
        roofline = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak,
                    "traffic": main_kernel_traffic(w.name, det, "bwd_simt_kernel"),
                    "peak_source": f"{FP32_SMS} SMs x 128 fp32 FMA lanes x 2 flops x {sm_mhz:.0f} MHz "
                                   f"({peak_src} sm_max_mhz)",
                    "kernel": kernel, "kernel_ms": main_ms,
                    "preprocess_ms": ms_pre / max(calls, 1), "finalize_ms": ms_fin / max(calls, 1),
                    "step_frac": (flops / (ms / 1e3) / 1e12) / peak}
    else:
        peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
        traffic = main_kernel_traffic(w.name, det, main_kernel_family(w))
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak, "traffic": traffic, "peak_source": f"{peak_src} bf16_tflops (burst)",
                    "kernel": kernel, "kernel_ms": main_ms,
                    "preprocess_ms": ms_pre / max(calls, 1), "finalize_ms": ms_fin / max(calls, 1),
                    "frac_of_sustained": achieved / float(peaks.get("bf16_tflops_sustained", 1700.0)),
                    "step_frac": (flops / (ms / 1e3) / 1e12) / peak}

    # ---- end to end through the host-buffer entry point (no sliding window or
    # deterministic mode there)
    e2e = None
    if w.window == 0 and not det:
        e2e = run_e2e(args, fa, w, dO, Q, K, V, O, LSE, flops, world, device)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_oracle_time(w, Q, K, V, dO, O, LSE, args.cpu_batches)

    clocks = sampler.summary(t_wall0, t_wall1)
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
                "data": "synthetic (seeded normal inputs of the workload's shapes)",
                "config": workload_config(w, {"l2": "flushed between steps (256 MiB write, outside the events)",
                                              "parallelism": "replicas" if world > 1 else "single GPU",
                                              "deterministic_dq": det}),
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": 3 * args.steps, "clocks": clocks,
                "memset_nodes_per_step": 1 if det else 0,
                "pct_of_bf16_peak": 100.0 * (flops / (ms / 1e3) / 1e12) / peak,
                "timed_region_s": t_wall1 - t_wall0}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
