#!/usr/bin/env python3
"""Benchmark of the split-K BF16 decode GEMM on GB300.

Default workload: the single-token decode projection, M=1 token, N=7168
weight rows, K=2048, L=1, split_k=4 (29 MB of bf16 weights, pure weight
streaming).  Metric: achieved HBM TB/s of algorithmic bytes
2*L*(N*K + M*K + M*N) per step; the roofline fraction is reported beside it.

A step is one call of the GEMM on one batch of activations.  Timed steps run
back to back on one stream (captured in CUDA graphs, programmatic dependent
launch between steps, as a decode model chains its projections), each step
reading the next of R weight copies whose total exceeds 4x the L2 cache, so
every step streams its weights from HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload decode_m1|...] [--sweep]

Under torchrun (N > 1) every rank runs an independent replica of the
workload on its own GPU (weak scaling, no data exchange); rank 0 prints the
JSON line with the max-over-ranks time.  `--impl reference` times the CPU
oracle (float64, all host cores) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "achieved HBM TB/s (and % of roofline) vs M for BF16 split-K decode GEMM"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
KERNEL_SOURCES = ["split_bf16_gemm_swapped_gb300/csrc/splitk_kernel.cu",
                  "split_bf16_gemm_swapped_gb300/csrc/splitk_device.cuh",
                  "split_bf16_gemm_swapped_gb300/csrc/splitk_internal.h"]


# ----------------------------------------------------------------- helpers
def workload_by_name(name: str):
    from split_bf16_gemm_swapped_gb300 import workloads as W
    table = {"tiny": W.TINY, "decode_m1": W.DECODE_M1, "decode_m16": W.DECODE_M16,
             "wide_s2": W.WIDE_S2, "wide_s4": W.WIDE_S4}
    if name in table:
        return table[name]
    if name.startswith("sweep_m"):
        m, s = name[len("sweep_m"):].split("_s")
        return W.sweep(int(m), int(s))
    raise SystemExit(f"unknown workload {name}")


def describe(w) -> str:
    return f"{w.name}: M={w.M} N={w.N} K={w.K} L={w.L} split_k={w.split_k}"


def peaks():
    path = ROOT / "MEASURED_PEAKS.json"
    if path.exists():
        try:
            d = json.loads(path.read_text())
            hbm = d.get("hbm_gbs")
            bf16 = d.get("bf16_tflops")
            bf16s = d.get("bf16_tflops_sustained", bf16)
            if hbm:
                return float(hbm), float(bf16 or FALLBACK_BF16_TFLOPS), float(bf16s or FALLBACK_BF16_TFLOPS), "measured"
        except (ValueError, TypeError):
            pass
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def kernel_sha() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        h.update((ROOT / rel).read_bytes())
    return h.hexdigest()[:16]


def committed_traffic(workload_key: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source."""
    path = ROOT / "profiles" / f"splitk_{workload_key}_traffic.txt"
    if not path.exists():
        return None
    kv = {}
    for line in path.read_text().splitlines():
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            kv[k.strip()] = v.strip()
    if kv.get("kernel_sha256") != kernel_sha():
        return None
    try:
        return int(float(kv["traffic_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()
        return False

    def summary(self):
        if not self.out:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def clock_verdict(summary: dict) -> str:
    """Whether a timed region's clock record makes its number acceptable:
    thermal or hardware slowdown, or an SM clock well below its maximum with
    no reason given (a leftover clock lock), rejects it; a power cap is
    noted (normal for a long dense run on this part)."""
    reasons = summary.get("reasons") or []
    bad = [r for r in reasons if r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")]
    if bad:
        return "rejected: " + ", ".join(bad)
    sm, smax = summary.get("sm_mhz"), summary.get("sm_max_mhz")
    if sm is None or smax is None:
        return "unsampled"
    if "sw_power_cap" in reasons:
        return "ok (sw_power_cap noted)"
    if sm < 0.8 * smax:
        return f"rejected: SM clock {sm:.0f} of {smax:.0f} MHz with no reason"
    return "ok"


def with_verdict(summary: dict) -> dict:
    return dict(summary, verdict=clock_verdict(summary))


def max_over_ranks(value: float, device=None) -> float:
    """The largest `value` over all ranks (the job's time is its slowest
    rank's); the value itself when no process group is running."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tbps(world: int, bytes_per_step: int, steps: int, elapsed_ms: float) -> float:
    """Whole-job throughput: every rank moves bytes_per_step per step."""
    return world * bytes_per_step * steps / (elapsed_ms * 1e-3) / 1e12


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def host_cpu_name() -> str:
    """The host processor as /proc/cpuinfo names it (x86: model name; Arm:
    implementer and part numbers), else the platform's machine string."""
    import platform
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                k, _, v = line.partition(":")
                fields.setdefault(k.strip(), v.strip())
    except OSError:
        pass
    if fields.get("model name"):
        return fields["model name"]
    if fields.get("CPU part"):
        return (f"{platform.machine()} implementer {fields.get('CPU implementer', '?')} "
                f"part {fields['CPU part']}")
    return platform.machine() or "unknown"


# ----------------------------------------------------------------- CPU arms
def cpu_oracle_rate(w, budget_s: float, threads: int):
    """Times the oracle on the whole workload (or on a prefix of the weight
    rows when one pass would exceed the budget); returns (TB/s, sample, used)."""
    import oracle
    a = w.make_a()
    b = w.make_b()
    # calibrate on a slice of 128 weight rows
    rows = min(w.N, 128)
    t0 = time.perf_counter()
    oracle.gemm_threaded(np.ascontiguousarray(a[:, :rows]), b, threads)
    per_row = (time.perf_counter() - t0) / rows
    n = w.N if per_row * w.N <= budget_s else max(1, int(budget_s / max(per_row, 1e-9)))
    a_s = np.ascontiguousarray(a[:, :n])
    reps, elapsed, used = 0, 0.0, 1
    while True:
        t0 = time.perf_counter()
        _, used = oracle.gemm_threaded(a_s, b, threads)
        elapsed += time.perf_counter() - t0
        reps += 1
        if elapsed >= budget_s or reps >= 100000:
            break
    sample_bytes = 2 * w.L * (n * w.K + w.M * w.K + w.M * n)
    rate = sample_bytes * reps / elapsed / 1e12
    sample = (f"{'whole workload' if n == w.N else f'first {n} of {w.N} weight rows'} "
              f"x {reps} repetitions, {elapsed:.1f} s")
    return rate, sample, used


def run_cpu_table(args):
    """Extra lines, no GPU: the oracle on the host cores, all of them and one,
    for the tiny, decode and sweep (M = 1, 16, 128) workloads, each a bounded
    sample (a prefix of the weight rows when a pass would exceed the budget)."""
    from split_bf16_gemm_swapped_gb300 import workloads as W
    sweep = {w.M: w for w in W.all_sweep() if w.split_k == 1}
    cases = [W.TINY, W.DECODE_M1, W.DECODE_M16, sweep[1], sweep[16], sweep[128]]
    budget = max(1.0, args.cpu_budget / 4)
    cores = host_cores()
    for w in cases:
        for threads in (cores, 1):
            rate, sample, used = cpu_oracle_rate(w, budget, threads)
            print(json.dumps({"cpu_table": describe(w), "impl": "oracle", "TB/s": rate,
                              "GFLOP/s": rate * 1e3 * w.flops / w.bytes, "cores": used,
                              "cpu": host_cpu_name(), "sample": sample}), flush=True)


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    threads = host_cores()
    a = w.make_a()
    b = w.make_b()
    total_steps = args.steps + args.warmup
    per_step_budget = max(1e-3, min(1.0, 120.0 / max(1, total_steps)))
    rows = min(w.N, 128)
    t0 = time.perf_counter()
    oracle.gemm_threaded(np.ascontiguousarray(a[:, :rows]), b, threads)
    per_row = (time.perf_counter() - t0) / rows
    n = max(1, min(w.N, int(per_step_budget / max(per_row, 1e-9))))
    a_s = np.ascontiguousarray(a[:, :n])
    for _ in range(args.warmup):
        oracle.gemm_threaded(a_s, b, threads)
    used = 1
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _, used = oracle.gemm_threaded(a_s, b, threads)
    elapsed = time.perf_counter() - t0
    sample_bytes = 2 * w.L * (n * w.K + w.M * w.K + w.M * n)
    value = sample_bytes * args.steps / elapsed / 1e12
    sample = f"first {n} of {w.N} weight rows per step" if n < w.N else "whole workload per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": elapsed / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_block(w, None),
        "cpu_baseline": {"value": value, "unit": "TB/s", "cores": used, "kind": "oracle",
                         "sample": sample, "cpu": host_cpu_name()},
        "e2e": {"value": value, "unit": "TB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_block(w, rotation):
    c = {"workload": describe(w), "M": w.M, "N": w.N, "K": w.K, "L": w.L,
         "split_k": w.split_k, "bytes_per_step": w.bytes, "flops_per_step": w.flops}
    if rotation is not None:
        c["l2"] = rotation
    return c


# ----------------------------------------------------------------- GPU arm
def to_dev(bits: np.ndarray, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def run_ours(args, w):
    import torch
    import torch.distributed as dist

    import split_bf16_gemm_swapped_gb300 as sk

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    sk.load_library()

    a_host = w.make_a()
    b_host = w.make_b()
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or 0) or 126 * 1024 * 1024
    a_bytes = a_host.nbytes
    R = args.rotate if args.rotate else max(2, math.ceil(4 * l2 / a_bytes))
    a0 = to_dev(a_host, dev)
    As = [a0] + [a0.clone() for _ in range(R - 1)]
    b = to_dev(b_host, dev)
    c = torch.empty((w.L, w.M, w.N), dtype=torch.bfloat16, device=dev)
    plan = sk.splitk_plan(w.M, w.N, w.K, w.L, w.split_k)
    rotation = (f"rotating {R} weight copies ({R * a_bytes / 1e6:.0f} MB, "
                f"{R * a_bytes / l2:.1f}x the {l2 / 2**20:.0f} MiB L2)")

    stream = torch.cuda.Stream(dev)
    torch.cuda.synchronize(dev)

    def step(i):
        sk.splitk_gemm_bf16(As[i % R], b, c, split_k=w.split_k, stream=stream)

    # warm-up: eager launches (also builds every tensor map before capture)
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, R)):
            step(i)
    stream.synchronize()
    if sk.splitk_get_status() != 0:
        raise SystemExit(f"kernel fault during warm-up: {sk.splitk_get_fault()}")

    # graphs of G steps (and a tail graph) so the host never limits the rate
    G = min(args.steps, R * max(1, 1024 // R))
    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                step(i)
        return g
    g_main = capture(G) if G > 0 else None
    reps, tail = divmod(args.steps, G)
    g_tail = capture(tail) if tail else None
    with torch.cuda.stream(stream):
        g_main.replay()
    stream.synchronize()

    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    # the timed region in 5 consecutive parts (events between graph replays)
    parts = 5 if reps >= 5 else 1
    bounds = [reps * j // parts for j in range(parts + 1)]
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(parts)]
    with ClockSampler(local) as clocks:
        with torch.cuda.stream(stream):
            start.record(stream)
            for j in range(parts):
                for _ in range(bounds[j + 1] - bounds[j]):
                    g_main.replay()
                marks[j].record(stream)
            if g_tail is not None:
                g_tail.replay()
            end.record(stream)
        end.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
    elapsed_ms = max_over_ranks(start.elapsed_time(end), dev)
    if sk.splitk_get_status() != 0:
        raise SystemExit(f"kernel fault in the timed region: {sk.splitk_get_fault()}")

    ms_per_step = elapsed_ms / args.steps
    value = job_tbps(world, w.bytes, args.steps, elapsed_ms)
    hbm, bf16, bf16s, src = peaks()
    achieved_gbs = w.bytes / (ms_per_step * 1e-3) / 1e9
    flops_tfs = w.flops / (ms_per_step * 1e-3) / 1e12
    t_roof = max(w.bytes / (hbm * 1e9), w.flops / (bf16s * 1e12))
    bound = "hbm" if w.bytes / (hbm * 1e9) >= w.flops / (bf16s * 1e12) else "tensor"
    key = args.workload
    roofline = {"bound": bound, "achieved": round(achieved_gbs, 1), "peak": hbm,
                "unit": "GB/s", "frac": round(achieved_gbs / hbm, 4),
                "traffic": committed_traffic(key), "peak_source": src,
                "roofline_time_frac": round(t_roof / (ms_per_step * 1e-3), 4),
                "tflops": round(flops_tfs, 2),
                "note": f"frac of {src} HBM copy bandwidth; launch duration = timed region / steps"}
    if bound == "tensor":
        roofline.update({"achieved": round(flops_tfs, 2), "peak": bf16s, "unit": "TFLOP/s",
                         "frac": round(flops_tfs / bf16s, 4)})

    # isolated single-launch time: one launch per graph replay, so no
    # neighbour overlaps it and host launch overhead is not on the GPU clock
    g_one = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_one, stream=stream):
        step(0)
    iso = []
    with torch.cuda.stream(stream):
        for i in range(20):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g_one.replay()
            e1.record(stream)
            e1.synchronize()
            iso.append(e0.elapsed_time(e1))
    iso_us = statistics.median(iso) * 1e3

    # the parts of the timed region, and a hot-L2 figure (one weight copy
    # that stays in L2; labelled, not the metric)
    part_tbps = []
    prev = start
    for j in range(parts):
        n = (bounds[j + 1] - bounds[j]) * G
        part_tbps.append(round(w.bytes * n / (prev.elapsed_time(marks[j]) * 1e-3) / 1e12, 3))
        prev = marks[j]
    g_hot = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_hot, stream=stream):
        for _ in range(G):
            sk.splitk_gemm_bf16(As[0], b, c, split_k=w.split_k, stream=stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g_hot.replay()
        e0.record(stream)
        for _ in range(5):
            g_hot.replay()
        e1.record(stream)
    e1.synchronize()
    hot_ms = e0.elapsed_time(e1) / (5 * G)
    del g_hot
    if sk.splitk_get_status() != 0:
        raise SystemExit(f"kernel fault in the hot-L2 run: {sk.splitk_get_fault()}")

    # end to end through the C ABI: pinned host activations in, host output out
    e2e = None
    if args.e2e_steps > 0:
        b_pin = torch.from_numpy(b_host.view(np.int16)).view(torch.bfloat16).pin_memory()
        c_pin = torch.empty((w.L, w.M, w.N), dtype=torch.bfloat16).pin_memory()
        n_e2e = min(args.steps, args.e2e_steps)

        def timed_calls(call, graph_steps):
            """ms per call: eager (one host call per step), or captured in a
            CUDA graph of `graph_steps` calls (how a decode loop issues them)."""
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                for i in range(min(args.warmup, 10)):
                    call(i)
                stream.synchronize()
                if graph_steps == 0:
                    e0.record(stream)
                    for i in range(n_e2e):
                        call(i)
                    e1.record(stream)
                    e1.synchronize()
                    return e0.elapsed_time(e1) / n_e2e, n_e2e
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for i in range(graph_steps):
                        call(i)
                g.replay()
                stream.synchronize()
                reps = max(1, n_e2e // graph_steps)
                e0.record(stream)
                for _ in range(reps):
                    g.replay()
                e1.record(stream)
                e1.synchronize()
                return e0.elapsed_time(e1) / (reps * graph_steps), reps * graph_steps

        def copies(i):      # copy engines: b_pin -> b, GEMM, c -> c_pin
            sk.splitk_gemm_bf16_hostio(As[i % R], b_pin, c_pin, b, c, w.split_k, stream)

        def zero_copy(i):   # the kernel reads b_pin and writes c_pin itself
            sk.splitk_gemm_bf16_zerocopy(As[i % R], b_pin, c_pin, w.split_k, stream)

        G = 50
        copy_eager_ms, _ = timed_calls(copies, 0)
        try:
            zero_copy(0)
            zc = True
        except sk.SplitKError:
            zc = False      # shape without thread-loaded activations
        stream.synchronize()
        if zc:
            zc_eager_ms, _ = timed_calls(zero_copy, 0)
            e2e_ms, steps_e2e = timed_calls(zero_copy, G)
        else:
            e2e_ms, steps_e2e = timed_calls(copies, G)
        tbps = lambda ms: world * w.bytes / (ms * 1e-3) / 1e12
        e2e = {"value": tbps(e2e_ms), "unit": "TB/s",
               "h2d_bytes_per_step": int(b_host.nbytes), "d2h_bytes_per_step": int(w.L * w.M * w.N * 2),
               "steps": steps_e2e, "ms_per_step": e2e_ms,
               "path": "splitk_gemm_bf16_zerocopy" if zc else "splitk_gemm_bf16_hostio",
               "copy_engine_eager_ms_per_step": copy_eager_ms,
               "zero_copy_eager_ms_per_step": zc_eager_ms if zc else None,
               "note": ("weights resident in HBM; every step the activations cross from pinned host memory "
                        "and the output back to pinned host memory; value: "
                        + ("the kernel loads and stores them itself (splitk_gemm_bf16_zerocopy), "
                           if zc else "copy engines around the kernel (splitk_gemm_bf16_hostio), ")
                        + f"calls captured in a CUDA graph of {G} steps; *_eager_*: one host call per step, "
                        "copy_engine: splitk_gemm_bf16_hostio")}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        rate, sample, used = cpu_oracle_rate(w, args.cpu_budget, host_cores())
        cpu = {"value": rate, "unit": "TB/s", "cores": used, "kind": "oracle", "sample": sample,
               "cpu": host_cpu_name()}
        one, one_sample, _ = cpu_oracle_rate(w, max(1.0, args.cpu_budget / 4), 1)
        cpu["single_core"] = {"value": one, "unit": "TB/s", "sample": one_sample}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": config_block(w, rotation) | {
                "plan": {k: v for k, v in plan.as_dict().items()
                         if k in ("mma_n", "stages", "split_k", "grid", "smem_bytes",
                                  "mailbox_dedicated", "reduce_rounds", "reduce_scatter",
                                  "b_resident", "a_tmem_tiles", "mma_issuers", "pdl_trigger")},
                "launch": "CUDA graphs of back-to-back launches with programmatic dependent launch",
                "isolated_launch_us": round(iso_us, 2),
                "isolated_note": "one launch per graph replay, events around the replay"},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": args.steps, "clocks": with_verdict(clocks.summary()),
            "parts": {"tbps": part_tbps, "median": statistics.median(part_tbps),
                      "note": f"the timed region in {parts} consecutive parts; value covers all of it"},
            "hot_l2": {"value": round(w.bytes / (hot_ms * 1e-3) / 1e12, 3), "unit": "TB/s",
                       "ms_per_step": hot_ms,
                       "note": "one weight copy, L2-resident after the first pass; not the metric"},
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_sweep_w4(args):
    """Extra lines for the A16W4 variant (4-bit E2M1 weights with E8M0 scales
    per 32 k, bf16 activations) on the decode shapes: HBM TB/s of the bytes
    it moves (codes, scales, activations, output) and the step time next to
    the bf16 kernel's on the same shape."""
    import torch

    import split_bf16_gemm_swapped_gb300 as sk
    from split_bf16_gemm_swapped_gb300 import synthetic
    from split_bf16_gemm_swapped_gb300 import workloads as W
    dev = torch.device("cuda:0")
    hbm, bf16, bf16s, src = peaks()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size

    def timed(launch, R):
        s = torch.cuda.Stream(dev)
        with torch.cuda.stream(s):
            for i in range(R + 3):
                launch(i % R, s)
        s.synchronize()
        n = max(R, 240 // R * R)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for i in range(n):
                launch(i % R, s)
        with torch.cuda.stream(s):
            g.replay()
        s.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 10
        with torch.cuda.stream(s):
            e0.record(s)
            for _ in range(reps):
                g.replay()
            e1.record(s)
        e1.synchronize()
        return e0.elapsed_time(e1) / (reps * n) * 1e-3

    for w in (W.DECODE_M1, W.DECODE_M16, W.TINY, W.DECODE_M1.with_(M=8), W.DECODE_M1.with_(M=32),
              W.DECODE_M1.with_(L=8), W.DECODE_M16.with_(L=4)):
        aq, a_s = synthetic.w4_weights(w.L, w.N, w.K, w.seed)
        q0 = torch.from_numpy(aq).to(dev)
        s0 = torch.from_numpy(a_s).to(dev)
        w4_bytes = w.L * (w.N * w.K // 2 + w.N * w.K // 32 + 2 * w.M * w.K + 2 * w.M * w.N)
        R = max(2, min(64, math.ceil(4 * l2 / (aq.nbytes + a_s.nbytes))))
        Qs = [q0] + [q0.clone() for _ in range(R - 1)]
        Ss = [s0] + [s0.clone() for _ in range(R - 1)]
        b = to_dev(w.make_b(), dev)
        c = torch.empty((w.L, w.M, w.N), dtype=torch.bfloat16, device=dev)
        t4 = timed(lambda i, st: sk.splitk_gemm_w4a16(Qs[i], Ss[i], b, c, split_k=w.split_k, stream=st), R)
        a0 = to_dev(w.make_a(), dev)
        Rb = max(2, min(20, math.ceil(4 * l2 / (a0.numel() * 2))))
        As = [a0] + [a0.clone() for _ in range(Rb - 1)]
        tb = timed(lambda i, st: sk.splitk_gemm_bf16(As[i], b, c, split_k=w.split_k, stream=st), Rb)
        p = sk.splitk_plan_w4a16(w.M, w.N, w.K, w.L, w.split_k)
        print(json.dumps({"sweep": "A16W4 " + describe(w), "us": round(t4 * 1e6, 2),
                          "TB/s": round(w4_bytes / t4 / 1e12, 3), "bytes_per_call": w4_bytes,
                          "hbm_frac": round(w4_bytes / t4 / 1e9 / hbm, 3), "peak_source": src,
                          "bf16_us": round(tb * 1e6, 2), "speedup_vs_bf16": round(tb / t4, 2),
                          "plan": {k: v for k, v in p.as_dict().items()
                                   if k in ("mma_n", "split_k", "stages", "a_tmem_tiles", "smem_bytes",
                                            "ctas_per_sm", "reduce_scatter", "b_loader")}}), flush=True)
        del Qs, Ss, As, b, c
        torch.cuda.empty_cache()
    if sk.splitk_get_status() != 0:
        raise SystemExit(f"kernel fault during the sweep: {sk.splitk_get_fault()}")


def run_sweep(args):
    """Extra lines, one per workload (not the contract line): TB/s, TFLOP/s and
    roofline fraction vs M and split."""
    import torch

    import split_bf16_gemm_swapped_gb300 as sk
    from split_bf16_gemm_swapped_gb300 import workloads as W
    dev = torch.device("cuda:0")
    hbm, bf16, bf16s, src = peaks()
    ws = list(W.ALL_FIXED) + W.all_sweep() if args.sweep == "all" else W.all_sweep()
    cache = {}
    for w in ws:
        key = (w.N, w.K, w.L, w.seed)
        if key not in cache:
            cache.clear()
            cache[key] = to_dev(w.make_a(), dev)
        a0 = cache[key]
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        R = max(2, math.ceil(3 * l2 / a0.numel() / 2))
        As = [a0] + [a0.clone() for _ in range(R - 1)] if R * a0.numel() * 2 < 8e9 else [a0]
        R = len(As)
        b = to_dev(w.make_b(), dev)
        c = torch.empty((w.L, w.M, w.N), dtype=torch.bfloat16, device=dev)
        s = torch.cuda.Stream(dev)
        with torch.cuda.stream(s):
            for i in range(R + 3):
                sk.splitk_gemm_bf16(As[i % R], b, c, split_k=w.split_k, stream=s)
        s.synchronize()
        n = max(R, 64 // R * R)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for i in range(n):
                sk.splitk_gemm_bf16(As[i % R], b, c, split_k=w.split_k, stream=s)
        with torch.cuda.stream(s):
            g.replay()
        s.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 5
        with torch.cuda.stream(s):
            e0.record(s)
            for _ in range(reps):
                g.replay()
            e1.record(s)
        e1.synchronize()
        t = e0.elapsed_time(e1) / (reps * n) * 1e-3
        tb = w.bytes / t / 1e12
        tf = w.flops / t / 1e12
        t_roof = max(w.bytes / (hbm * 1e9), w.flops / (bf16s * 1e12))
        p = sk.splitk_plan(w.M, w.N, w.K, w.L, w.split_k)
        print(json.dumps({"sweep": describe(w), "us": round(t * 1e6, 2), "TB/s": round(tb, 3),
                          "TFLOP/s": round(tf, 1), "roofline_frac": round(t_roof / t, 3),
                          "hbm_frac": round(tb * 1e3 / hbm, 3), "peak_source": src,
                          "plan": {k: v for k, v in p.as_dict().items()
                                   if k in ("mma_n", "stages", "grid", "smem_bytes",
                                            "mailbox_dedicated", "reduce_rounds", "ctas_per_sm",
                                            "reduce_scatter", "b_resident", "a_tmem_tiles",
                                            "mma_issuers", "pdl_trigger")}}),
              flush=True)
        del As, b, c, g
        torch.cuda.empty_cache()
    if sk.splitk_get_status() != 0:
        raise SystemExit(f"kernel fault during the sweep: {sk.splitk_get_fault()}")


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1,
                    help="GPUs (one rank each under torch.distributed.run; each runs a replica)")
    ap.add_argument("--steps", type=int, default=200000, help="timed steps (one GEMM call each)")
    ap.add_argument("--warmup", type=int, default=100, help="untimed steps first (at least 3)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours",
                    help="reference: the float64 CPU oracle on the host cores")
    ap.add_argument("--workload", default="decode_m1",
                    help="decode_m1 (the default line), decode_m16, tiny, wide_s2, wide_s4, sweep_m<M>_s<split>")
    ap.add_argument("--sweep", choices=["sweep", "all", "w4a16"], default=None,
                    help="extra lines: the M x split sweep, that plus the fixed workloads, or A16W4")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the timed oracle leg")
    ap.add_argument("--rotate", type=int, default=0,
                    help="weight copies to rotate (default: enough for 4x the L2 cache)")
    ap.add_argument("--e2e-steps", type=int, default=2000,
                    help="steps of the end-to-end host-I/O measurement (0 skips it)")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of host time for the CPU oracle baseline")
    ap.add_argument("--cpu-table", action="store_true",
                    help="time the oracle alone (all host cores and one) on the fixed and sweep workloads")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.steps < 1:
        raise SystemExit("--steps must be >= 1")
    w = workload_by_name(args.workload)
    if args.cpu_table:
        run_cpu_table(args)
    elif args.impl == "reference":
        run_reference(args, w)
    elif args.sweep == "w4a16":
        run_sweep_w4(args)
    elif args.sweep:
        run_sweep(args)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
