#!/usr/bin/env python3
"""Benchmark of the split-K BF16 decode GEMM on GB300.

Default workload: the M x split sweep, M in {1, 2, 4, 8, 16, 32, 64, 128}
tokens x split_k in {1, 2, 4, 8}, N=7168 weight rows, K=16384, L=2
independent weight sets (470 MB of bf16 weights per call).  Metric: achieved
HBM TB/s of algorithmic bytes 2*L*(N*K + M*K + M*N) per call, with the
roofline fraction beside it, at every point.  The line's `value` is the
lowest TB/s over the points with M <= 16 (the decode shapes that the 75 %
HBM target covers); every point is listed under `per_point`, and the two
fixed decode workloads (M=1, N=7168, K=2048, split 4; M=16, N=4096, K=7168,
split 8) under `decode`.

A step is one call of the GEMM on one batch of activations.  For each point,
`--steps` calls run back to back on one stream (captured in a CUDA graph,
programmatic dependent launch between calls, as a decode model chains its
projections), each reading the next of R weight copies whose total exceeds
4x the L2 cache, so every call streams its weights from HBM.  The graph is
replayed back to back at least 5 times and for at least `--min-ms` per
point, each replay bracketed by CUDA events; the point's time is the median
replay / steps.  The two decode workloads run graphs of at least 200 calls
(a decode step chains hundreds of such projections), with the `--steps`-long
graph's figure beside it when that is shorter (`short_graph`).  All points
are captured first and timed in one block, so the clock sampler sees the GPU
under load.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload sweep|decode_m1|...] [--sweep fixed|w4a16|w8a16|persistent]

Under torchrun (N > 1) every rank runs an independent replica of the
workload on its own GPU (weak scaling, no data exchange); rank 0 prints the
JSON line with the max-over-ranks time of each point.  `--impl reference`
times the CPU oracle (float64, all host cores) on bounded samples of the
same workload.
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
                  "split_bf16_gemm_swapped_gb300/csrc/splitk_persistent.cu",
                  "split_bf16_gemm_swapped_gb300/csrc/splitk_kernel_common.cuh",
                  "split_bf16_gemm_swapped_gb300/csrc/splitk_device.cuh",
                  "split_bf16_gemm_swapped_gb300/csrc/splitk_internal.h"]
TRAFFIC_TABLE = ROOT / "profiles" / "splitk_dram_traffic.txt"
SWEEP_DESC = ("sweep: M in {1,2,4,8,16,32,64,128} x split_k in {1,2,4,8}, N=7168, K=16384, L=2 "
              "independent weight sets")
EXTRA_MIN_STEPS = 200   # calls per graph of the decode workloads, at least
VALUE_RULE = "lowest TB/s over the points with M <= 16 (the decode shapes the 75 % HBM target covers)"


# ----------------------------------------------------------------- helpers
def workload_key(w) -> str:
    """The name bench.py and the traffic table use for a workload."""
    from split_bf16_gemm_swapped_gb300 import workloads as W
    fixed = {W.TINY: "tiny", W.DECODE_M1: "decode_m1", W.DECODE_M16: "decode_m16",
             W.WIDE_S2: "wide_s2", W.WIDE_S4: "wide_s4"}
    if w in fixed:
        return fixed[w]
    if w.name == "sweep":
        return f"sweep_m{w.M}_s{w.split_k}"
    return f"shape_m{w.M}_n{w.N}_k{w.K}_l{w.L}_s{w.split_k}"


def workload_by_name(name: str):
    from split_bf16_gemm_swapped_gb300 import workloads as W
    table = {"tiny": W.TINY, "decode_m1": W.DECODE_M1, "decode_m16": W.DECODE_M16,
             "wide_s2": W.WIDE_S2, "wide_s4": W.WIDE_S4}
    if name in table:
        return table[name]
    if name.startswith("sweep_m"):
        m, s = name[len("sweep_m"):].split("_s")
        return W.sweep(int(m), int(s))
    if name.startswith("shape_"):
        # shape_m<M>_n<N>_k<K>_l<L>_s<split>: decode-like inputs (seed 1) of any shape
        f = dict((part[0], int(part[1:])) for part in name[len("shape_"):].split("_"))
        return W.DECODE_M1.with_(name="shape", M=f["m"], N=f["n"], K=f["k"], L=f["l"], split_k=f["s"])
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


def traffic_table() -> dict:
    """DRAM bytes per launch by workload key, from the committed ncu table,
    if it was taken on the current kernel sources (else empty)."""
    if not TRAFFIC_TABLE.exists():
        return {}
    sha, rows = None, {}
    for line in TRAFFIC_TABLE.read_text().splitlines():
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        k, _, v = line.partition(":")
        k, v = k.strip(), v.strip()
        if k == "kernel_sha256":
            sha = v
        elif k.startswith("traffic "):
            try:
                rows[k[len("traffic "):]] = int(float(v.split()[0]))
            except (ValueError, IndexError):
                pass
    return rows if sha == kernel_sha() else {}


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


def repeats_for(one_replay_ms: float, min_ms: float, at_least: int = 5, at_most: int = 100000) -> int:
    """Back-to-back replays of a graph to time: at least `at_least`, and
    enough to cover `min_ms` of GPU time."""
    if one_replay_ms <= 0:
        return at_least
    return int(min(at_most, max(at_least, math.ceil(min_ms / one_replay_ms))))


def headline(points: list) -> dict:
    """The point the line's value is quoted on: the lowest TB/s among the
    points with M <= 16 (all points when none has)."""
    small = [p for p in points if p["M"] <= 16] or points
    return min(small, key=lambda p: p["tbps"])


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


def sweep_config(ws):
    return {"workload": SWEEP_DESC, "M": sorted({w.M for w in ws}), "N": ws[0].N, "K": ws[0].K,
            "L": ws[0].L, "split_k": sorted({w.split_k for w in ws}), "value_rule": VALUE_RULE}


def single_config(w):
    return {"workload": describe(w), "M": w.M, "N": w.N, "K": w.K, "L": w.L,
            "split_k": w.split_k, "bytes_per_step": w.bytes, "flops_per_step": w.flops}


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


def run_reference(args):
    """The reference arm: the float64 CPU oracle on the host cores, on the
    same workload and metric.  Each step is a bounded sample (a prefix of the
    weight rows) of every timed point; the oracle has no split, so the sweep
    is timed once per M (M <= 16, the points the value is quoted on)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    from split_bf16_gemm_swapped_gb300 import workloads as W
    threads = host_cores()
    if args.workload == "sweep":
        ws = [W.sweep(m, 1) for m in W.SWEEP_M if m <= 16]
        config = sweep_config(W.all_sweep())
    else:
        ws = [workload_by_name(args.workload)]
        config = single_config(ws[0])
    total_steps = args.steps + args.warmup
    per_step_budget = max(1e-3, min(1.0, 60.0 / max(1, total_steps * len(ws))))
    points, used, a_cache = [], 1, {}
    for w in ws:
        key = (w.N, w.K, w.L, w.seed)
        if key not in a_cache:
            a_cache.clear()
            a_cache[key] = w.make_a()
        a = a_cache[key]
        b = w.make_b()
        rows = min(w.N, 128)
        t0 = time.perf_counter()
        oracle.gemm_threaded(np.ascontiguousarray(a[:, :rows]), b, threads)
        per_row = (time.perf_counter() - t0) / rows
        n = max(1, min(w.N, int(per_step_budget / max(per_row, 1e-9))))
        a_s = np.ascontiguousarray(a[:, :n])
        for _ in range(args.warmup):
            oracle.gemm_threaded(a_s, b, threads)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            _, used = oracle.gemm_threaded(a_s, b, threads)
        elapsed = time.perf_counter() - t0
        sample_bytes = 2 * w.L * (n * w.K + w.M * w.K + w.M * n)
        points.append({"M": w.M, "tbps": sample_bytes * args.steps / elapsed / 1e12,
                       "ms_per_step": elapsed / args.steps * 1e3,
                       "sample": f"first {n} of {w.N} weight rows per step" if n < w.N else "whole workload per step"})
    top = headline(points)
    value = top["tbps"]
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": top["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config | {"value_point": f"M={top['M']}"},
        "per_point": points,
        "cpu_baseline": {"value": value, "unit": "TB/s", "cores": used, "kind": "oracle",
                         "sample": top["sample"], "cpu": host_cpu_name()},
        "e2e": {"value": value, "unit": "TB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- GPU arm
def to_dev(bits: np.ndarray, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


class Point:
    """One workload prepared for timing: its weight copies, activations,
    output and the CUDA graph of `steps` back-to-back calls."""

    def __init__(self, w, weights, dev, stream, steps, warmup):
        import torch
        import split_bf16_gemm_swapped_gb300 as sk
        self.w = w
        self.As = weights
        self.R = len(weights)
        self.b = to_dev(w.make_b(), dev)
        self.c = torch.empty((w.L, w.M, w.N), dtype=torch.bfloat16, device=dev)
        self.stream = stream
        self.steps = steps
        self.plan = sk.splitk_plan(w.M, w.N, w.K, w.L, w.split_k)
        with torch.cuda.stream(stream):
            for i in range(max(warmup, self.R)):        # also builds every tensor map
                self.step(i)
        stream.synchronize()
        if sk.splitk_get_status() != 0:
            raise SystemExit(f"kernel fault during warm-up of {describe(w)}: {sk.splitk_get_fault()}")
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=stream):
            for i in range(steps):
                self.step(i)
        # one untimed replay: settles the graph and estimates a replay's time
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            self.graph.replay()
            e0.record(stream)
            self.graph.replay()
            e1.record(stream)
        e1.synchronize()
        self.replay_ms_estimate = e0.elapsed_time(e1)

    def step(self, i):
        import split_bf16_gemm_swapped_gb300 as sk
        sk.splitk_gemm_bf16(self.As[i % self.R], self.b, self.c, split_k=self.w.split_k, stream=self.stream)


def time_replays(graph, stream, reps):
    """Per-replay ms of `reps` back-to-back replays, each between two events."""
    import torch
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for j in range(reps):
            graph.replay()
            ev[j + 1].record(stream)
    ev[-1].synchronize()
    return [ev[j].elapsed_time(ev[j + 1]) for j in range(reps)]


def point_record(w, ms_per_step, reps, steps, plan, traffic, world):
    hbm, bf16, bf16s, src = peaks()
    t = ms_per_step * 1e-3
    tb = world * w.bytes / t / 1e12
    t_roof = max(w.bytes / (hbm * 1e9), w.flops / (bf16s * 1e12))
    return {"M": w.M, "split_k": w.split_k, "N": w.N, "K": w.K, "L": w.L, "key": workload_key(w),
            "us": round(ms_per_step * 1e3, 3), "tbps": tb, "tflops": round(world * w.flops / t / 1e12, 2),
            "hbm_frac": round(w.bytes / t / 1e9 / hbm, 4), "roofline_frac": round(t_roof / t, 4),
            "steps": steps, "repeats": reps, "launches": reps * steps,
            "traffic": traffic.get(workload_key(w)),
            "plan": {k: v for k, v in plan.as_dict().items()
                     if k in ("mma_n", "stages", "grid", "smem_bytes", "ctas_per_sm", "mailbox_dedicated",
                              "reduce_rounds", "reduce_scatter", "b_resident", "a_tmem_tiles",
                              "mma_issuers", "b_loader", "pdl_trigger", "persistent", "b_stages")}}


def e2e_point(w, weights, dev, stream, steps, reps, warmup, world):
    """The faster of the end-to-end entry points that apply to the workload's
    plan (e2e_path), with the other's TB/s beside it."""
    import split_bf16_gemm_swapped_gb300 as sk
    plan = sk.splitk_plan(w.M, w.N, w.K, w.L, w.split_k)
    paths = ["hostio"] + (["zerocopy"] if plan.b_resident else [])
    runs = [e2e_path(w, weights, dev, stream, steps, reps, warmup, world, p) for p in paths]
    best = max(runs, key=lambda r: r["value"])
    if len(runs) > 1:
        best["other_paths"] = {r["path"]: round(r["value"], 4) for r in runs if r is not best}
    return best


def e2e_path(w, weights, dev, stream, steps, reps, warmup, world, path):
    """The same metric end to end through the C ABI: every step copies its
    activations in from pinned host memory and its output back to pinned host
    memory -- through splitk_gemm_bf16_hostio (for pinned buffers, copy
    kernels chained to the GEMM by programmatic dependent launch), or the
    kernel itself through the buffers' device mappings
    (splitk_gemm_bf16_zerocopy, plans that load activations with their
    threads).  One stream, calls in order.  Timed like the device-resident value: a graph of `steps` calls
    replayed `reps` times back to back, median replay / steps."""
    import torch
    import split_bf16_gemm_swapped_gb300 as sk
    R = len(weights)
    b_host = w.make_b()
    b_pin = torch.from_numpy(b_host.view(np.int16)).view(torch.bfloat16).pin_memory()
    c_pin = torch.empty((w.L, w.M, w.N), dtype=torch.bfloat16).pin_memory()
    b_dev = torch.empty((w.L, w.M, w.K), dtype=torch.bfloat16, device=dev)
    c_dev = torch.empty((w.L, w.M, w.N), dtype=torch.bfloat16, device=dev)
    zc = path == "zerocopy"

    def call(i):
        if zc:
            sk.splitk_gemm_bf16_zerocopy(weights[i % R], b_pin, c_pin, w.split_k, stream)
        else:
            sk.splitk_gemm_bf16_hostio(weights[i % R], b_pin, c_pin, b_dev, c_dev, w.split_k, stream)

    with torch.cuda.stream(stream):
        for i in range(max(warmup, R)):
            call(i)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(steps):
            call(i)
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    ms = statistics.median(time_replays(g, stream, reps)) / steps
    if sk.splitk_get_status() != 0:
        raise SystemExit(f"kernel fault in the end-to-end run: {sk.splitk_get_fault()}")
    # the last step's output reached the host with the device path's bits
    ref = sk.splitk_gemm_bf16(weights[(steps - 1) % R], b_dev.copy_(b_pin), split_k=w.split_k)
    torch.cuda.synchronize(dev)
    if not torch.equal(c_pin.view(torch.int16), ref.view(torch.int16).cpu()):
        raise SystemExit("the end-to-end output differs from the device-resident call")
    ms = max_over_ranks(ms, dev)
    del g
    return {"value": world * w.bytes / (ms * 1e-3) / 1e12, "unit": "TB/s",
            "h2d_bytes_per_step": int(b_host.nbytes), "d2h_bytes_per_step": int(w.L * w.M * w.N * 2),
            "ms_per_step": ms, "steps": steps, "repeats": reps, "workload": describe(w),
            "path": "splitk_gemm_bf16_zerocopy" if zc else "splitk_gemm_bf16_hostio",
            "note": ("weights resident in HBM; every step the activations cross from pinned host memory and "
                     "the output back to pinned host memory, inside the timed region; "
                     + ("the kernel loads and stores them itself through their device mappings"
                        if zc else "copy kernels through the buffers' device mappings, chained to the GEMM "
                                   "by programmatic dependent launch")
                     + f"; one stream; graph of {steps} calls replayed {reps} times, median replay / steps")}


def weight_copies(w, dev, l2, rotate, cache):
    """R device copies of the workload's weights (R * bytes >= 4x L2 unless
    `rotate` fixes R), shared by the workloads with the same weights."""
    key = (w.N, w.K, w.L, w.seed)
    a_bytes = 2 * w.L * w.N * w.K
    R = rotate if rotate else max(2, math.ceil(4 * l2 / a_bytes))
    if key not in cache:
        a0 = to_dev(w.make_a(), dev)
        cache[key] = [a0]
    copies = cache[key]
    while len(copies) < R:
        copies.append(copies[0].clone())
    return copies[:R], (f"rotating {R} weight copies ({R * a_bytes / 1e6:.0f} MB, "
                        f"{R * a_bytes / l2:.1f}x the {l2 / 2**20:.0f} MiB L2)")


def kernel_name(plan: dict) -> str:
    """The kernel a bf16 plan launches, as the profiler names it."""
    if plan.get("persistent"):
        one_ring = plan.get("b_stages", 0) in (0, plan["stages"])
        return f"splitk_persistent_kernel<{plan['mma_n']}, {1 if one_ring else 0}>"
    return f"splitk_gemm_bf16_kernel<{plan['mma_n']}, 0, 1>"


def hot_l2_ms(pt, stream, reps) -> float:
    """Milliseconds per call of the point's plan over one weight copy (a
    graph of the point's step count, every call on the same weights)."""
    import torch

    import split_bf16_gemm_swapped_gb300 as sk
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(pt.steps):
            sk.splitk_gemm_bf16_planned(pt.As[0], pt.b, pt.c, pt.plan, 0, stream)
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    ms = statistics.median(time_replays(g, stream, reps)) / pt.steps
    del g
    return ms


def run_ours(args):
    import torch
    import torch.distributed as dist

    import split_bf16_gemm_swapped_gb300 as sk
    from split_bf16_gemm_swapped_gb300 import workloads as W

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    sk.load_library()
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or 0) or 126 * 1024 * 1024
    stream = torch.cuda.Stream(dev)
    traffic = traffic_table()

    sweep_mode = args.workload == "sweep"
    main_ws = W.all_sweep() if sweep_mode else [workload_by_name(args.workload)]
    extra_ws = [W.DECODE_M1, W.DECODE_M16] if sweep_mode and not args.no_extras else []

    # prepare every point (weights, activations, graph) before timing any.
    # The decode workloads run graphs of at least EXTRA_MIN_STEPS calls (a
    # decode step runs hundreds of such GEMMs back to back; the sweep's own
    # protocol is `--steps` exactly), and, when --steps is shorter, a graph of
    # --steps calls as well, reported beside it.
    cache, rotations, prepared = {}, {}, []
    extra_steps = max(args.steps, EXTRA_MIN_STEPS)
    short_extra = extra_steps != args.steps
    for w in main_ws + extra_ws + (extra_ws if short_extra else []):
        copies, rot = weight_copies(w, dev, l2, args.rotate, cache)
        rotations[workload_key(w)] = rot
        is_extra = w in extra_ws and len(prepared) < len(main_ws) + len(extra_ws)
        prepared.append(Point(w, copies, dev, stream, extra_steps if is_extra else args.steps, args.warmup))
    torch.cuda.synchronize(dev)

    # time every point in one block: barrier + synchronize on both sides of
    # each point's replays, median replay / steps, max over ranks
    results = []
    launches = 0
    with ClockSampler(local) as clocks:
        for pt in prepared:
            reps = repeats_for(pt.replay_ms_estimate, args.min_ms)
            if world > 1:
                dist.barrier()
            torch.cuda.synchronize(dev)
            per_rep = time_replays(pt.graph, stream, reps)
            torch.cuda.synchronize(dev)
            if world > 1:
                dist.barrier()
            ms = max_over_ranks(statistics.median(per_rep) / pt.steps, dev)
            launches += reps * pt.steps
            results.append((pt, ms, reps))
    if sk.splitk_get_status() != 0:
        raise SystemExit(f"kernel fault in the timed region: {sk.splitk_get_fault()}")

    records = [point_record(pt.w, ms, reps, pt.steps, pt.plan, traffic, world) for pt, ms, reps in results]
    main_recs = records[:len(main_ws)]
    extra_recs = records[len(main_ws):len(main_ws) + len(extra_ws)]
    for rec, short in zip(extra_recs, records[len(main_ws) + len(extra_ws):]):
        rec["short_graph"] = {"steps": args.steps, "us": short["us"], "tbps": short["tbps"],
                              "hbm_frac": short["hbm_frac"], "repeats": short["repeats"]}
    # the decode workloads' single-launch time (one call per graph replay):
    # what the first call of every timed graph costs, with no predecessor to
    # overlap its start with
    for rec, (pt, _, _) in zip(extra_recs, results[len(main_ws):len(main_ws) + len(extra_ws)]):
        g1 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g1, stream=stream):
            pt.step(0)
        with torch.cuda.stream(stream):
            g1.replay()
        stream.synchronize()
        rec["isolated_launch_us"] = round(statistics.median(time_replays(g1, stream, 50)) * 1e3, 2)
        del g1
    # the decode workloads with one weight copy, L2-resident after the first
    # call (labelled, not the metric: the weights of these two fit in L2)
    for rec, (pt, _, reps) in zip(extra_recs, results[len(main_ws):len(main_ws) + len(extra_ws)]):
        hot_ms = hot_l2_ms(pt, stream, reps)
        rec["hot_l2"] = {"us": round(hot_ms * 1e3, 3), "tbps": pt.w.bytes / (hot_ms * 1e-3) / 1e12,
                         "note": "one weight copy, L2-resident after the first call; not the metric"}
    top = headline(main_recs)
    top_i = main_recs.index(top)
    top_pt, top_ms, top_reps = results[top_i]
    w = top_pt.w

    hbm, bf16, bf16s, src = peaks()
    achieved_gbs = w.bytes / (top_ms * 1e-3) / 1e9
    t_roof = max(w.bytes / (hbm * 1e9), w.flops / (bf16s * 1e12))
    roofline = {"bound": "hbm", "achieved": round(achieved_gbs, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved_gbs / hbm, 4), "traffic": top["traffic"], "peak_source": src,
                "kernel": kernel_name(top["plan"]),
                "roofline_time_frac": round(t_roof / (top_ms * 1e-3), 4), "tflops": top["tflops"],
                "note": (f"frac of {src} HBM copy bandwidth ({hbm:.0f} GB/s) at the value's point; launch "
                         "duration = median graph replay / steps, CUDA events on the launching stream")}

    # end to end on the value's point (and on the decode workloads)
    e2e = None
    e2e_decode = {}
    if args.e2e:
        for pt, ms, reps in [results[top_i]] + results[len(main_ws):len(main_ws) + len(extra_ws)]:
            rec = e2e_point(pt.w, pt.As, dev, stream, pt.steps, reps, args.warmup, world)
            if pt is top_pt:
                e2e = rec
            else:
                e2e_decode[workload_key(pt.w)] = rec

    # the hot-L2 figure of the single-workload mode: one weight copy that
    # stays in L2 (labelled, not the metric)
    hot = None
    if not sweep_mode:
        hot_ms = hot_l2_ms(top_pt, stream, top_reps)
        hot = {"value": round(w.bytes / (hot_ms * 1e-3) / 1e12, 3), "unit": "TB/s", "ms_per_step": hot_ms,
               "note": "one weight copy, L2-resident after the first pass; not the metric"}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        rate, sample, used = cpu_oracle_rate(w, args.cpu_budget, host_cores())
        cpu = {"value": rate, "unit": "TB/s", "cores": used, "kind": "oracle",
               "sample": f"{describe(w)}: {sample}", "cpu": host_cpu_name()}
        one, one_sample, _ = cpu_oracle_rate(w, max(1.0, args.cpu_budget / 4), 1)
        cpu["single_core"] = {"value": one, "unit": "TB/s", "sample": one_sample}

    if rank == 0:
        if sweep_mode:
            config = sweep_config(main_ws) | {
                "value_point": f"M={w.M} split_k={w.split_k}", "bytes_per_step": w.bytes,
                "flops_per_step": w.flops, "l2": rotations[workload_key(w)]}
        else:
            config = single_config(w) | {"l2": rotations[workload_key(w)], "plan": top["plan"]}
        config["launch"] = ("CUDA graph of --steps back-to-back calls with programmatic dependent launch, "
                            f"replayed back to back at least 5 times and for at least {args.min_ms:g} ms "
                            "per point; the median replay / steps is the point's time")
        line = {
            "metric": METRIC, "value": top["tbps"], "unit": "TB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": top_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic", "config": config,
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches, "clocks": with_verdict(clocks.summary()),
            "per_point": main_recs,
        }
        if extra_recs:
            line["decode"] = {r["key"]: r | ({"e2e": e2e_decode[r["key"]]} if r["key"] in e2e_decode else {})
                              for r in extra_recs}
        if hot is not None:
            line["hot_l2"] = hot
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_profile_case(args):
    """A short eager run for ncu: for one workload (or, with `all`, every
    fixed and sweep workload in turn), one weight copy (so ncu's memory save
    and restore stays small), `--warmup` launches, then `--steps` launches;
    no graphs, no CPU oracle.  `--w4` (`--w8`) runs the A16W4 (A16W8)
    kernel on the same shapes: 4-bit (8-bit) codes with their scales."""
    import torch

    import split_bf16_gemm_swapped_gb300 as sk
    from split_bf16_gemm_swapped_gb300 import synthetic
    from split_bf16_gemm_swapped_gb300 import workloads as W
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    ws = list(W.ALL_FIXED) + W.all_sweep() if args.profile_case == "all" else [workload_by_name(args.profile_case)]
    a_cache = {}
    for w in ws:
        b = to_dev(w.make_b(), dev)
        c = torch.empty((w.L, w.M, w.N), dtype=torch.bfloat16, device=dev)
        if args.w4 or args.w8:
            aq, a_s = (synthetic.w4_weights if args.w4 else synthetic.w8_weights)(w.L, w.N, w.K, w.seed)
            q, s = torch.from_numpy(aq).to(dev), torch.from_numpy(a_s).to(dev)
            gemm = sk.splitk_gemm_w4a16 if args.w4 else sk.splitk_gemm_w8a16
            call = lambda: gemm(q, s, b, c, split_k=w.split_k)  # noqa: E731
        else:
            key = (w.N, w.K, w.L, w.seed)
            if key not in a_cache:
                a_cache.clear()
                torch.cuda.empty_cache()
                a_cache[key] = to_dev(w.make_a(), dev)
            a = a_cache[key]
            call = lambda: sk.splitk_gemm_bf16(a, b, c, split_k=w.split_k)  # noqa: E731
        for _ in range(args.warmup + args.steps):
            call()
        torch.cuda.synchronize(dev)
        rc = sk.splitk_get_status()
        print(json.dumps({"profile_case": describe(w), "key": workload_key(w), "w4": bool(args.w4), "w8": bool(args.w8),
                          "launches": args.warmup + args.steps, "status": rc}), flush=True)
        if rc != 0:
            raise SystemExit(1)


def ncu_traffic_table(csv_path: str, log_path: str, use_last: int) -> str:
    """The committed DRAM-traffic table from an ncu CSV of `--profile-case`
    runs (metrics dram__bytes_read.sum, dram__bytes_write.sum and
    gpu__time_duration.sum) and the run's own log, which names the workloads
    in launch order: per workload, the mean over its last `use_last`
    launches (the earlier ones are warm-up)."""
    import csv
    keys, per = [], []
    for line in Path(log_path).read_text().splitlines():
        if line.startswith("{"):
            d = json.loads(line)
            keys.append(d["key"])
            per.append(int(d["launches"]))
    launches = {}
    with open(csv_path) as f:
        rows = [r for r in csv.reader(f) if len(r) > 14]
    head = rows[0]
    col = {n: head.index(n) for n in ("ID", "Kernel Name", "Metric Name", "Metric Value")}
    for r in rows[1:]:
        i = int(r[col["ID"]])
        d = launches.setdefault(i, {"kernel": r[col["Kernel Name"]]})
        d[r[col["Metric Name"]]] = float(r[col["Metric Value"]].replace(",", ""))
    from split_bf16_gemm_swapped_gb300 import workloads as W  # noqa: F401
    out = []
    first = 0
    for key, n in zip(keys, per):
        ids = list(range(first + n - use_last, first + n))
        first += n
        got = [launches[i] for i in ids if i in launches]
        if not got:
            continue
        traffic = statistics.mean(g["dram__bytes_read.sum"] + g["dram__bytes_write.sum"] for g in got)
        dur = statistics.mean(g.get("gpu__time_duration.sum", 0.0) for g in got)
        w = workload_by_name(key)
        name = got[-1]["kernel"].replace("void ", "").split("(")[0]
        out.append(f"traffic {key}: {traffic:.0f} B  (algorithmic {w.bytes} B, {traffic / w.bytes:.3f}x; "
                   f"{name}; ncu duration {dur / 1e3:.1f} us, serialised)")
    return "\n".join(out)


NCU_SUMMARY_METRICS = [
    ("gpu__time_duration.sum", "duration (serialised, cold caches)"),
    ("dram__bytes_read.sum", "DRAM read"),
    ("dram__bytes_write.sum", "DRAM write"),
    ("gpu__dram_throughput.avg.pct_of_peak_sustained_elapsed", "DRAM throughput, % of peak"),
    ("lts__throughput.avg.pct_of_peak_sustained_elapsed", "L2 throughput, % of peak"),
    ("sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_elapsed", "tensor pipe active, % of elapsed"),
    ("sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_active", "tensor pipe active, % of SM-active"),
    ("sm__issue_active.avg.pct_of_peak_sustained_elapsed", "SM issue active, %"),
    ("sm__warps_active.avg.pct_of_peak_sustained_active", "warps active, % of peak"),
    ("smsp__inst_executed.sum", "warp instructions executed"),
    ("sm__icc_request_hit_rate.pct", "SM instruction-cache hit rate, %"),
    ("launch__registers_per_thread", "registers per thread"),
    ("launch__shared_mem_per_block_dynamic", "dynamic shared memory per CTA"),
    ("launch__grid_size", "CTAs"),
    ("launch__cluster_size", "cluster size"),
    ("launch__cluster_max_active", "clusters resident at once (max)"),
]


def quant_bytes(w, bits: int) -> int:
    """Bytes one quantized-weight call moves: the codes (`bits` a weight),
    the E8M0 scales (one byte per 32 weights), activations and output."""
    return w.L * (w.N * w.K * bits // 8 + w.N * w.K // 32 + 2 * w.M * w.K + 2 * w.M * w.N)


def ncu_summary(rep: str, key: str, w4: bool = False, w8: bool = False) -> str:
    """A markdown summary of one `ncu --set full` report: the kernel, its
    launch shape, duration, DRAM bytes against the algorithmic bytes of the
    workload `key`, DRAM / L2 / tensor-pipe utilisation and the top warp
    stall reasons."""
    import csv
    import io
    out = subprocess.run(["ncu", "-i", rep, "--page", "raw", "--csv"], capture_output=True, text=True,
                         check=True).stdout
    rows = list(csv.reader(io.StringIO(out)))
    head, units, vals = rows[0], rows[1], rows[2]
    get = {h: (u, v) for h, u, v in zip(head, units, vals)}
    w = workload_by_name(key)
    alg = quant_bytes(w, 4) if w4 else quant_bytes(w, 8) if w8 else w.bytes
    lines = [f"kernel: `{get.get('Kernel Name', ('', '?'))[1]}`",
             f"workload: {describe(w)}{' (A16W4 weights)' if w4 else ' (A16W8 weights)' if w8 else ''}; algorithmic bytes per launch {alg}", "",
             "| metric | value |", "|---|---|"]
    for m, label in NCU_SUMMARY_METRICS:
        if m in get and get[m][1] != "":
            u, v = get[m]
            lines.append(f"| {label} (`{m}`) | {v} {u} |")
    def to_bytes(m):
        u, v = get.get(m, ("", "0"))
        f = float(v.replace(",", "") or 0)
        return f * {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}.get(u, 1)
    traffic = to_bytes("dram__bytes_read.sum") + to_bytes("dram__bytes_write.sum")
    lines.append(f"| DRAM traffic / algorithmic bytes | {traffic / alg:.3f} |")
    stalls = []
    for h, (u, v) in get.items():
        if h.startswith("smsp__average_warps_issue_stalled_") and h.endswith("_per_issue_active.ratio"):
            try:
                stalls.append((float(v), h[len("smsp__average_warps_issue_stalled_"):-len("_per_issue_active.ratio")]))
            except ValueError:
                pass
    stalls.sort(reverse=True)
    lines.append("")
    lines.append("top warp stall reasons (warps stalled per issued instruction): " +
                 ", ".join(f"{n} {v:.2f}" for v, n in stalls[:5]))
    return "\n".join(lines)


def run_sweep_quant(args, bits: int):
    """Extra lines for the quantized-weight variants (A16W4: 4-bit E2M1
    weights, A16W8: 8-bit E4M3 weights, both with E8M0 scales per 32 k and
    bf16 activations) on the decode shapes: HBM TB/s of the bytes it moves
    (codes, scales, activations, output) and the step time next to the bf16
    kernel's on the same shape, both timed like the main line."""
    import torch

    import split_bf16_gemm_swapped_gb300 as sk
    from split_bf16_gemm_swapped_gb300 import synthetic
    from split_bf16_gemm_swapped_gb300 import workloads as W
    dev = torch.device("cuda:0")
    hbm, bf16, bf16s, src = peaks()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    s = torch.cuda.Stream(dev)

    def timed(launch, R):
        with torch.cuda.stream(s):
            for i in range(R + args.warmup):
                launch(i % R, s)
        s.synchronize()
        n = max(args.steps, R)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for i in range(n):
                launch(i % R, s)
        with torch.cuda.stream(s):
            g.replay()
        s.synchronize()
        one = time_replays(g, s, 1)[0]
        per = time_replays(g, s, repeats_for(one, args.min_ms))
        return statistics.median(per) / n * 1e-3

    for w in (W.DECODE_M1, W.DECODE_M16, W.TINY, W.DECODE_M1.with_(M=8), W.DECODE_M1.with_(M=32),
              W.DECODE_M1.with_(L=8), W.DECODE_M16.with_(L=4), W.DECODE_M1.with_(split_k=8)):
        aq, a_s = (synthetic.w4_weights if bits == 4 else synthetic.w8_weights)(w.L, w.N, w.K, w.seed)
        q0 = torch.from_numpy(aq).to(dev)
        s0 = torch.from_numpy(a_s).to(dev)
        w4_bytes = quant_bytes(w, bits)
        R = max(2, min(64, math.ceil(4 * l2 / (aq.nbytes + a_s.nbytes))))
        Qs = [q0] + [q0.clone() for _ in range(R - 1)]
        Ss = [s0] + [s0.clone() for _ in range(R - 1)]
        b = to_dev(w.make_b(), dev)
        c = torch.empty((w.L, w.M, w.N), dtype=torch.bfloat16, device=dev)
        gemm = sk.splitk_gemm_w4a16 if bits == 4 else sk.splitk_gemm_w8a16
        gemm_planned = sk.splitk_gemm_w4a16_planned if bits == 4 else sk.splitk_gemm_w8a16_planned
        plan = sk.splitk_plan_w4a16 if bits == 4 else sk.splitk_plan_w8a16
        t4 = timed(lambda i, st: gemm(Qs[i], Ss[i], b, c, split_k=w.split_k, stream=st), R)
        # the other decoder count, for comparison
        p_alt = plan(w.M, w.N, w.K, w.L, w.split_k)
        p_alt.w4_decoders = 3 - p_alt.w4_decoders
        try:
            t4_alt = timed(lambda i, st: gemm_planned(Qs[i], Ss[i], b, c, p_alt, 0, st), R)
        except sk.SplitKError:
            t4_alt = None
        a0 = to_dev(w.make_a(), dev)
        Rb = max(2, min(20, math.ceil(4 * l2 / (a0.numel() * 2))))
        As = [a0] + [a0.clone() for _ in range(Rb - 1)]
        tb = timed(lambda i, st: sk.splitk_gemm_bf16(As[i], b, c, split_k=w.split_k, stream=st), Rb)
        p = plan(w.M, w.N, w.K, w.L, w.split_k)
        print(json.dumps({"sweep": f"A16W{bits} " + describe(w), "us": round(t4 * 1e6, 2),
                          "TB/s": round(w4_bytes / t4 / 1e12, 3), "bytes_per_call": w4_bytes,
                          "hbm_frac": round(w4_bytes / t4 / 1e9 / hbm, 3), "peak_source": src,
                          "bf16_us": round(tb * 1e6, 2), "speedup_vs_bf16": round(tb / t4, 3),
                          f"us_with_{p_alt.w4_decoders}_decoders": round(t4_alt * 1e6, 2) if t4_alt else None,
                          "plan": {k: v for k, v in p.as_dict().items()
                                   if k in ("mma_n", "split_k", "stages", "a_tmem_tiles", "smem_bytes",
                                            "ctas_per_sm", "reduce_scatter", "b_loader", "mma_issuers",
                                            "w4_smem_tiles", "w4_decoders")}}), flush=True)
        del Qs, Ss, As, b, c
        torch.cuda.empty_cache()
    if sk.splitk_get_status() != 0:
        raise SystemExit(f"kernel fault during the sweep: {sk.splitk_get_fault()}")


def run_sweep_persistent(args):
    """Extra lines: for every sweep point with split >= 2 and the wide
    projection, the per-tile kernel's plan against the persistent kernel at
    each ring depth, each timed like the main line (a graph of --steps calls,
    median of back-to-back replays)."""
    import torch

    import split_bf16_gemm_swapped_gb300 as sk
    from split_bf16_gemm_swapped_gb300 import workloads as W
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = props.L2_cache_size
    stream = torch.cuda.Stream(dev)
    cache = {}
    ws = [w for w in W.all_sweep() if w.split_k >= 2] + [W.WIDE_S2, W.WIDE_S4]
    for w in ws:
        copies, _ = weight_copies(w, dev, l2, args.rotate, cache)
        R = len(copies)
        b = to_dev(w.make_b(), dev)
        c = torch.empty((w.L, w.M, w.N), dtype=torch.bfloat16, device=dev)
        cands = sk.splitk_plan_candidates_for(w.M, w.N, w.K, w.L, w.split_k, props.multi_processor_count,
                                              props.shared_memory_per_multiprocessor,
                                              props.shared_memory_per_block_optin)
        ring = next(p for p in cands if not p.persistent)
        plans = [("per-tile", ring)] + [(f"persistent n{p.mma_n} s{p.stages} r{p.reduce_rounds}", p)
                                        for p in cands if p.persistent]
        out = {}
        for name, plan in plans:
            def call(i, plan=plan):
                sk.splitk_gemm_bf16_planned(copies[i % R], b, c, plan, 0, stream)
            with torch.cuda.stream(stream):
                for i in range(max(args.warmup, R)):
                    call(i)
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(args.steps):
                    call(i)
            with torch.cuda.stream(stream):
                g.replay()
            stream.synchronize()
            one = time_replays(g, stream, 1)[0]
            ms = statistics.median(time_replays(g, stream, repeats_for(one, args.min_ms))) / args.steps
            out[name] = round(ms * 1e3, 2)
            del g
        best = min(out, key=out.get)
        hbm = peaks()[0]
        print(json.dumps({"sweep": "persistent vs per-tile " + describe(w), "us": out, "best": best,
                          "best_hbm_frac": round(w.bytes / (out[best] * 1e-6) / 1e9 / hbm, 3),
                          "planner": "persistent" if cands[0].persistent else "per-tile"}), flush=True)
        del b, c
    if sk.splitk_get_status() != 0:
        raise SystemExit(f"kernel fault during the sweep: {sk.splitk_get_fault()}")


def run_sweep_fixed(args):
    """Extra lines, one per fixed workload (tiny, the two decode shapes, the
    wide projection at both splits), timed like the main line."""
    import torch

    import split_bf16_gemm_swapped_gb300 as sk
    from split_bf16_gemm_swapped_gb300 import workloads as W
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    stream = torch.cuda.Stream(dev)
    traffic = traffic_table()
    cache = {}
    for w in W.ALL_FIXED:
        copies, rot = weight_copies(w, dev, l2, args.rotate, cache)
        pt = Point(w, copies, dev, stream, args.steps, args.warmup)
        reps = repeats_for(pt.replay_ms_estimate, args.min_ms)
        ms = statistics.median(time_replays(pt.graph, stream, reps)) / args.steps
        rec = point_record(w, ms, reps, args.steps, pt.plan, traffic, 1)
        print(json.dumps({"sweep": describe(w), "l2": rot} | rec), flush=True)
        del pt
        cache.clear()
        torch.cuda.empty_cache()
    if sk.splitk_get_status() != 0:
        raise SystemExit(f"kernel fault during the sweep: {sk.splitk_get_fault()}")


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1,
                    help="GPUs (one rank each under torch.distributed.run; each runs a replica)")
    ap.add_argument("--steps", type=int, default=200, help="calls per timed graph (one GEMM call each)")
    ap.add_argument("--warmup", type=int, default=10, help="untimed calls first, per point (at least 3)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours",
                    help="reference: the float64 CPU oracle on the host cores")
    ap.add_argument("--workload", default="sweep",
                    help="sweep (the default line), decode_m1, decode_m16, tiny, wide_s2, wide_s4, "
                         "sweep_m<M>_s<split>")
    ap.add_argument("--min-ms", type=float, default=40.0,
                    help="GPU time each point's back-to-back replays cover at least")
    ap.add_argument("--sweep", choices=["fixed", "w4a16", "w8a16", "persistent"], default=None,
                    help="extra lines instead of the contract line: the fixed workloads, A16W4, A16W8, or "
                         "the per-tile against the persistent kernel")
    ap.add_argument("--no-extras", action="store_true", help="skip the decode workloads of the sweep line")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the timed oracle leg")
    ap.add_argument("--no-e2e", dest="e2e", action="store_false", help="skip the end-to-end measurement")
    ap.add_argument("--rotate", type=int, default=0,
                    help="weight copies to rotate (default: enough for 4x the L2 cache)")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of host time for the CPU oracle baseline")
    ap.add_argument("--cpu-table", action="store_true",
                    help="time the oracle alone (all host cores and one) on the fixed and sweep workloads")
    ap.add_argument("--profile-case", default=None,
                    help="a short eager run for ncu of one workload, or `all` of them in turn "
                         "(no graphs, one weight copy)")
    ap.add_argument("--w4", action="store_true", help="with --profile-case: the A16W4 kernel")
    ap.add_argument("--w8", action="store_true", help="with --profile-case: the A16W8 kernel")
    ap.add_argument("--ncu-summary", nargs=2, metavar=("REPORT", "WORKLOAD"), default=None,
                    help="print a markdown summary of an ncu --set full report of WORKLOAD (with --w4 / --w8: "
                         "A16W4 / A16W8)")
    ap.add_argument("--ncu-table", nargs=2, metavar=("CSV", "LOG"), default=None,
                    help="print the DRAM-traffic table from an ncu CSV of a --profile-case run and its log")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.steps < 1:
        raise SystemExit("--steps must be >= 1")
    if args.w4 and args.w8:
        raise SystemExit("--w4 and --w8 exclude each other")
    if args.workload != "sweep":
        workload_by_name(args.workload)
    if args.profile_case not in (None, "all"):
        workload_by_name(args.profile_case)
    if args.ncu_summary:
        print(ncu_summary(args.ncu_summary[0], args.ncu_summary[1], args.w4, args.w8))
    elif args.ncu_table:
        print(ncu_traffic_table(args.ncu_table[0], args.ncu_table[1], args.steps))
    elif args.cpu_table:
        run_cpu_table(args)
    elif args.impl == "reference":
        run_reference(args)
    elif args.profile_case:
        run_profile_case(args)
    elif args.sweep in ("w4a16", "w8a16"):
        run_sweep_quant(args, 4 if args.sweep == "w4a16" else 8)
    elif args.sweep == "fixed":
        run_sweep_fixed(args)
    elif args.sweep == "persistent":
        run_sweep_persistent(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
