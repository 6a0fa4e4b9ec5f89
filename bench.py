#!/usr/bin/env python3
"""Benchmark of the quantized-gradient hot path on GB300.

Default workload: one qgZ single-hop step (8 simulated ranks, gradients of
one d=2048/ffn=5504 Llama-2 layer, block 256, LoCo error feedback s=1,
beta=0.5): the error-feedback int4 quantization of every rank followed by
the dequant-reduce of every destination shard.  Metric: gradient elements
per second (R*N per step) through both kernels.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload qgz_single_hop|qgz_fused|qgz_bf16ef|qgz_int8ef|qgz_hier_ef|
                                qgz_hier_fused|qgz_hier_ef_fused|qgz_bf16ef_fused|
                                qgz_int8ef_fused|qgz_tiny|qgz_hierarchical|qwz|sr|all]

The other workloads: the same step as one fused kernel (qgz_fused), with a
bf16 or an int8 error buffer (qgz_bf16ef, qgz_int8ef; fused: qgz_bf16ef_fused,
qgz_int8ef_fused), the 16-rank two-hop reduce without and with
first-hop error feedback (qgz_hierarchical, qgz_hier_ef), the same with its
first stage as one kernel (qgz_hier_fused, qgz_hier_ef_fused), the L2-resident
4-rank step (qgz_tiny), the qwZ int8 round trip and one-pass replica (qwz),
and the bf16 stochastic-rounding accumulate (sr).

One JSON line on rank 0 (per workload).  Under torchrun each rank runs an
independent replica on its own GPU ("weak" scaling; the simulated ranks live
in one GPU, there is no cross-GPU exchange); the time is the max over ranks.
`--impl reference` times the CPU oracle (a plain single-threaded C
statement of the same computation) on a bounded sample of the workload.
"""
from __future__ import annotations

import argparse
import dataclasses
import datetime as _dt
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time
from pathlib import Path

import numpy as np
import torch

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

from weight_communication_gb300 import workloads as wl  # noqa: E402

METRIC = "qgZ grad elements/s (EF-quant + dequant-reduce) and HBM GB/s vs GB300 peak"
# --impl reference: total oracle time to aim for, and a conservative
# single-threaded oracle rate on the host (gradient elements per second)
REFERENCE_BUDGET_S = 150.0
ORACLE_ELEMENTS_PER_S = 1.2e8
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024


# ---------------------------------------------------------------------------
# environment
# ---------------------------------------------------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws: int, use_cuda: bool):
    if ws <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group("nccl" if use_cuda else "gloo")
    return dist


def max_over_ranks(value: float, dist, device) -> float:
    """Largest value across ranks (the job's time is the slowest rank's)."""
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank_step: float, ws: int, max_ms_per_step: float) -> float:
    """Whole-job rate: every replica processes the same units per step and
    the job advances at the pace of the slowest rank."""
    return units_per_rank_step * ws / (max_ms_per_step / 1e3)


def barrier(dist):
    if dist is not None:
        dist.barrier()


def measured_peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            d = json.loads(p.read_text())
            return float(d["hbm_gbs"]), "measured"
        except (ValueError, KeyError):
            pass
    return FALLBACK_HBM_GBS, "fallback"


def host_cpu():
    model = ""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    return os.cpu_count() or 1, model


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons (read-only)."""
    QUERY = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int, period_ms: int = 20):
        self.proc = None
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-i", str(gpu_index), "-lms", str(period_ms)],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        rows = Path(self.file.name).read_text().splitlines()
        os.unlink(self.file.name)
        return self.parse(rows, t0, t1)

    @classmethod
    def parse(cls, rows, t0: float, t1: float):
        """Median SM clock, max clock and active throttle reasons of the
        samples taken between host times t0 and t1."""
        sm, smax, reasons = [], [], set()
        for row in rows:
            f = [x.strip() for x in row.split(",")]
            if len(f) < 9:
                continue
            try:
                ts = _dt.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                continue
            if not (t0 - 0.05 <= ts <= t1 + 0.05):
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, v in zip(cls.REASONS, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# traffic figures from the committed ncu summaries
# ---------------------------------------------------------------------------

KERNEL_SOURCES = {
    "ef_quant_int4": ["weight_communication_gb300/csrc/qgz_quant.cu",
                      "weight_communication_gb300/csrc/int8_error_block.cuh",
                      "weight_communication_gb300/csrc/wc_device.cuh"],
    "dequant_reduce": ["weight_communication_gb300/csrc/qgz_reduce.cu",
                       "weight_communication_gb300/csrc/wc_device.cuh"],
    "dequant_reduce_requant": ["weight_communication_gb300/csrc/qgz_hop1.cu",
                               "weight_communication_gb300/csrc/wc_device.cuh"],
    "qwz_quant_int8": ["weight_communication_gb300/csrc/qwz.cu",
                       "weight_communication_gb300/csrc/wc_device.cuh"],
    "qwz_dequant_int8": ["weight_communication_gb300/csrc/qwz.cu",
                         "weight_communication_gb300/csrc/wc_device.cuh"],
    "sr_accumulate": ["weight_communication_gb300/csrc/sr_accumulate.cu",
                      "weight_communication_gb300/csrc/wc_device.cuh"],
    "qgz_step_fused": ["weight_communication_gb300/csrc/qgz_fused.cu",
                      "weight_communication_gb300/csrc/int8_error_block.cuh",
                       "weight_communication_gb300/csrc/wc_device.cuh"],
    "qgz_first_hop_fused": ["weight_communication_gb300/csrc/qgz_fused.cu",
                           "weight_communication_gb300/csrc/int8_error_block.cuh",
                            "weight_communication_gb300/csrc/wc_device.cuh"],
    "qgz_first_hop_fused_ef1": ["weight_communication_gb300/csrc/qgz_fused.cu",
                               "weight_communication_gb300/csrc/int8_error_block.cuh",
                                "weight_communication_gb300/csrc/wc_device.cuh"],
}


def kernel_source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        h.update((ROOT / rel).read_bytes())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str, units: float):
    """DRAM bytes per launch from profiles/traffic.txt, scaled to `units`
    elements, or None when absent or taken on a different kernel source."""
    p = ROOT / "profiles" / "traffic.txt"
    if not p.exists():
        return None
    for line in p.read_text().splitlines():
        f = line.split()
        if len(f) < 5 or line.startswith("#"):
            continue
        k, wname, bytes_, units_measured, src = f[:5]
        if k == kernel and wname == workload and src == kernel_source_hash(kernel):
            return float(bytes_) * units / float(units_measured)
    return None


# ---------------------------------------------------------------------------
# timed loops
# ---------------------------------------------------------------------------

def clocks_begin(args, dev):
    """Start sampling the SM clocks before a timed region (None when off)."""
    if not args.clocks:
        return None
    sampler = ClockSampler(dev.index or 0)
    time.sleep(0.2)
    return sampler


def flush_l2(buf: torch.Tensor):
    buf.add_(1)


def percentiles(xs):
    """{median, p10, p90} of a list of times (nearest-rank percentiles)."""
    ys = sorted(xs)
    pick = lambda q: ys[min(len(ys) - 1, max(0, int(math.ceil(q * len(ys))) - 1))]
    return {"median": round(statistics.median(ys), 5), "p10": round(pick(0.10), 5),
            "p90": round(pick(0.90), 5)}


class Timer:
    """CUDA events on the launching stream around every kernel of a step."""

    def __init__(self, names, steps):
        self.names = names
        self.ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
                   for _ in range(steps)]

    def mark(self, step, i):
        self.ev[step][i].record()

    def per_kernel_ms(self):
        out = {}
        for j, n in enumerate(self.names):
            out[n] = statistics.mean(e[j].elapsed_time(e[j + 1]) for e in self.ev)
        return out

    def per_kernel_percentiles(self):
        """Median, 10th and 90th percentile of each kernel's launch times (ms)."""
        out = {}
        for j, n in enumerate(self.names):
            out[n] = percentiles([e[j].elapsed_time(e[j + 1]) for e in self.ev])
        return out

    def step_sum_ms(self):
        return statistics.mean(e[0].elapsed_time(e[-1]) for e in self.ev)


def wire_bytes(w: wl.QgzWorkload) -> dict:
    """Bytes each gradient element puts on the wire per exchange: a 4-bit code
    plus its share of the block's fp32 scale, against bf16 (2 bytes) and an
    ideal int4 with no scales (0.5)."""
    return {"int4_blocked": 0.5 + 4 / w.B, "bf16": 2.0, "int4_no_scales": 0.5,
            "exchanges_per_step": 2 if w.G > 1 else 1}


def launch_overhead(red, g: torch.Tensor, dev, dist, n: int) -> dict:
    """The same step issued n times back to back (no flush between steps),
    once as eager calls and once as replays of a CUDA graph of the step
    (qgz.GraphedStep): the difference is the host's launch work."""
    from weight_communication_gb300.qgz import GraphedStep
    ev = lambda: torch.cuda.Event(enable_timing=True)
    gv = g.reshape(-1)
    for _ in range(3):
        red.step(gv)
    torch.cuda.synchronize(dev)
    a, b = ev(), ev()
    a.record()
    for _ in range(n):
        red.step(gv)
    b.record()
    torch.cuda.synchronize(dev)
    eager = a.elapsed_time(b) / n
    graphed = GraphedStep(red)
    graphed.g.copy_(gv)
    for _ in range(3):
        graphed.replay()
    torch.cuda.synchronize(dev)
    a, b = ev(), ev()
    a.record()
    for _ in range(n):
        graphed.replay()
    b.record()
    torch.cuda.synchronize(dev)
    graph = a.elapsed_time(b) / n
    return {"eager_ms_per_step": max_over_ranks(eager, dist, dev),
            "graph_ms_per_step": max_over_ranks(graph, dist, dev), "steps": n,
            "how": "steps back to back, no flush: eager binding calls vs one CUDA-graph "
                   "replay per step (qgz.GraphedStep)"}


EF_DTYPES = {"fp32": torch.float32, "bf16": torch.bfloat16, "int8": torch.int8}


def run_qgz(w: wl.QgzWorkload, args, dev, dist, ws, ef: str = "fp32", hop1_ef: bool = False):
    """One qgZ step per timed iteration; ef names the error buffer's form
    ("fp32", "bf16": wc_ef_quant_int4_bf16ef, "int8": wc_ef_quant_int4_int8ef);
    hop1_ef adds error feedback to the first hop's requantization
    (hierarchical only)."""
    from weight_communication_gb300.qgz import QgzReducer
    out_dtype = torch.bfloat16 if w.out_bf16 else torch.float32
    red = QgzReducer(w.N, w.R, w.G, w.B, w.err_scale, w.err_beta, out_dtype=out_dtype, device=dev,
                     ef_dtype=EF_DTYPES[ef], hop1_ef=hop1_ef)
    g_bytes = w.R * w.N * 2
    nbatch = max(1, min(args.batches, (8 << 30) // g_bytes))
    batches = [wl.qgz_gradients(w, t, device=dev) for t in range(nbatch)]
    stream = torch.cuda.Stream(dev)
    l2_resident = (w.R * w.N * (2 + 4 + 4) + w.N * 4) < 2 * L2_BYTES
    flush = torch.empty(4 * L2_BYTES // 4, dtype=torch.float32, device=dev) if l2_resident else None
    names = ["ef_quant_int4"] + (["dequant_reduce_requant"] if w.G > 1 else []) + ["dequant_reduce"]

    def step(i, timer=None, ti=None):
        g = batches[i % nbatch]
        if timer is not None:
            timer.mark(ti, 0)
        red.quantize(g, stream)
        if timer is not None:
            timer.mark(ti, 1)
        if w.G > 1:
            red.reduce_first_hop(stream)
            if timer is not None:
                timer.mark(ti, 2)
        red.reduce_last_hop(stream)
        if timer is not None:
            timer.mark(ti, len(names))

    # Headline: steps one after another on one stream, each kernel bracketed
    # by events (with an L2 flush between steps for L2-resident workloads).
    # For the others a second, shorter pass runs the steps through
    # DevicePipeline (each reduce on a second stream beside the next
    # quantization) and is reported beside it; --no-overlap skips that pass.
    overlap = flush is None and not args.no_overlap
    sampler = None
    timer = Timer(names, args.steps)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
            if flush is not None:
                flush_l2(flush)
        torch.cuda.synchronize(dev)
        sampler = clocks_begin(args, dev)
        barrier(dist)
        torch.cuda.synchronize(dev)
        t0 = time.time()
        start.record()
        for i in range(args.steps):
            step(args.warmup + i, timer, i)
            if flush is not None:
                flush_l2(flush)
        end.record()
        torch.cuda.synchronize(dev)
        t1 = time.time()
        barrier(dist)
    per_kernel = timer.per_kernel_ms()
    per_kernel_pct = timer.per_kernel_percentiles()
    # with a flush the step time is the kernels' span (the flush is not part of it)
    ms_local = timer.step_sum_ms() if flush is not None else start.elapsed_time(end) / args.steps
    overlapped = None
    if overlap:
        from weight_communication_gb300.qgz import DevicePipeline
        pipe = DevicePipeline(red)
        n_ov = max(1, min(args.steps, 200))
        for i in range(3):
            pipe.step(batches[i % nbatch])
        torch.cuda.synchronize(dev)
        o0, o1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        o0.record(pipe.quant_stream)
        for i in range(n_ov):
            pipe.step(batches[i % nbatch])
        o1.record(pipe.reduce_stream)
        torch.cuda.synchronize(dev)
        overlapped = max_over_ranks(o0.elapsed_time(o1) / n_ov, dist, dev)
    clocks = sampler.stop(t0, t1) if sampler else None
    ms = max_over_ranks(ms_local, dist, dev)
    units = w.R * w.N
    value = job_throughput(units, ws, ms)

    # roofline of the dominant kernel (the error-feedback quantization), from
    # its launches inside the timed region
    peak, peak_kind = measured_peaks()
    # error buffer bytes per element, read and written: fp32 4 + 4, bf16 2 + 2,
    # int8 1 + 1 plus the block scale's share both ways
    ef_rw = {"fp32": 8.0, "bf16": 4.0, "int8": 2.0 + 8.0 / w.B}[ef]
    efq_bytes = w.R * w.N * (2 + ef_rw + 0.5) + w.R * w.N // w.B * 4
    efq_ms = per_kernel["ef_quant_int4"]
    achieved = efq_bytes / (efq_ms / 1e3) / 1e9
    efq_kernel = {"fp32": "ef_quant_int4", "bf16": "ef_quant_int4_bf16ef",
                  "int8": "ef_quant_int4_int8ef"}[ef]
    traffic = ncu_traffic(efq_kernel, w.name.split()[0], units) if ef == "fp32" else None
    kernels = {}
    S = w.S
    for n in names:
        if n == "ef_quant_int4":
            b = efq_bytes
        elif n == "dequant_reduce_requant":
            b = w.G * w.N * (w.L + 1) * (0.5 + 4 / w.B) + (8 * w.G * w.N if hop1_ef else 0)
        else:
            nsrc = w.G if w.G > 1 else w.R
            b = w.N * (nsrc * (0.5 + 4 / w.B) + (2 if w.out_bf16 else 4))
        t = per_kernel[n]
        kernels[n] = {"ms": round(t, 5), "ms_percentiles": per_kernel_pct[n],
                      "algorithmic_bytes": int(b),
                      "GB/s": round(b / (t / 1e3) / 1e9, 1),
                      "frac": round(b / (t / 1e3) / 1e9 / peak, 4)}
    line = {
        "metric": METRIC, "value": value, "unit": "elements/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded normal gradients with sparse outliers)",
        "config": {"workload": w.name + (f" {ef} error buffer" if ef != "fp32" else "")
                   + (" + first-hop error feedback" if hop1_ef else ""),
                   "R": w.R, "N": w.N, "G": w.G, "B": w.B,
                   "err_scale": w.err_scale, "err_beta": w.err_beta,
                   "ef": ef,
                   "out": "bf16" if w.out_bf16 else "fp32",
                   "l2": ("flushed between steps (untimed 516 MB write)" if flush is not None
                          else f"inputs exceed L2 ({units * 10 / 1e9:.1f} GB per step)"),
                   "steps": "one after another on one stream",
                   "parallelism": f"replicas x{ws}"},
        "roofline": {"bound": "hbm", "kernel": efq_kernel, "achieved": round(achieved, 1),
                     "peak": peak, "peak_kind": f"hbm_gbs of {peak_kind}", "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": traffic, "algorithmic_bytes": int(efq_bytes),
                     "dram_GB/s": (round(traffic / (efq_ms / 1e3) / 1e9, 1)
                                   if traffic is not None else None)},
        "kernels": kernels,
        "wire_bytes_per_element": wire_bytes(w),
        "gpu_launches": args.steps * len(names),
        "clocks": clocks,
    }
    line["launch_overhead"] = launch_overhead(red, batches[0], dev, dist,
                                              max(1, min(args.steps, 200)))
    if overlapped is not None:
        line["overlapped_ms_per_step"] = overlapped
        line["overlapped_how"] = ("each step's reduce on a second stream beside the next "
                                  "step's EF-quant, event-ordered (qgz.DevicePipeline)")
    if not args.no_e2e:
        line["e2e"] = run_qgz_e2e(w, red, batches[0], args, dev, dist, ws, stream)
    return line, batches[0]


EF_DTYPES = {"fp32": torch.float32, "bf16": torch.bfloat16, "int8": torch.int8}
EF_BYTES = {"fp32": 4, "bf16": 2, "int8": 1}     # per element, each way


def run_qgz_fused(w: wl.QgzWorkload, args, dev, dist, ws, ef_kind: str = "fp32"):
    """The flat step as one fused launch (EF-quant of every rank + reduce),
    writing the error buffers (fp32, bf16, or int8 with block scales), the
    send buffers and the shards."""
    from weight_communication_gb300 import binding
    assert w.G == 1
    out_dtype = torch.bfloat16 if w.out_bf16 else torch.float32
    ef = torch.zeros(w.R * w.N, dtype=EF_DTYPES[ef_kind], device=dev)
    ef_scales = (torch.zeros(w.R * w.N // w.B, dtype=torch.float32, device=dev)
                 if ef_kind == "int8" else None)
    codes = torch.empty(w.R * w.N // 2, dtype=torch.uint8, device=dev)
    scales = torch.empty(w.R * w.N // w.B, dtype=torch.float32, device=dev)
    out = torch.empty(w.N, dtype=out_dtype, device=dev)
    nbatch = max(1, min(args.batches, (8 << 30) // (w.R * w.N * 2)))
    batches = [wl.qgz_gradients(w, t, device=dev) for t in range(nbatch)]
    stream = torch.cuda.Stream(dev)
    names = ["qgz_step_fused"]
    with torch.cuda.stream(stream):
        def step(i):
            binding.qgz_step_fused(batches[i % nbatch].view(-1), ef, codes, scales, out, w.N,
                                   w.R, w.B, w.err_scale, w.err_beta, 1.0, stream,
                                   ef_scales=ef_scales)
        for i in range(args.warmup):
            step(i)
        torch.cuda.synchronize(dev)
        timer = Timer(names, args.steps)
        sampler = clocks_begin(args, dev)
        barrier(dist)
        t0 = time.time()
        for i in range(args.steps):
            timer.mark(i, 0)
            step(args.warmup + i)
            timer.mark(i, 1)
        torch.cuda.synchronize(dev)
        t1 = time.time()
        barrier(dist)
    clocks = sampler.stop(t0, t1) if sampler else None
    ms = max_over_ranks(timer.step_sum_ms(), dist, dev)
    peak, kind = measured_peaks()
    eb = EF_BYTES[ef_kind]
    b = (w.R * w.N * (2 + 2 * eb + 0.5) + w.R * w.N // w.B * (12 if ef_kind == "int8" else 4)
         + w.N * (2 if w.out_bf16 else 4))
    achieved = b / (ms / 1e3) / 1e9
    tag = "fused single kernel" + ("" if ef_kind == "fp32" else f", {ef_kind} error buffer")
    return {"metric": METRIC + f" [{tag}]", "value": job_throughput(w.R * w.N, ws, ms),
            "unit": "elements/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic (seeded normal gradients with sparse outliers)",
            "config": {"workload": w.name + (" fused" if ef_kind == "fp32"
                                             else f" fused {ef_kind} error buffer"),
                       "R": w.R, "N": w.N, "G": 1, "B": w.B, "ef": ef_kind,
                       "err_scale": w.err_scale, "err_beta": w.err_beta,
                       "l2": f"inputs exceed L2 ({b / 1e9:.1f} GB per step)"},
            "roofline": {"bound": "hbm", "kernel": "qgz_step_fused", "achieved": round(achieved, 1),
                         "peak": peak, "peak_kind": f"hbm_gbs of {kind}", "unit": "GB/s",
                         "frac": round(achieved / peak, 4),
                         "traffic": (ncu_traffic("qgz_step_fused", "qgz_single_hop", w.R * w.N)
                                     if ef_kind == "fp32" else None),
                         "algorithmic_bytes": int(b)},
            "kernels": {"qgz_step_fused": {"ms": round(ms, 5),
                                           "ms_percentiles": timer.per_kernel_percentiles()[
                                               "qgz_step_fused"],
                                           "algorithmic_bytes": int(b),
                                           "GB/s": round(achieved, 1),
                                           "frac": round(achieved / peak, 4)}},
            "gpu_launches": args.steps, "clocks": clocks}, None


def run_qgz_hier_fused(w: wl.QgzWorkload, args, dev, dist, ws, hop1_ef: bool = False):
    """The hierarchical step with its first stage as one kernel (every rank's
    EF-quant fused with the first hop, writing the error buffers, the send
    buffers and the first hop's output; with hop1_ef the first hop also keeps
    its own error buffer), then the second hop."""
    from weight_communication_gb300 import binding
    assert w.G > 1
    ef = torch.zeros(w.R * w.N, dtype=torch.float32, device=dev)
    ef1 = torch.zeros(w.G * w.N, dtype=torch.float32, device=dev) if hop1_ef else None
    codes = torch.empty(w.R * w.N // 2, dtype=torch.uint8, device=dev)
    scales = torch.empty(w.R * w.N // w.B, dtype=torch.float32, device=dev)
    c1 = torch.empty(w.G * w.N // 2, dtype=torch.uint8, device=dev)
    s1 = torch.empty(w.G * w.N // w.B, dtype=torch.float32, device=dev)
    out = torch.empty(w.N, dtype=torch.bfloat16 if w.out_bf16 else torch.float32, device=dev)
    nbatch = max(1, min(args.batches, (8 << 30) // (w.R * w.N * 2)))
    batches = [wl.qgz_gradients(w, t, device=dev) for t in range(nbatch)]
    stream = torch.cuda.Stream(dev)
    names = ["qgz_first_hop_fused", "dequant_reduce"]
    with torch.cuda.stream(stream):
        def step(i, timer=None, ti=None):
            if timer is not None:
                timer.mark(ti, 0)
            binding.qgz_first_hop_fused(batches[i % nbatch].view(-1), ef, codes, scales, c1, s1,
                                        w.N, w.R, w.G, w.B, w.err_scale, w.err_beta, stream,
                                        ef1=ef1)
            if timer is not None:
                timer.mark(ti, 1)
            binding.dequant_reduce(c1, s1, out, w.N, w.R, w.G, w.B, 1.0, stream)
            if timer is not None:
                timer.mark(ti, 2)
        for i in range(args.warmup):
            step(i)
        torch.cuda.synchronize(dev)
        timer = Timer(names, args.steps)
        sampler = clocks_begin(args, dev)
        barrier(dist)
        t0 = time.time()
        for i in range(args.steps):
            step(args.warmup + i, timer, i)
        torch.cuda.synchronize(dev)
        t1 = time.time()
        barrier(dist)
    clocks = sampler.stop(t0, t1) if sampler else None
    ms = max_over_ranks(timer.step_sum_ms(), dist, dev)
    per = timer.per_kernel_ms()
    pct = timer.per_kernel_percentiles()
    peak, kind = measured_peaks()
    kb = {"qgz_first_hop_fused": int(w.R * w.N * (2 + 8 + 0.5) + w.R * w.N // w.B * 4
                                     + w.G * w.N * (0.5 + 4 / w.B + (8 if hop1_ef else 0))),
          "dequant_reduce": int(w.N * (w.G * (0.5 + 4 / w.B) + (2 if w.out_bf16 else 4)))}
    kernels = {n: {"ms": round(per[n], 5), "ms_percentiles": pct[n], "algorithmic_bytes": kb[n],
                   "GB/s": round(kb[n] / (per[n] / 1e3) / 1e9, 1),
                   "frac": round(kb[n] / (per[n] / 1e3) / 1e9 / peak, 4)} for n in names}
    tag = "fused first stage with first-hop EF" if hop1_ef else "fused first stage"
    return {"metric": METRIC + f" [hierarchical, {tag}]",
            "value": job_throughput(w.R * w.N, ws, ms), "unit": "elements/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded normal gradients with sparse outliers)",
            "config": {"workload": f"{w.name} {tag}", "R": w.R, "N": w.N, "G": w.G,
                       "B": w.B, "err_scale": w.err_scale, "err_beta": w.err_beta,
                       "ef1": "fp32" if hop1_ef else None,
                       "l2": f"inputs exceed L2 ({w.R * w.N * 10 / 1e9:.1f} GB per step)"},
            "roofline": {"bound": "hbm", "kernel": "qgz_first_hop_fused",
                         "achieved": kernels["qgz_first_hop_fused"]["GB/s"], "peak": peak,
                         "peak_kind": f"hbm_gbs of {kind}", "unit": "GB/s",
                         "frac": kernels["qgz_first_hop_fused"]["frac"],
                         "traffic": ncu_traffic("qgz_first_hop_fused_ef1" if hop1_ef
                                                else "qgz_first_hop_fused", "qgz_hierarchical",
                                                w.R * w.N),
                         "algorithmic_bytes": kb["qgz_first_hop_fused"]},
            "kernels": kernels, "gpu_launches": 2 * args.steps, "clocks": clocks}, None


def parse_cpulist(text: str) -> list[int]:
    """'0-3,8,10-11' -> [0, 1, 2, 3, 8, 10, 11]."""
    cpus = []
    for part in text.strip().split(","):
        if not part:
            continue
        if "-" in part:
            a, b = part.split("-")
            cpus.extend(range(int(a), int(b) + 1))
        else:
            cpus.append(int(part))
    return cpus


def bind_host_to_gpu(dev) -> str:
    """Run this process on the CPUs next to the GPU, so that pinned host
    buffers allocated afterwards sit in that socket's memory.  Best effort:
    returns what was done."""
    try:
        out = subprocess.run(["nvidia-smi", "--query-gpu=pci.bus_id", "--format=csv,noheader",
                              "-i", str(dev.index or 0)], capture_output=True, text=True,
                             timeout=20).stdout.strip()
        dom, bus, rest = out.split(":")
        path = Path(f"/sys/bus/pci/devices/{int(dom, 16):04x}:{bus.lower()}:{rest.lower()}")
        cpus = parse_cpulist((path / "local_cpulist").read_text())
        online = set(os.sched_getaffinity(0))
        cpus = [c for c in cpus if c in online]
        if not cpus:
            return "not bound (no local CPUs)"
        os.sched_setaffinity(0, cpus)
        return f"bound to {len(cpus)} CPUs local to the GPU"
    except (OSError, ValueError, subprocess.SubprocessError):
        return "not bound (topology unavailable)"


def run_qgz_e2e(w, red, g_example, args, dev, dist, ws, stream):
    """Same metric through the public API with host buffers: every step copies
    its gradients host -> device (pinned), runs the kernels and copies the
    reduced shards device -> host, all inside the timed region.  The steps run
    through HostPipeline, so one step's copies overlap its neighbours' work;
    the serial form (copy, kernels, copy, then the next step) is reported
    beside it."""
    from weight_communication_gb300.qgz import HostPipeline
    binding_note = bind_host_to_gpu(dev)
    g_bytes = g_example.numel() * g_example.element_size()
    n_host = 2 if g_bytes <= (2 << 30) else 1
    g_host = [g_example.cpu().pin_memory() for _ in range(n_host)]
    out_host = [torch.empty(red.out.shape, dtype=red.out.dtype).pin_memory() for _ in range(2)]
    steps = max(1, min(args.steps, 200))
    pipe = HostPipeline(red)

    def seq(n):
        return [g_host[i % n_host] for i in range(n)], [out_host[i % 2] for i in range(n)]

    pipe.run(*seq(max(2, args.warmup)))
    torch.cuda.synchronize(dev)
    barrier(dist)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(pipe.h2d)
    pipe.run(*seq(steps))
    pipe.d2h.wait_stream(pipe.h2d)
    end.record(pipe.d2h)
    torch.cuda.synchronize(dev)
    barrier(dist)
    ms = max_over_ranks(start.elapsed_time(end) / steps, dist, dev)

    # serial form for comparison
    g_dev = torch.empty_like(g_example)
    with torch.cuda.stream(stream):
        red.step_host(g_host[0], g_dev, out_host[0], stream)
        torch.cuda.synchronize(dev)
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_serial = max(1, min(steps, 50))
        s0.record()
        for _ in range(n_serial):
            red.step_host(g_host[0], g_dev, out_host[0], stream)
        s1.record()
        torch.cuda.synchronize(dev)
    serial_ms = max_over_ranks(s0.elapsed_time(s1) / n_serial, dist, dev)
    return {"value": w.R * w.N * ws / (ms / 1e3), "unit": "elements/s", "ms_per_step": ms,
            "h2d_bytes_per_step": g_bytes,
            "d2h_bytes_per_step": out_host[0].numel() * out_host[0].element_size(),
            "pipelined": True, "serial_ms_per_step": serial_ms, "host_memory": binding_note}


def run_qwz(w: wl.QwzWorkload, args, dev, dist, ws):
    from weight_communication_gb300 import binding
    wd = wl.qwz_weights(w, device=dev)
    codes = torch.empty(w.n, dtype=torch.int8, device=dev)
    scales = torch.empty(w.n // w.B, dtype=torch.float32, device=dev)
    back = torch.empty(w.n, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(dev)
    names = ["qwz_quant_int8", "qwz_dequant_int8"]
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            binding.qwz_quant_int8(wd, codes, scales, w.B, stream)
            binding.qwz_dequant_int8(codes, scales, back, w.B, stream)
        torch.cuda.synchronize(dev)
        timer = Timer(names, args.steps)
        sampler = clocks_begin(args, dev)
        barrier(dist)
        t0 = time.time()
        for i in range(args.steps):
            timer.mark(i, 0)
            binding.qwz_quant_int8(wd, codes, scales, w.B, stream)
            timer.mark(i, 1)
            binding.qwz_dequant_int8(codes, scales, back, w.B, stream)
            timer.mark(i, 2)
        torch.cuda.synchronize(dev)
        t1 = time.time()
        barrier(dist)
    clocks = sampler.stop(t0, t1) if sampler else None
    # the one-pass variant that writes the codes and the bf16 replica, timed
    # on its own (not part of the round-trip step)
    rep_steps = max(1, min(args.steps, 200))
    with torch.cuda.stream(stream):
        for _ in range(3):
            binding.qwz_quant_replica_int8(wd, codes, scales, back, w.B, stream)
        rtimer = Timer(["qwz_quant_replica_int8"], rep_steps)
        for i in range(rep_steps):
            rtimer.mark(i, 0)
            binding.qwz_quant_replica_int8(wd, codes, scales, back, w.B, stream)
            rtimer.mark(i, 1)
        torch.cuda.synchronize(dev)
    per = timer.per_kernel_ms()
    per.update(rtimer.per_kernel_ms())
    pct = timer.per_kernel_percentiles()
    pct.update(rtimer.per_kernel_percentiles())
    ms = max_over_ranks(timer.step_sum_ms(), dist, dev)
    peak, kind = measured_peaks()
    qb = w.n * (2 + 1) + w.n // w.B * 4
    kb = {"qwz_quant_int8": qb, "qwz_dequant_int8": qb,
          "qwz_quant_replica_int8": qb + 2 * w.n}
    kernels = {n: {"ms": round(per[n], 5), "ms_percentiles": pct[n], "algorithmic_bytes": kb[n],
                   "GB/s": round(kb[n] / (per[n] / 1e3) / 1e9, 1),
                   "frac": round(kb[n] / (per[n] / 1e3) / 1e9 / peak, 4)} for n in kb}
    return {"metric": "qwZ weights/s (int8 quantize + dequantize round trip)",
            "value": w.n * ws / (ms / 1e3), "unit": "weights/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded N(0, 0.02) weights)",
            "config": {"workload": w.name, "n": w.n, "B": w.B,
                       "l2": f"inputs exceed L2 ({w.n * 6 / 1e9:.1f} GB per step)"},
            "roofline": {"bound": "hbm", "kernel": "qwz_quant_int8",
                         "achieved": kernels["qwz_quant_int8"]["GB/s"], "peak": peak,
                         "peak_kind": f"hbm_gbs of {kind}", "unit": "GB/s",
                         "frac": kernels["qwz_quant_int8"]["frac"],
                         "traffic": ncu_traffic("qwz_quant_int8", "qwz", w.n)},
            "kernels": kernels, "gpu_launches": 2 * args.steps, "clocks": clocks}, \
        (wd, codes, scales, back, stream)


def run_sr(w: wl.SrWorkload, args, dev, dist, ws):
    from weight_communication_gb300 import binding
    dst = torch.zeros(w.n, dtype=torch.bfloat16, device=dev)
    pristine = [wl.sr_micro_gradient(w, t, device=dev) for t in range(w.micro_steps)]
    srcs = [p.clone() for p in pristine]
    stream = torch.cuda.Stream(dev)
    names = [f"sr_accumulate[{t}]" for t in range(w.micro_steps)]
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            for t in range(w.micro_steps):
                binding.sr_accumulate_bf16(dst, srcs[t], w.seed, t, stream)
            for s, p in zip(srcs, pristine):
                s.copy_(p)
        torch.cuda.synchronize(dev)
        timer = Timer(names, args.steps)
        sampler = clocks_begin(args, dev)
        barrier(dist)
        t0 = time.time()
        for i in range(args.steps):
            for t in range(w.micro_steps):
                timer.mark(i, t)
                binding.sr_accumulate_bf16(dst, srcs[t], w.seed, t, stream)
            timer.mark(i, w.micro_steps)
            for s, p in zip(srcs, pristine):      # refill the sources, untimed
                s.copy_(p)
        torch.cuda.synchronize(dev)
        t1 = time.time()
        barrier(dist)
    clocks = sampler.stop(t0, t1) if sampler else None
    per = timer.per_kernel_ms()
    launch_pct = percentiles([e[j].elapsed_time(e[j + 1]) for e in timer.ev
                              for j in range(len(timer.names))])
    ms = max_over_ranks(timer.step_sum_ms(), dist, dev)
    peak, kind = measured_peaks()
    b = w.n * 8
    launch_ms = statistics.mean(per.values())
    achieved = b / (launch_ms / 1e3) / 1e9
    return {"metric": "ZeRO-2 SR accumulate elements/s (8 micro-steps, source zeroed)",
            "value": w.n * w.micro_steps * ws / (ms / 1e3), "unit": "elements/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded N(0, 1e-4) micro-gradients)",
            "config": {"workload": w.name, "n": w.n, "micro_steps": w.micro_steps,
                       "l2": "inputs exceed L2 (1 GB per launch)"},
            "roofline": {"bound": "hbm", "kernel": "sr_accumulate", "achieved": round(achieved, 1),
                         "peak": peak, "peak_kind": f"hbm_gbs of {kind}", "unit": "GB/s",
                         "frac": round(achieved / peak, 4),
                         "traffic": ncu_traffic("sr_accumulate", "sr", w.n)},
            "kernels": {"sr_accumulate": {"ms": round(launch_ms, 5), "ms_percentiles": launch_pct,
                                          "algorithmic_bytes": b,
                                          "GB/s": round(achieved, 1),
                                          "frac": round(achieved / peak, 4)}},
            "gpu_launches": w.micro_steps * args.steps, "clocks": clocks}, \
        (dst, srcs, pristine, stream)


# ---------------------------------------------------------------------------
# the other configurations, summarized on the default line
# ---------------------------------------------------------------------------

def qgz_parity_on_sample(w: wl.QgzWorkload, fraction: int, steps: int, dev) -> dict:
    """`steps` chained steps of a 1/fraction sample of w, oracle against the
    CUDA path (every shard and error-buffer element)."""
    import oracle
    orc = oracle.get()
    sw = qgz_sample(w, fraction)
    g = wl.as_u16(wl.qgz_gradients(sw, 0)).ravel().copy()
    ef = np.zeros(sw.R * sw.N, np.float32)
    for _ in range(steps):
        out = oracle_qgz_step(orc, sw, g, ef)
    return gpu_parity_on_sample(sw, g, steps, out, ef, dev)


def variant_parity_on_sample(w: wl.QgzWorkload, variant: str, fraction: int, steps: int,
                             dev) -> dict:
    """`steps` chained steps of a 1/fraction sample of w through one of the
    step's other forms, oracle against the CUDA path: every shard and every
    element of every error buffer the form keeps.
      hier_ef    -- the two-hop step with the first hop's own error buffer
      bf16ef     -- the step with a bf16 error buffer
      int8ef     -- the step with an int8 error buffer and a scale per block
      fused      -- the flat step as one kernel (wc_qgz_step_fused)
      hier_fused -- the two-hop step with its first stage as one kernel
                    (wc_qgz_first_hop_fused), then the second hop
      hier_ef_fused -- the same with the first hop's own error buffer
      bf16ef_fused, int8ef_fused -- the flat fused step with the bf16 or int8
                    error buffer"""
    import oracle
    from weight_communication_gb300 import binding
    from weight_communication_gb300.qgz import QgzReducer
    orc = oracle.get()
    sw = qgz_sample(w, fraction)
    N, R, G, B, s, beta = sw.N, sw.R, sw.G, sw.B, sw.err_scale, sw.err_beta
    g = wl.as_u16(wl.qgz_gradients(sw, 0)).ravel().copy()
    bufs = {}                                     # oracle error buffers by name
    if variant in ("bf16ef", "bf16ef_fused"):
        bufs["ef"] = np.zeros(R * N, np.uint16)
    elif variant in ("int8ef", "int8ef_fused"):
        bufs["ef"] = np.zeros(R * N, np.int8)
        bufs["ef_scales"] = np.zeros(R * N // B, np.float32)
    else:
        bufs["ef"] = np.zeros(R * N, np.float32)
    if variant in ("hier_ef", "hier_ef_fused"):
        bufs["ef1"] = np.zeros(G * N, np.float32)
    for _ in range(steps):
        if variant in ("bf16ef", "bf16ef_fused"):
            codes, scales = orc.ef_quant_int4_bf16ef(g, bufs["ef"], N, R, G, B, s, beta)
        elif variant in ("int8ef", "int8ef_fused"):
            codes, scales = orc.ef_quant_int4_int8ef(g, bufs["ef"], bufs["ef_scales"], N, R, G,
                                                     B, s, beta)
        else:
            codes, scales = orc.ef_quant_int4(g, bufs["ef"], N, R, G, B, s, beta)
        if G > 1:
            codes, scales = orc.dequant_reduce_requant_ef(codes, scales, N, R, G, B,
                                                          bufs.get("ef1"), s, beta)
        want = orc.dequant_reduce(codes, scales, N, R, G, B, 1.0, sw.out_bf16)
    out_dtype = torch.bfloat16 if sw.out_bf16 else torch.float32
    gd = wl.from_u16(g, dev)
    got = {}
    if variant in ("bf16ef_fused", "int8ef_fused"):
        kind = variant[:4]
        ef = torch.zeros(R * N, dtype=EF_DTYPES[kind], device=dev)
        ef_scales = (torch.zeros(R * N // B, dtype=torch.float32, device=dev)
                     if kind == "int8" else None)
        out = torch.empty(N, dtype=out_dtype, device=dev)
        for _ in range(steps):
            binding.qgz_step_fused(gd, ef, None, None, out, N, R, B, s, beta, ef_scales=ef_scales)
        got["ef"] = ef
        if ef_scales is not None:
            got["ef_scales"] = ef_scales
    elif variant in ("fused", "hier_fused", "hier_ef_fused"):
        ef = torch.zeros(R * N, dtype=torch.float32, device=dev)
        ef1 = (torch.zeros(G * N, dtype=torch.float32, device=dev)
               if variant == "hier_ef_fused" else None)
        out = torch.empty(N, dtype=out_dtype, device=dev)
        c1 = torch.empty(G * N // 2, dtype=torch.uint8, device=dev)
        s1 = torch.empty(G * N // B, dtype=torch.float32, device=dev)
        for _ in range(steps):
            if variant == "fused":
                binding.qgz_step_fused(gd, ef, None, None, out, N, R, B, s, beta)
            else:
                binding.qgz_first_hop_fused(gd, ef, None, None, c1, s1, N, R, G, B, s, beta,
                                            ef1=ef1)
                binding.dequant_reduce(c1, s1, out, N, R, G, B)
        got["ef"] = ef
        if ef1 is not None:
            got["ef1"] = ef1
    else:
        ef_dtype = {"bf16ef": torch.bfloat16, "int8ef": torch.int8}.get(variant, torch.float32)
        red = QgzReducer(N, R, G, B, s, beta, out_dtype=out_dtype, device=dev,
                         ef_dtype=ef_dtype, hop1_ef=variant == "hier_ef")
        gv = gd.view(R, N)
        for _ in range(steps):
            red.step(gv)
        out = red.out
        got["ef"] = red.ef
        if variant == "int8ef":
            got["ef_scales"] = red.ef_scales
        if variant == "hier_ef":
            got["ef1"] = red.ef1
    torch.cuda.synchronize(dev)
    same = {"shards": np.array_equal(np.ascontiguousarray(out.cpu().view(torch.uint8).numpy()),
                                     want.view(np.uint8))}
    for name, t in got.items():
        same[name] = np.array_equal(t.cpu().view(torch.uint8).numpy(), bufs[name].view(np.uint8))
    return {"verdict": "bit-exact" if all(same.values()) else "MISMATCH",
            **{k: bool(v) for k, v in same.items()},
            "compared": f"every shard and error-buffer element after {steps} steps of a 1/{fraction} "
                        f"sample (R={R}, N={N}), against the oracle"}


def qwz_parity(w: wl.QwzWorkload, tensors, dev) -> dict:
    """Sampled block ranges (the first and the last 2^20 weights) of the
    full-size qwZ run against the oracle: the one-pass replica kernel's codes,
    scales and bf16 replica, then the dequant kernel's bf16 weights."""
    import oracle
    from weight_communication_gb300 import binding
    orc = oracle.get()
    wd, codes, scales, back, stream = tensors
    m = min(w.n, 1 << 20) // w.B * w.B
    ranges = [(0, m), (w.n - m, w.n)]
    with torch.cuda.stream(stream):
        binding.qwz_quant_replica_int8(wd, codes, scales, back, w.B, stream)
        torch.cuda.synchronize(dev)
        rep = [back[a:b].clone() for a, b in ranges]
        binding.qwz_dequant_int8(codes, scales, back, w.B, stream)
        torch.cuda.synchronize(dev)
    ok = True
    for (a, b), r in zip(ranges, rep):
        wc, ws_, wr = orc.qwz_quant_replica_int8(wl.as_u16(wd[a:b]).copy(), w.B)
        ok &= np.array_equal(codes[a:b].cpu().numpy(), wc)
        ok &= np.array_equal(scales[a // w.B:b // w.B].cpu().numpy().view(np.uint32), ws_.view(np.uint32))
        ok &= np.array_equal(wl.as_u16(r), wr)
        ok &= np.array_equal(wl.as_u16(back[a:b]), orc.qwz_dequant_int8(wc, ws_, w.B))
    return {"verdict": "bit-exact" if ok else "MISMATCH",
            "compared": f"codes, scales, replica and dequantized weights of the first and last "
                        f"{m} weights of the full-size run, against the oracle"}


def sr_parity(w: wl.SrWorkload, tensors, dev) -> dict:
    """One more full-size launch (micro-step 0) from the timed run's state;
    its first 2^22 outputs and zeroed sources against the oracle."""
    import oracle
    from weight_communication_gb300 import binding
    orc = oracle.get()
    dst, srcs, pristine, stream = tensors
    m = min(w.n, 1 << 22)
    with torch.cuda.stream(stream):
        srcs[0].copy_(pristine[0])
        torch.cuda.synchronize(dev)
        d0 = wl.as_u16(dst[:m]).copy()
        s0 = wl.as_u16(srcs[0][:m]).copy()
        binding.sr_accumulate_bf16(dst, srcs[0], w.seed, 0, stream)
        torch.cuda.synchronize(dev)
    orc.sr_accumulate_bf16(d0, s0, w.seed, 0)
    ok = np.array_equal(wl.as_u16(dst[:m]), d0) and np.array_equal(wl.as_u16(srcs[0][:m]), s0)
    return {"verdict": "bit-exact" if ok else "MISMATCH",
            "compared": f"the first {m} outputs and zeroed sources of one full-size launch "
                        f"(seed {w.seed}, micro-step 0), against the oracle"}


def other_workloads(args, dev, dist, ws, rank) -> dict:
    """The hierarchical two-hop step, qwZ and the SR accumulate at full size,
    plus the single-hop step's low-precision error buffers and fused form:
    per kernel the mean and median event time, algorithmic bytes and fraction
    of the HBM peak, over at most 20 timed steps each.  With the CPU legs on
    (rank 0 of a single process), every entry also carries a parity verdict
    from a sample through the CUDA path against the oracle."""
    sub = argparse.Namespace(**vars(args))
    sub.steps = max(1, min(args.steps, 20))
    sub.warmup = 3
    sub.no_e2e = True
    sub.no_overlap = True
    check = rank == 0 and ws == 1 and not args.no_cpu_baseline

    def entry(line, parity=None):
        e = {"workload": line["config"]["workload"], "steps": sub.steps,
             "ms_per_step": round(line["ms_per_step"], 5), "kernels": line["kernels"],
             "clocks": line["clocks"]}
        if parity is not None:
            e["parity"] = parity
        return e

    out = {}
    line, _ = run_qgz(wl.QGZ_HIERARCHICAL, sub, dev, dist, ws)
    out["qgz_hierarchical"] = entry(
        line, qgz_parity_on_sample(wl.QGZ_HIERARCHICAL, 64, 2, dev) if check else None)
    torch.cuda.empty_cache()
    for name, variant, runner, w in (
            ("qgz_hier_ef", "hier_ef", lambda w: run_qgz(w, sub, dev, dist, ws, hop1_ef=True),
             wl.QGZ_HIERARCHICAL),
            ("qgz_hier_fused", "hier_fused", lambda w: run_qgz_hier_fused(w, sub, dev, dist, ws),
             wl.QGZ_HIERARCHICAL),
            ("qgz_hier_ef_fused", "hier_ef_fused",
             lambda w: run_qgz_hier_fused(w, sub, dev, dist, ws, hop1_ef=True),
             wl.QGZ_HIERARCHICAL),
            ("qgz_bf16ef", "bf16ef", lambda w: run_qgz(w, sub, dev, dist, ws, ef="bf16"),
             wl.QGZ_SINGLE_HOP),
            ("qgz_int8ef", "int8ef", lambda w: run_qgz(w, sub, dev, dist, ws, ef="int8"),
             wl.QGZ_SINGLE_HOP),
            ("qgz_fused", "fused", lambda w: run_qgz_fused(w, sub, dev, dist, ws),
             wl.QGZ_SINGLE_HOP),
            ("qgz_bf16ef_fused", "bf16ef_fused",
             lambda w: run_qgz_fused(w, sub, dev, dist, ws, ef_kind="bf16"), wl.QGZ_SINGLE_HOP),
            ("qgz_int8ef_fused", "int8ef_fused",
             lambda w: run_qgz_fused(w, sub, dev, dist, ws, ef_kind="int8"), wl.QGZ_SINGLE_HOP)):
        line, _ = runner(w)
        torch.cuda.empty_cache()
        out[name] = entry(line, variant_parity_on_sample(w, variant, 64, 2, dev) if check else None)
    line, t = run_qwz(wl.QWZ_WEIGHTS, sub, dev, dist, ws)
    out["qwz"] = entry(line, qwz_parity(wl.QWZ_WEIGHTS, t, dev) if check else None)
    del t
    torch.cuda.empty_cache()
    line, t = run_sr(wl.SR_ACCUMULATE, sub, dev, dist, ws)
    out["sr"] = entry(line, sr_parity(wl.SR_ACCUMULATE, t, dev) if check else None)
    del t
    torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------------------
# CPU oracle legs
# ---------------------------------------------------------------------------

def qgz_sample(w: wl.QgzWorkload, fraction: int) -> wl.QgzWorkload:
    """The workload with each rank's gradient cut to N/fraction elements
    (same R, G, B, error-feedback parameters and value distribution)."""
    unit = w.R * w.B
    n = max(unit, (w.N // fraction) // unit * unit)
    return w.scaled(n, f"{w.name.split()[0]} sample R={w.R} N={n} B={w.B}")


def oracle_qgz_step(orc, w: wl.QgzWorkload, g_u16: np.ndarray, ef: np.ndarray):
    codes, scales = orc.ef_quant_int4(g_u16, ef, w.N, w.R, w.G, w.B, w.err_scale, w.err_beta)
    if w.G > 1:
        c1, s1 = orc.dequant_reduce_requant(codes, scales, w.N, w.R, w.G, w.B)
        return orc.dequant_reduce(c1, s1, w.N, w.R, w.G, w.B, 1.0, w.out_bf16)
    return orc.dequant_reduce(codes, scales, w.N, w.R, 1, w.B, 1.0, w.out_bf16)


def oracle_qgz_step_threaded(orc, w: wl.QgzWorkload, g_u16: np.ndarray, ef: np.ndarray, pool,
                             pieces: int = 1):
    """The same step with the oracle's independent pieces run on a thread
    pool (the oracle's C calls release the interpreter lock):
      * quantization by (rank, slice): every block lies in one slice, so a
        slice is quantized as a one-rank problem of S elements and its codes
        and scales are placed at the slice's send position;
      * the first hop by unit;
      * each destination's reduce in `pieces` block-aligned output ranges
        (every output is its own sum)."""
    N, R, G, B = w.N, w.R, w.G, w.B
    S = N // R
    codes = np.empty(R * N // 2, np.uint8)
    scales = np.empty(R * N // B, np.float32)

    def quant(item):
        r, k = divmod(item, R)
        x0 = r * N + k * S
        c, sc = orc.ef_quant_int4_rank(g_u16[x0:x0 + S], ef[x0:x0 + S], S, 1, 1, B,
                                       w.err_scale, w.err_beta)
        y0 = r * N + orc.send_position(k, R, G) * S
        codes[y0 // 2:(y0 + S) // 2] = c
        scales[y0 // B:(y0 + S) // B] = sc

    list(pool.map(quant, range(R * R)))
    if G > 1:
        L = R // G
        units = list(pool.map(lambda u: orc.dequant_reduce_requant_unit(
            codes, scales, N, R, G, B, u // L, u % L), range(R)))
        codes = np.concatenate([u[0] for u in units])
        scales = np.concatenate([u[1] for u in units])
    out = np.empty(N, np.uint16 if w.out_bf16 else np.float32)
    blocks = S // B
    bounds = [B * (blocks * j // pieces) for j in range(pieces + 1)]

    def reduce(item):
        k, j = divmod(item, pieces)
        i0, i1 = bounds[j], bounds[j + 1]
        out[k * S + i0:k * S + i1] = orc.dequant_reduce_dest_range(
            codes, scales, N, R, G, B, k, i0, i1, 1.0, w.out_bf16)

    list(pool.map(reduce, range(R * pieces)))
    return out


def cpu_baseline_qgz_threaded(w: wl.QgzWorkload, steps: int, fraction: int, g_u16: np.ndarray):
    """The oracle on all host cores: the pieces of oracle_qgz_step_threaded
    spread over one thread per core."""
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    orc = oracle.get()
    sw = qgz_sample(w, fraction)
    cores, _ = host_cpu()
    threads = max(1, cores)
    pieces = max(1, -(-2 * threads // sw.R))  # at least two reduce pieces per thread
    ef = np.zeros(sw.R * sw.N, np.float32)
    with ThreadPoolExecutor(threads) as pool:
        t0 = time.perf_counter()
        for _ in range(steps):
            oracle_qgz_step_threaded(orc, sw, g_u16, ef, pool, pieces)
        dt = time.perf_counter() - t0
    return {"value": sw.R * sw.N * steps / dt, "unit": "elements/s", "cores": threads,
            "kind": "oracle",
            "sample": f"the same {steps} steps, {dt:.1f} s on {threads} threads "
                      f"(quantization by rank and slice, first hop by unit, each "
                      f"destination's reduce in {pieces} ranges)"}


def gpu_parity_on_sample(sw: wl.QgzWorkload, g_u16: np.ndarray, steps: int,
                         want_out: np.ndarray, want_ef: np.ndarray, dev) -> dict:
    """The CUDA path on the CPU baseline's sample: the same steps on the same
    bytes, its last shards and error buffers compared bit for bit with the
    oracle's."""
    from weight_communication_gb300.qgz import QgzReducer
    red = QgzReducer(sw.N, sw.R, sw.G, sw.B, sw.err_scale, sw.err_beta,
                     out_dtype=torch.bfloat16 if sw.out_bf16 else torch.float32, device=dev)
    gd = wl.from_u16(g_u16, dev).view(sw.R, sw.N)
    for _ in range(steps):
        red.step(gd)
    torch.cuda.synchronize(dev)
    out = wl.as_u16(red.out) if sw.out_bf16 else red.out.cpu().numpy()
    same_out = np.array_equal(np.ascontiguousarray(out).view(np.uint8), want_out.view(np.uint8))
    same_ef = np.array_equal(red.ef.cpu().numpy().view(np.uint32), want_ef.view(np.uint32))
    return {"verdict": "bit-exact" if (same_out and same_ef) else "MISMATCH",
            "shards": bool(same_out), "error_buffers": bool(same_ef),
            "compared": f"every shard and error-buffer element after {steps} steps of the "
                        f"CPU baseline's sample (R={sw.R}, N={sw.N}), against the oracle"}


def cpu_baseline_qgz(w: wl.QgzWorkload, steps: int, fraction: int, g_full_example=None,
                     dev=None):
    """The oracle, as it stands, timed on this host on a bounded sample; with
    dev, the CUDA path also runs the sample and its result is compared with
    the oracle's ("parity" entry)."""
    import oracle
    orc = oracle.get()
    sw = qgz_sample(w, fraction)
    if g_full_example is not None:
        g = wl.as_u16(g_full_example[:, :sw.N]).ravel().copy()
    else:
        g = wl.as_u16(wl.qgz_gradients(sw, 0)).ravel().copy()
    ef = np.zeros(sw.R * sw.N, np.float32)
    t0 = time.perf_counter()
    for _ in range(steps):
        out = oracle_qgz_step(orc, sw, g, ef)
    dt = time.perf_counter() - t0
    cores, model = host_cpu()
    res = {"value": sw.R * sw.N * steps / dt, "unit": "elements/s", "cores": 1,
           "host_cores": cores, "cpu": model, "kind": "oracle",
           "sample": f"{steps} steps of R={sw.R} ranks x N={sw.N} elements "
                     f"(1/{fraction} of each rank's gradient; same B, G, LoCo parameters), "
                     f"{dt:.1f} s single-threaded",
           "all_cores": cpu_baseline_qgz_threaded(w, steps, fraction, g)}
    if dev is not None:
        res["parity"] = gpu_parity_on_sample(sw, g, steps, out, ef, dev)
    return res


def run_reference(w_name: str, args, ws, rank):
    """--impl reference: the CPU oracle on the same metric and config."""
    if ws > 1 and rank != 0:
        return None
    import oracle
    orc = oracle.get()
    w = wl.QGZ_WORKLOADS.get(w_name)
    if w is None:
        return {"impl": "reference", "unavailable": f"no oracle leg for workload {w_name}"}
    # Each step is a bounded sample of the workload, sized so that all
    # warm-up and timed steps take about REFERENCE_BUDGET_S of oracle work
    # (never more than the fixed fraction below).
    fraction = {"qgz_tiny": 1, "qgz_single_hop": 4, "qgz_hierarchical": 32}[w_name]
    per_step = REFERENCE_BUDGET_S * ORACLE_ELEMENTS_PER_S / max(1, args.steps + args.warmup)
    fraction = max(fraction, math.ceil(w.R * w.N / per_step))
    sw = qgz_sample(w, fraction)
    batches = [wl.as_u16(wl.qgz_gradients(sw, t)).ravel().copy() for t in range(2)]
    ef = np.zeros(sw.R * sw.N, np.float32)
    for i in range(args.warmup):
        oracle_qgz_step(orc, sw, batches[i % 2], ef)
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle_qgz_step(orc, sw, batches[i % 2], ef)
    dt = time.perf_counter() - t0
    ms = dt * 1e3 / args.steps
    value = sw.R * sw.N / (ms / 1e3)
    cores, model = host_cpu()
    sample = (f"each step R={sw.R} ranks x N={sw.N} elements (1/{fraction} of each rank's "
              f"gradient of {w.name}; same B, G, LoCo parameters)")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "elements/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded normal gradients with sparse outliers)",
            "config": {"workload": w.name, "R": w.R, "N": w.N, "G": w.G, "B": w.B,
                       "err_scale": w.err_scale, "err_beta": w.err_beta,
                       "parallelism": "single host thread"},
            "cpu_baseline": {"value": value, "unit": "elements/s", "cores": 1,
                             "host_cores": cores, "cpu": model, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "elements/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


# ---------------------------------------------------------------------------

def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="qgz_single_hop",
                    choices=["qgz_single_hop", "qgz_fused", "qgz_bf16ef", "qgz_int8ef",
                             "qgz_hier_ef", "qgz_hier_fused", "qgz_hier_ef_fused",
                             "qgz_bf16ef_fused", "qgz_int8ef_fused", "qgz_tiny",
                             "qgz_hierarchical", "qwz", "sr", "all"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-overlap", action="store_true",
                    help="skip the extra pass that overlaps each reduce with the next EF-quant")
    ap.add_argument("--no-clocks", dest="clocks", action="store_false")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the summary of the other configurations on the default line")
    ap.add_argument("--scale", type=int, default=1,
                    help="divide each rank's gradient by this (profiling a smaller case)")
    ap.add_argument("--batches", type=int, default=4,
                    help="distinct gradient batches cycled through the timed steps")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3                       # at least 3 untimed warm-up steps
    ws, rank, local = dist_env()

    if args.impl == "reference":
        line = run_reference(args.workload if args.workload in wl.QGZ_WORKLOADS
                             else "qgz_single_hop", args, ws, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return 0

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the kernels have no CPU path)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from weight_communication_gb300 import binding
    binding.load()                            # fail loudly if the library is missing
    dist = init_dist(ws, True)
    names = (["qgz_single_hop", "qgz_fused", "qgz_bf16ef", "qgz_int8ef", "qgz_tiny",
              "qgz_hierarchical", "qgz_hier_ef", "qgz_hier_fused", "qgz_hier_ef_fused",
              "qgz_bf16ef_fused", "qgz_int8ef_fused", "qwz", "sr"]
             if args.workload == "all" else [args.workload])
    for name in names:
        if name == "qgz_hier_ef":
            w = wl.QGZ_HIERARCHICAL if args.scale == 1 else qgz_sample(wl.QGZ_HIERARCHICAL, args.scale)
            line, _ = run_qgz(w, args, dev, dist, ws, hop1_ef=True)
        elif name in ("qgz_bf16ef", "qgz_int8ef"):
            w = wl.QGZ_SINGLE_HOP if args.scale == 1 else qgz_sample(wl.QGZ_SINGLE_HOP, args.scale)
            line, _ = run_qgz(w, args, dev, dist, ws, ef=name[4:8])
        elif name in ("qgz_fused", "qgz_bf16ef_fused", "qgz_int8ef_fused"):
            w = wl.QGZ_SINGLE_HOP if args.scale == 1 else qgz_sample(wl.QGZ_SINGLE_HOP, args.scale)
            line, _ = run_qgz_fused(w, args, dev, dist, ws,
                                    ef_kind={"qgz_fused": "fp32", "qgz_bf16ef_fused": "bf16",
                                             "qgz_int8ef_fused": "int8"}[name])
        elif name in ("qgz_hier_fused", "qgz_hier_ef_fused"):
            w = (wl.QGZ_HIERARCHICAL if args.scale == 1
                 else qgz_sample(wl.QGZ_HIERARCHICAL, args.scale))
            line, _ = run_qgz_hier_fused(w, args, dev, dist, ws,
                                         hop1_ef=name == "qgz_hier_ef_fused")
        elif name in wl.QGZ_WORKLOADS:
            w = wl.QGZ_WORKLOADS[name]
            if args.scale > 1:
                w = qgz_sample(w, args.scale)
            line, g_example = run_qgz(w, args, dev, dist, ws)
            if rank == 0 and ws == 1 and not args.no_cpu_baseline:
                fraction = {"qgz_tiny": 1, "qgz_single_hop": 4, "qgz_hierarchical": 32}[name]
                # about 12 s of single-threaded oracle work on the sample
                line["cpu_baseline"] = cpu_baseline_qgz(w, 20, fraction, g_example.cpu(), dev)
                line["parity"] = line["cpu_baseline"].pop("parity")
            del g_example
            if name == "qgz_single_hop" and args.scale == 1 and not args.no_workloads:
                torch.cuda.empty_cache()
                line["workloads"] = other_workloads(args, dev, dist, ws, rank)
        elif name == "qwz":
            qw = wl.QWZ_WEIGHTS
            if args.scale > 1:
                n = max(qw.B, (qw.n // args.scale) // qw.B * qw.B)
                qw = dataclasses.replace(qw, n=n, name=f"qwz sample n={n} B={qw.B}")
            line, _ = run_qwz(qw, args, dev, dist, ws)
        else:
            sw = wl.SR_ACCUMULATE
            if args.scale > 1:
                n = max(8, (sw.n // args.scale) // 8 * 8)
                sw = dataclasses.replace(sw, n=n, name=f"sr_accumulate sample n={n} x{sw.micro_steps}")
            line, _ = run_sr(sw, args, dev, dist, ws)
        if rank == 0:
            print(json.dumps(line), flush=True)
        torch.cuda.empty_cache()
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
