#!/usr/bin/env python
"""Benchmark: fused forward + full VJP of ragged GQA attention on GB300.

One step = one library call (schedule, forward, preprocess, dk/dv, dq) over
the long balanced workload: 24 sequences with Lq = Lk ~ U[6144, 12288],
Hq = 96 query heads sharing one K/V head, head_dim 160, bf16, token-strided
(step 2) views, ALiBi slopes 2^(-8h/96).  Throughput counts 4 Lq Lk d
forward and 10 Lq Lk d backward flops per head (TFLOP/s); latency is
ms_per_step.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the fp64 CPU oracle
on a bounded sample of the same workload instead.  The end-to-end leg runs
the same call through the host-buffer entry point (``--e2e-chunks``).

Variants of the workload (each a separate line, named in config.workload):
``--causal`` / ``--window-left`` / ``--window-right`` (flops counted over the
admissible pairs only), ``--hkv`` (K/V heads), ``--head-dim`` (128 or 64),
``--dropout RATE``, ``--length-scale`` (small cases for profiling).
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
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from ragged_gqa_attention_varlen_gb300 import workloads  # noqa: E402

METRIC = "fwd+full-VJP TFLOP/s & latency (d=160, Hq 48-96, Hkv=1), % of GB300 tensor peak"
UNIT = "TFLOP/s"
HEAD_DIM = 160


def scored_pairs(p) -> int:
    """(query, key) pairs the mask admits, summed over sequences: Lq Lk
    without a mask.  Key j is admissible for query i when
    i + Lk - Lq - wl <= j <= i + Lk - Lq + wr (causal: wr = 0; a negative
    window is unbounded)."""
    import numpy as np

    if not (p.causal or p.window_left >= 0 or p.window_right >= 0):
        return p.sum_lq_lk()
    wr = 0 if p.causal else p.window_right
    total = 0
    for lq, lk in zip(*p.lengths()):
        k0 = np.arange(lq, dtype=np.int64) + (lk - lq)
        lo = np.maximum(0, k0 - p.window_left) if p.window_left >= 0 else np.zeros_like(k0)
        hi = np.minimum(lk - 1, k0 + wr) if wr >= 0 else np.full_like(k0, lk - 1)
        total += int(np.clip(hi - lo + 1, 0, None).sum())
    return total


def counted_flops(p) -> float:
    """4 d (forward) + 10 d (backward) per admissible (query, key) pair and
    query head: 14 Lq Lk d per head without a mask."""
    return 14.0 * p.q.shape[-1] * p.Hq * scored_pairs(p)


def kernel_flops(p) -> dict:
    """Algorithmic flops each kernel contributes to the counted total: the
    forward's two matmuls (4d), dk/dv's four (S^T, dP^T, dV, dK: 8d) and dq's
    dQ = dS K (2d); dq's recompute of S and dP is not counted."""
    u = p.q.shape[-1] * p.Hq * scored_pairs(p)
    return {"forward": 4 * u, "dkdv": 8 * u, "dq": 2 * u, "schedule": 0.0, "preprocess": 0.0}


# Transcendental (MUFU) operations per (head, query, key) unit in each kernel:
# the forward, dk/dv and dq each take one tanh (softcap) and one exp2 (P)
# per element; without a softcap there is no tanh.  Issue rates measured on
# this GPU with one CTA of eight elementwise warps per SM (tanh.approx.f32 16,
# ex2.approx 32 per clock per SM).
MUFU_RATE = {"tanh": 16.0, "ex2": 32.0}


def mufu_bound(p, call_ms, kernel_ms, sm_mhz, sms):
    """Time the MUFU alone needs for the call's transcendentals at the
    measured issue rates and the sampled SM clock, next to the measured
    times: the co-bound of the tensor-core roofline."""
    units = p.Hq * scored_pairs(p)
    per = {"tanh": 1.0 if p.softcap > 0 else 0.0, "ex2": 1.0}
    clk_per_unit = sum(per[k] / MUFU_RATE[k] for k in per)  # SM clocks per unit per kernel
    mhz = sm_mhz or 2070.0
    one_kernel_ms = units * clk_per_unit / sms / (mhz * 1e6) * 1e3
    out = {"ops_per_unit_per_kernel": per, "rate_per_clk_per_sm": MUFU_RATE,
           "rate_source": "measured issue rate (probe, 8 warps per SM)", "sms": sms,
           "sm_mhz": mhz, "units": units, "bound_ms": 3 * one_kernel_ms, "call_ms": call_ms,
           "frac": 3 * one_kernel_ms / call_ms}
    if kernel_ms:
        out["per_kernel"] = {k: {"bound_ms": one_kernel_ms, "kernel_ms": kernel_ms[k],
                                 "frac": one_kernel_ms / kernel_ms[k]}
                             for k in ("forward", "dkdv", "dq") if k in kernel_ms}
    return out


def mask_name(p) -> str:
    """Suffix naming the mask of a workload ('' without one)."""
    parts = []
    if p.causal:
        parts.append("causal")
    if p.window_left >= 0 or p.window_right >= 0:
        parts.append(f"window ({p.window_left}, {p.window_right})")
    return (", " + " + ".join(parts)) if parts else ""


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        try:
            bus = torch.cuda.get_device_properties(device_index).pci_bus_id
        except Exception:
            bus = None
        self.target = bus

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "200"]
            if self.target:
                cmd += ["-i", self.target]
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"),
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------- distributed plumbing

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


def max_over_ranks(x: float, world: int) -> float:
    """Largest value of x over all ranks (timing only; no data path)."""
    if world == 1:
        return x
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(flops_per_rank: float, seconds_per_rank: float, steps: int, world: int):
    """Whole-job throughput: all ranks' counted flops over the slowest rank's
    time.  Returns (TFLOP/s, ms per step)."""
    t = max_over_ranks(seconds_per_rank, world)
    return flops_per_rank * steps * world / t / 1e12, t / steps * 1e3


# ---------------------------------------------------------------- CPU oracle

def oracle_sample(seconds: float, seed: int = 5):
    """Time the fp64 oracle on whole sequences of the long balanced workload
    scaled to 1/8 of its lengths (same structure, heads, slopes), one sequence
    after another until ``seconds`` pass.  Returns (TFLOP/s, threads, text)."""
    import oracle

    oracle.build()
    p = workloads.long_balanced(seed=seed, length_scale=0.125)
    lq, lk = p.lengths()
    flops, t0, done, nthreads = 0.0, time.perf_counter(), 0, 0
    for b in range(p.B):
        r = oracle.fvjp(p, seq_sel=[b])
        nthreads = r["threads"]
        flops += 14.0 * HEAD_DIM * p.Hq * lq[b] * lk[b]
        done += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    text = (f"oracle fvjp (fp64, all outputs) on {done} whole sequence(s) of the long balanced "
            f"workload at 1/8 length (Lq=Lk={lq[0]}..), Hq={p.Hq}; {dt:.1f} s")
    return flops / dt / 1e12, nthreads, text, dt


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    import oracle

    oracle.build()
    p = workloads.long_balanced(seed=5, length_scale=0.1)
    lq, lk = p.lengths()
    b = min(range(p.B), key=lambda i: lq[i] * lk[i])  # shortest sequence: bounded step
    flops = 14.0 * HEAD_DIM * p.Hq * lq[b] * lk[b]
    for _ in range(args.warmup):
        oracle.fvjp(p, seq_sel=[b])
    times = []
    nthreads = 0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        r = oracle.fvjp(p, seq_sel=[b])
        times.append(time.perf_counter() - t0)
        nthreads = r["threads"]
    sec = sum(times) / len(times)
    value = flops / sec / 1e12
    sample = (f"one step = oracle fvjp (fp64) of sequence {b} of the long balanced workload at "
              f"1/10 length (Lq=Lk={lq[b]}, Hq={p.Hq})")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "long_balanced", "sample": "1/10 length, one sequence"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": nthreads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU arm

def dram_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` on the long balanced workload, from
    the committed ncu capture in profiles/, or None when the capture does not
    apply to the kernel as built now (its source file changed since)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic_long_balanced.json")
    try:
        with open(path) as f:
            rec = json.load(f)["kernels"][kernel]
        with open(os.path.join(ROOT, rec["source"]), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != rec["sha256"]:
                return None
        return rec["dram_read_bytes"] + rec["dram_write_bytes"]
    except (OSError, KeyError, ValueError):
        return None


def run_gpu(args, world, rank, local):
    from ragged_gqa_attention_varlen_gb300 import _build, binding

    _build.build()
    binding.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    p = workloads.long_balanced(seed=5 + rank, device=dev, poison=False,
                                length_scale=args.length_scale, Hkv=args.hkv, d=args.head_dim)
    p.causal, p.window_left, p.window_right = args.causal, args.window_left, args.window_right
    drop = {} if args.dropout is None else dict(dropout_seed=1234, dropout_rate=args.dropout)
    if drop and not args.dropout_regen:  # keep bits stored by the forward, read by the backward
        drop["keep_mask"] = torch.empty(binding.dropout_mask_bytes(p.cu_q, p.cu_k, p.Hq, args.hkv),
                                        dtype=torch.uint8, device=dev)
    flops = counted_flops(p)
    kflops = kernel_flops(p)
    out = torch.empty(p.q.shape, dtype=p.q.dtype, device=dev)
    dq = torch.empty(p.q.shape, dtype=p.q.dtype, device=dev)
    dk = torch.empty(p.k.shape, dtype=p.k.dtype, device=dev)
    dv = torch.empty(p.v.shape, dtype=p.v.dtype, device=dev)
    lse = torch.empty((p.total_q, p.Hq), dtype=torch.float32, device=dev)
    ws = torch.empty(binding.workspace_size(p.B, p.Hq, p.total_q, p.total_k), dtype=torch.uint8,
                     device=dev)
    stream = torch.cuda.current_stream(dev)
    kw = dict(out=out, dq=dq, dk=dk, dv=dv, lse=lse, workspace=ws, stream=stream)

    def call():
        binding.attention_varlen_fvjp(p.q, p.k, p.v, p.cu_q, p.cu_k, p.alibi_slopes, p.dout,
                                      p.causal, p.window_left, p.window_right, p.softcap,
                                      p.scale_multiplier, **kw, **drop)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    status = binding.device_status(ws)
    if status != 0:
        raise RuntimeError(f"device status {status:#x}")

    # ---- device-resident timing, per-kernel events on the launching stream
    nk = len(binding.KERNELS)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)] for _ in range(args.steps)]
    for row in ev:  # torch creates the CUDA event at its first record
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    start.record(stream)
    for s in range(args.steps):
        call()
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    total_s = start.elapsed_time(end) / 1e3
    status = binding.device_status(ws)
    if status != 0:
        raise RuntimeError(f"device status {status:#x}")
    value, ms = aggregate(flops, total_s, args.steps, world)
    launches = binding.launch_count(p.B, p.Hq, p.total_q, p.total_k, Hkv=args.hkv) * args.steps
    if "keep_mask" in drop:  # the mask kernel, once per call
        launches += args.steps
    pk, kind = peaks()
    peak = pk.get("bf16_tflops_sustained", pk["bf16_tflops"])
    if args.hkv == 1:
        # per-kernel split from separate calls with an event between every two
        # kernels (the events keep dq from overlapping the tail of dk/dv, so
        # the timed calls above carry none)
        for s in range(args.steps):
            binding.record_events_next_call(ev[s])
            call()
        torch.cuda.synchronize()
        per_kernel = {name: sum(ev[s][i].elapsed_time(ev[s][i + 1]) for s in range(args.steps)) /
                      args.steps for i, name in enumerate(binding.KERNELS)}
        # ---- roofline of the dominant kernel
        dom = max(per_kernel, key=per_kernel.get)
        achieved = kflops[dom] / (per_kernel[dom] / 1e3) / 1e12
        roofline = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak,
                    "unit": "TFLOP/s", "frac": achieved / peak,
                    "traffic": dram_traffic(dom) if (args.length_scale == 1.0 and not mask_name(p)
                                                     and args.head_dim == HEAD_DIM
                                                     and args.dropout is None) else None,
                    "peak_kind": f"{kind} bf16 sustained"}
    else:
        # one call runs a forward, dk/dv and dq per K/V head group: the
        # roofline is that of the whole call (executed MMA flops: 4d + 8d + 6d)
        per_kernel = None
        achieved = 18.0 / 14.0 * flops / (total_s / args.steps) / 1e12
        roofline = {"bound": "tensor", "kernel": "whole call", "achieved": achieved,
                    "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak, "traffic": None,
                    "peak_kind": f"{kind} bf16 sustained"}
    whole_frac = value / world / pk["bf16_tflops"]

    # ---- end to end: pinned host inputs in, results out, every step
    e2e = None
    if not args.no_e2e and args.dropout is None:
        e2e = run_e2e(args, p, kw, flops, stream, world)

    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mufu = mufu_bound(p, ms, per_kernel, clk.get("sm_mhz"), sms)
    executed = None
    if per_kernel:  # executed MMA flops per kernel (dq's recompute included)
        u = p.q.shape[-1] * p.Hq * scored_pairs(p)
        executed = {k: {"tflops": f * u / (per_kernel[k] / 1e3) / 1e12, "ms": per_kernel[k]}
                    for k, f in (("forward", 4), ("dkdv", 8), ("dq", 6))}
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded, generated on device)",
            "config": {"workload": "long_balanced" + (
                           "" if args.length_scale == 1.0 else f" x{args.length_scale} length") +
                           mask_name(p) + ("" if args.hkv == 1 else f", Hkv={args.hkv}") +
                           ("" if args.head_dim == HEAD_DIM else f", d={args.head_dim}") +
                           ("" if args.dropout is None else f", dropout {args.dropout}" + (
                               " (keep bits regenerated)" if args.dropout_regen else
                               " (keep bits stored)")),
                       "B": p.B, "Hq": p.Hq, "Hkv": args.hkv,
                       "head_dim": args.head_dim, "token_step": 2, "total_q": p.total_q,
                       "total_k": p.total_k, "sum_lq_lk": p.sum_lq_lk(),
                       "scored_pairs": scored_pairs(p),
                       "counted_tflop_per_step": flops / 1e12,
                       "l2": "inputs larger than L2 (q view alone is "
                             f"{p.q.numel() * 2 / 1e9:.1f} GB)"},
            "latency_ms": ms, "frac_of_bf16_peak": whole_frac,
            "kernel_ms": per_kernel, "executed_mma": executed, "roofline": roofline,
            "mufu": mufu, "gpu_launches": launches, "clocks": clk, "e2e": e2e}
    if (rank == 0 and world == 1 and not args.no_cpu and not mask_name(p) and args.hkv == 1
            and args.head_dim == HEAD_DIM and args.dropout is None):
        v, cores, sample, _ = oracle_sample(args.cpu_seconds)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": sample,
                                "extrapolated_full_s": flops / (v * 1e12),
                                "extrapolated_note": "the full workload's counted flops at "
                                                     "the sample's rate (extrapolation, not "
                                                     "a run)"}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_shard(args, world, rank, local):
    """Strong scaling of ONE batch over the ranks with the library's shard
    plan: every rank builds the same long balanced batch, takes its share
    (whole sequences, longest processing time first; head parts of a
    dominant sequence), and a step is the share's calls plus the exchange of
    partial dk/dv (point-to-point to the rank holding part 0, then the
    library's fixed-order sum).  Gathering a rank's sequences into its own
    packed copy happens once, before timing."""
    from ragged_gqa_attention_varlen_gb300 import _build, binding, shard

    _build.build()
    binding.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    p = workloads.long_balanced(seed=5, device=dev, poison=False,
                                length_scale=args.length_scale, Hkv=args.hkv, d=args.head_dim)
    p.causal, p.window_left, p.window_right = args.causal, args.window_left, args.window_right
    flops = counted_flops(p)
    plan = shard.make_plan(p, world)
    mine = shard.shares(p, plan, rank)
    stream = torch.cuda.current_stream(dev)
    bufs = []
    for s_ in mine:
        q = s_.problem
        bufs.append(dict(out=torch.empty(q.q.shape, dtype=q.q.dtype, device=dev),
                         dq=torch.empty(q.q.shape, dtype=q.q.dtype, device=dev),
                         dk=torch.empty(q.k.shape, dtype=q.k.dtype, device=dev),
                         dv=torch.empty(q.v.shape, dtype=q.v.dtype, device=dev),
                         lse=torch.empty((q.total_q, q.Hq), dtype=torch.float32, device=dev),
                         workspace=torch.empty(binding.workspace_size(q.B, q.Hq, q.total_q,
                                                                      q.total_k),
                                               dtype=torch.uint8, device=dev),
                         stream=stream))
    dist = None
    if world > 1:
        import torch.distributed as dist

    def reduce(parts):
        out = torch.empty_like(parts[0])
        binding.sum_partials(parts, out, stream=stream)
        return out

    def step():
        results = []
        for s_, kw in zip(mine, bufs):
            q = s_.problem
            results.append(binding.attention_varlen_fvjp(
                q.q, q.k, q.v, q.cu_q, q.cu_k, q.alibi_slopes, q.dout, q.causal, q.window_left,
                q.window_right, q.softcap, q.scale_multiplier, **kw))
        return shard.exchange(p, plan, rank, mine, results, reduce, dist)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    for kw in bufs:
        st = binding.device_status(kw["workspace"])
        if st != 0:
            raise RuntimeError(f"device status {st:#x}")
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(args.steps):
        step()
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    t = max_over_ranks(start.elapsed_time(end) / 1e3, world)
    value, ms = flops * args.steps / t / 1e12, t / args.steps * 1e3
    pk, kind = peaks()
    launches = sum(binding.launch_count(s_.problem.B, s_.problem.Hq, s_.problem.total_q,
                                        s_.problem.total_k, Hkv=s_.problem.k.shape[1])
                   for s_ in mine) * args.steps
    mean = sum(plan.work) / max(len(plan.work), 1)
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded, generated on device)",
            "config": {"workload": f"long_balanced, one batch sharded over {world} rank(s)" +
                                   mask_name(p), "B": p.B, "Hq": p.Hq, "Hkv": args.hkv,
                       "head_dim": args.head_dim, "units": len(plan.units),
                       "cut_sequences": sum(1 for b in range(p.B) if len(plan.parts(b)) > 1),
                       "rank_work_max_over_mean": max(plan.work) / mean if mean else None,
                       "counted_tflop_per_step": flops / 1e12,
                       "l2": "inputs larger than L2"},
            "latency_ms": ms, "frac_of_bf16_peak": value / world / pk["bf16_tflops"],
            "gpu_launches": launches, "clocks": clk}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_gated(args, world, rank, local):
    """The sigmoid-gated variant on its own training-shape workload (8 causal
    sequences, Lq = Lk ~ U[1024, 16384], Hq 32 over 8 K/V heads, bf16, head
    size 128 and gate width 64 by default).  Counted flops per admissible
    (query, key) pair and head: 4d + 2R forward (S, W V, gate logits) and
    10d + 4R backward (the ungated 10d plus dq_g and dk_g); the roofline is
    the whole call's executed MMA flops (18d + 10R: dq recomputes S, dP and
    the gate logits, dk/dv recomputes S^T, dP^T and the gate logits) over its
    time."""
    from ragged_gqa_attention_varlen_gb300 import _build, binding

    _build.build()
    binding.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    d = 128 if args.head_dim == HEAD_DIM else args.head_dim
    R = args.gate_dim
    p = workloads.gated(seed=6 + rank, device=dev, poison=False, length_scale=args.length_scale,
                        d=d, R=R)
    pairs = scored_pairs(p)
    flops = (14.0 * d + 6.0 * R) * p.Hq * pairs
    executed = (18.0 * d + 10.0 * R) * p.Hq * pairs
    kw = dict(out=torch.empty(p.q.shape, dtype=p.q.dtype, device=dev),
              dq=torch.empty(p.q.shape, dtype=p.q.dtype, device=dev),
              dk=torch.empty(p.k.shape, dtype=p.k.dtype, device=dev),
              dv=torch.empty(p.v.shape, dtype=p.v.dtype, device=dev),
              dq_gate=torch.empty(p.q_gate.shape, dtype=p.q.dtype, device=dev),
              dk_gate=torch.empty(p.k_gate.shape, dtype=p.q.dtype, device=dev),
              lse=torch.empty((p.total_q, p.Hq), dtype=torch.float32, device=dev),
              workspace=torch.empty(binding.workspace_size(p.B, p.Hq, p.total_q, p.total_k),
                                    dtype=torch.uint8, device=dev))
    stream = torch.cuda.current_stream(dev)

    def call():
        binding.attention_varlen_gated(p.q, p.k, p.v, p.q_gate, p.k_gate, p.cu_q, p.cu_k,
                                       p.alibi_slopes, p.dout, p.causal, p.window_left,
                                       p.window_right, p.scale_multiplier, stream=stream, **kw)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    st = binding.device_status(kw["workspace"])
    if st != 0:
        raise RuntimeError(f"device status {st:#x}")
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(args.steps):
        call()
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    value, ms = aggregate(flops, start.elapsed_time(end) / 1e3, args.steps, world)
    pk, kind = peaks()
    peak = pk.get("bf16_tflops_sustained", pk["bf16_tflops"])
    achieved = executed / (ms / 1e3) / 1e12
    Hkv = p.k.shape[1]
    line = {"metric": "gated fwd+full-VJP TFLOP/s & latency (pairwise sigmoid gate)",
            "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded, generated on device)",
            "config": {"workload": "gated" + ("" if args.length_scale == 1.0
                                               else f" x{args.length_scale} length"),
                       "B": p.B, "Hq": p.Hq, "Hkv": Hkv, "head_dim": d, "gate_dim": R,
                       "causal": True, "total_q": p.total_q, "scored_pairs": pairs,
                       "counted_flops_per_pair_head": 14 * d + 6 * R,
                       "counted_tflop_per_step": flops / 1e12},
            "latency_ms": ms,
            "roofline": {"bound": "tensor", "kernel": "whole call", "achieved": achieved,
                         "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                         "traffic": None, "peak_kind": f"{kind} bf16 sustained"},
            "gpu_launches": binding.launch_count(p.B, p.Hq, p.total_q, p.total_k,
                                                 Hkv=Hkv) * args.steps,
            "clocks": clk}
    if rank == 0:
        print(json.dumps(line), flush=True)


def pinned_like(x: torch.Tensor) -> torch.Tensor:
    """A pinned host tensor with x's shape, strides and values (its whole
    storage copied, so padding keeps its place)."""
    n = x.untyped_storage().nbytes() // x.element_size()
    base = torch.empty(n, dtype=x.dtype, pin_memory=True)
    src = torch.empty(0, dtype=x.dtype, device=x.device).set_(x.untyped_storage())
    base.copy_(src)
    return base.as_strided(x.shape, x.stride(), x.storage_offset())


def gpu_local_cpus(dev):
    """The host CPUs attached to the GPU's own memory node (from sysfs), or
    None where that is not published."""
    try:
        pr = torch.cuda.get_device_properties(dev)
        if isinstance(pr.pci_bus_id, str):
            bus = pr.pci_bus_id.lower()
        else:  # integer ids: domain:bus:device.function
            bus = f"{pr.pci_domain_id:04x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0"
        with open(f"/sys/bus/pci/devices/{bus}/local_cpulist") as f:
            spec = f.read().strip()
        cpus = set()
        for part in spec.split(","):
            if "-" in part:
                a, b = part.split("-")
                cpus.update(range(int(a), int(b) + 1))
            elif part:
                cpus.add(int(part))
        return cpus or None
    except (OSError, ValueError, AttributeError):
        return None


def link_probe(dev, nbytes=1 << 30):
    """Host-to-device and device-to-host GB/s of one contiguous copy of
    pinned memory (the link the end-to-end leg runs over)."""
    h = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    out = {}
    for name, fn in (("h2d_gbs", lambda: d.copy_(h, non_blocking=True)),
                     ("d2h_gbs", lambda: h.copy_(d, non_blocking=True))):
        best = None
        for _ in range(3):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize()
            dt = time.perf_counter() - t0
            best = dt if best is None else min(best, dt)
        out[name] = nbytes / best / 1e9
    return out


def run_e2e(args, p, kw, flops, stream, world):
    """The same call through the host-buffer entry point: inputs in pinned
    host memory, results back in pinned host memory, every step.  The library
    cuts the batch into chunks of whole sequences and overlaps each chunk's
    copies over the host link with the kernels of the others; all of it lies
    inside the timed region.  The process first binds to the host CPUs of
    the GPU's memory node, so the pinned buffers are allocated next to it."""
    from ragged_gqa_attention_varlen_gb300 import binding

    local = gpu_local_cpus(p.q.device)
    saved = os.sched_getaffinity(0)
    if local:
        try:
            os.sched_setaffinity(0, local & set(saved) or local)
        except OSError:
            local = None
    try:
        return _e2e_timed(args, p, kw, flops, stream, world, local)
    finally:
        os.sched_setaffinity(0, saved)


def _e2e_timed(args, p, kw, flops, stream, world, local):
    from ragged_gqa_attention_varlen_gb300 import binding

    probe = link_probe(p.q.device)

    hq, hk, hv, hdo = (pinned_like(x) for x in (p.q, p.k, p.v, p.dout))
    hcu_q, hcu_k = p.cu_q.cpu(), p.cu_k.cpu()
    hsl = p.alibi_slopes.cpu() if p.alibi_slopes is not None else None
    d = p.q.shape[-1]
    chunks = args.e2e_chunks
    outs = dict(out=torch.empty(p.q.shape, dtype=p.q.dtype, pin_memory=True),
                dq=torch.empty(p.q.shape, dtype=p.q.dtype, pin_memory=True),
                dk=torch.empty(p.k.shape, dtype=p.k.dtype, pin_memory=True),
                dv=torch.empty(p.v.shape, dtype=p.v.dtype, pin_memory=True),
                lse=torch.empty((p.total_q, p.Hq), dtype=torch.float32, pin_memory=True),
                host_status=torch.zeros(chunks, dtype=torch.int32, pin_memory=True))
    buf = torch.empty(binding.host_buffer_size_for(p.cu_q, p.cu_k, p.Hq, args.hkv, d, chunks),
                      dtype=torch.uint8, device=p.q.device)
    # bytes the call moves: the elements of every input and output (padding
    # between heads or tokens is not copied), the rebased cu arrays, slopes
    h2d = (2 * p.q.numel() + 2 * p.k.numel()) * p.q.element_size() + \
        8 * (p.B + chunks) + (4 * p.alibi_slopes.numel() if hsl is not None else 0)
    d2h = (2 * p.q.numel() + 2 * p.k.numel()) * p.q.element_size() + \
        4 * p.total_q * p.Hq + 4 * chunks

    def step():
        binding.attention_varlen_fvjp_host(hq, hk, hv, hcu_q, hcu_k, hsl, hdo, p.causal,
                                           p.window_left, p.window_right, p.softcap,
                                           p.scale_multiplier, chunks=chunks, device_buffer=buf,
                                           stream=stream, **outs)

    for _ in range(max(1, min(args.warmup, 2))):
        step()
    torch.cuda.synchronize()
    if int(outs["host_status"].abs().sum()) != 0:
        raise RuntimeError(f"device status {outs['host_status'].tolist()}")
    # the results equal the device-resident call's (dk, dv, lse whole; out and
    # dq on their first and last 4096 tokens)
    for n in ("out", "dq", "dk", "dv", "lse"):
        h, g = outs[n], kw[n]
        sl = [slice(None)] if n in ("dk", "dv", "lse") else [slice(0, 4096), slice(-4096, None)]
        for s_ in sl:
            if not torch.equal(h[s_], g[s_].cpu()):
                raise RuntimeError(f"end-to-end {n} differs from the device call")
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(args.steps):
        step()
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    value, ms = aggregate(flops, start.elapsed_time(end) / 1e3, args.steps, world)
    nc = min(chunks, max(p.B, 1))
    return {"value": value, "unit": UNIT, "ms_per_step": ms, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "chunks": chunks,
            "device_buffer_gb": buf.numel() / 1e9,
            "link_gbs_average": (h2d + d2h) / (ms / 1e3) / 1e9,
            "link_probe": probe, "cpus_bound_to_gpu_node": bool(local),
            "gpu_launches": binding.launch_count(
                p.B, p.Hq, p.total_q, p.total_k, Hkv=args.hkv) * nc * args.steps}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--length-scale", type=float, default=1.0,
                    help="scale every sequence length (small cases for profiling)")
    ap.add_argument("--causal", action="store_true",
                    help="time the causal variant (flops counted over admissible pairs)")
    ap.add_argument("--window-left", type=int, default=-1)
    ap.add_argument("--window-right", type=int, default=-1)
    ap.add_argument("--head-dim", type=int, default=HEAD_DIM, choices=(64, 128, 160))
    ap.add_argument("--e2e-chunks", type=int, default=6,
                    help="sequence chunks of the end-to-end leg (copies overlap compute)")
    ap.add_argument("--dropout", type=float, default=None,
                    help="time with counter-based dropout at this rate (keep bits stored by "
                         "the forward, read by the backward)")
    ap.add_argument("--dropout-regen", action="store_true",
                    help="with --dropout: the backward regenerates the keep bits instead")
    ap.add_argument("--hkv", type=int, default=1,
                    help="K/V heads (query heads grouped consecutively over them)")
    ap.add_argument("--gated", action="store_true",
                    help="time the sigmoid-gated variant on its own workload")
    ap.add_argument("--gate-dim", type=int, default=64, help="gate width of --gated")
    ap.add_argument("--shard", action="store_true",
                    help="strong scaling: one batch split over the ranks by the shard plan")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("at least 3 warm-up steps")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    if args.shard:
        run_shard(args, world, rank, local)
        return 0
    if args.gated:
        run_gated(args, world, rank, local)
        return 0
    run_gpu(args, world, rank, local)
    return 0


if __name__ == "__main__":
    sys.exit(main())
