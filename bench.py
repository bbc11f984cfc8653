#!/usr/bin/env python
"""Benchmark of DDTree verify attention (MLA, absorbed form) on GB300.

One step = one mla_verify_attn call (metadata kernel, split-KV attention,
LSE combine) over the 200k-prefix workload: B=1, H=64, a 64-node draft tree
(depth <= 8), 200,000 prefix tokens at scattered page_size=1 slots of a
262,144-slot bf16 latent pool.  Inputs are seeded synthetic data of that shape.

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU float64
oracle instead, on bounded row samples of the same workload.

Multi-GPU: the call has no exchange step, so N GPUs run N independent
replicas of the workload (one process per GPU under torchrun); the timed
region is bracketed by a barrier and the slowest rank's time is reported.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mla_tree_verify_absorbed_gb300 import inputs as I  # noqa: E402

METRIC = "verify-attn µs/call & effective KV GB/s (% HBM roofline), H=64, 200k prefix"
UNIT = "us/call"
WORKLOAD = "c3"
WORKLOAD_DESC = {
    "c3": ("B=1 H=64 prefix=200000 tree=64 nodes (depth<=8) Dl=512 Dr=64 bf16 "
           "page_size=1 slots = seeded permutation of a 262144-slot pool"),
    "c6": ("B=1 H=64 prefix=200000 chain of 4 nodes (linear draft) Dl=512 Dr=64 bf16 "
           "page_size=1 slots = seeded permutation of a 262144-slot pool"),
}


def workload_desc(name: str, p) -> str:
    if name in WORKLOAD_DESC:
        return WORKLOAD_DESC[name]
    return (f"B={p.B} H={p.H} Q={p.Q} prefix={int(np.max(p.prefix_lens))} {p.dtype} "
            f"page_size={p.page_size}")
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0
KERNELS_PER_CALL = 4  # metadata (2), attention, combine


# ----------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ----------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def job_us_per_call(ms_per_step: float, world: int) -> float:
    """Whole-job figure of the replicas: each of the `world` ranks completes one
    call per step, so the job completes `world` calls in the slowest rank's
    step time."""
    return ms_per_step * 1000.0 / world


def max_over_ranks(dist, x: float, device="cpu") -> float:
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------
# workload arithmetic (counts for the roofline; not the method)
# ----------------------------------------------------------------------------
def workload_counts(p: I.Problem):
    n = p.kv_lens.astype(np.float64)
    rows = p.H * p.Q
    el = 2 if p.dtype == "bf16" else 4
    flops = float(2.0 * rows * n.sum() * (I.DL + I.DR + I.DL))   # 2 * rows * N * 1088
    kv_bytes = float(n.sum() * I.DK * el)
    q_bytes = float(p.B * rows * I.DK * el)
    o_bytes = float(p.B * rows * (I.DL * el + 4))
    idx_bytes = float(n.sum() * 4 + (p.B + 1) * 4 + p.B * 4 + p.B * p.Q * 4)
    return dict(flops=flops, kv_bytes=kv_bytes, q_bytes=q_bytes, o_bytes=o_bytes, idx_bytes=idx_bytes)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as fh:
                return json.load(fh), "measured"
        except Exception:
            pass
    return None, "fallback"


def peak_bf16_tflops():
    pk, src = measured_peaks()
    if pk:
        for k in ("bf16_tflops", "bf16_tflops_burst", "bf16_dense_tflops"):
            if k in pk and pk[k]:
                return float(pk[k]), src
    return FALLBACK_BF16_TFLOPS, "fallback"


def peak_hbm_gbs():
    pk, src = measured_peaks()
    if pk:
        for k in ("hbm_gbs", "hbm_copy_gbs"):
            if k in pk and pk[k]:
                return float(pk[k]), src
    return FALLBACK_HBM_GBS, "fallback"


def traffic_record(kernel_src: str):
    """DRAM bytes per launch of the timed kernel from the committed ncu summary,
    or None when that summary was taken on a different kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        rec = json.load(open(path))
        src = open(os.path.join(ROOT, "mla_tree_verify_absorbed_gb300", "csrc", kernel_src), "rb").read()
        if rec.get("source_sha256") != hashlib.sha256(src).hexdigest():
            return None
        return float(rec["dram_bytes_per_launch"])
    except Exception:
        return None


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_index=None):
        self.proc = None
        self.gpu_index = gpu_index

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if self.gpu_index is not None:
            cmd += ["-i", str(self.gpu_index)]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.25)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, smax, reasons, n = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for row in csv.reader(io.StringIO(out)):
            if len(row) < 9:
                continue
            try:
                sm.append(float(row[1]))
                smax.append(float(row[2]))
            except ValueError:
                continue
            n += 1
            for name, v in zip(names, row[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": n}


def physical_gpu_index(local_rank: int):
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        parts = [x.strip() for x in vis.split(",") if x.strip()]
        if local_rank < len(parts) and parts[local_rank].isdigit():
            return int(parts[local_rank])
        return None
    return local_rank


# ----------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline leg and the reference arm)
# ----------------------------------------------------------------------------
def time_oracle_rows(p: I.Problem, n_rows: int, seed: int):
    import oracle
    orc = oracle.get()
    rows_all = I.sample_rows(p, p.H, seed=seed)
    rng = np.random.default_rng(seed)
    rows = rows_all[rng.choice(len(rows_all), size=min(n_rows, len(rows_all)), replace=False)]
    t0 = time.perf_counter()
    orc.verify_rows(p, rows)
    dt = time.perf_counter() - t0
    return dt, len(rows), orc.num_threads()


def cpu_baseline(p: I.Problem, target_s: float = 12.0):
    """Oracle on a bounded row sample, scaled to microseconds per full call."""
    import oracle
    cores = oracle.get().num_threads()
    dt, n, _ = time_oracle_rows(p, cores, seed=101)            # calibrate: one row per thread
    per_row = dt / max(n, 1)
    n2 = int(min(max(cores, target_s / max(per_row, 1e-6) * 0.9), 4 * cores * 8))
    n2 = max(cores, (n2 // cores) * cores)
    dt2, n2, cores = time_oracle_rows(p, n2, seed=102)
    total_rows = p.B * p.H * p.Q
    us_call = dt2 / n2 * total_rows * 1e6
    return {"value": us_call, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n2} of {total_rows} query rows (seeded), {dt2:.2f} s wall; "
                      f"value = measured time per row x all rows"}


# ----------------------------------------------------------------------------
# arms
# ----------------------------------------------------------------------------
def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    p = I.make_config(args.workload)
    cores = oracle.get().num_threads()
    for w in range(args.warmup):
        time_oracle_rows(p, cores, seed=1000 + w)
    times, nrows = [], 0
    for k in range(args.steps):
        dt, n, cores = time_oracle_rows(p, cores, seed=2000 + k)
        times.append(dt / n)
        nrows += n
    total_rows = p.B * p.H * p.Q
    us_call = float(np.mean(times)) * total_rows * 1e6
    line = {
        "impl": "reference", "metric": METRIC, "value": us_call, "unit": UNIT, "n_gpus": world,
        "device": "host cores (the oracle uses no GPU)",
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": us_call / 1000.0,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": f"{args.workload}: {workload_desc(args.workload, p)}"},
        "cpu_baseline": {"value": us_call, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} steps x {cores} seeded query rows of "
                                   f"{total_rows}; value = mean time per row x all rows"},
        "e2e": {"value": us_call, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch
    from mla_tree_verify_absorbed_gb300 import api

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    api.load()

    p = I.make_config(args.workload)
    cnt = workload_counts(p)
    di = api.device_inputs(p, device=dev)
    algo = args.algo
    stream = torch.cuda.current_stream(dev)
    out = torch.empty((p.B, p.Q, p.H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((p.B, p.Q, p.H), dtype=torch.float32, device=dev)
    ws = api.alloc_workspace(api.workspace_size(di, args.num_splits, algo), dev)

    for _ in range(args.warmup):
        api.verify_attn(di, out=out, lse=lse, num_splits=args.num_splits, algo=algo, workspace=ws)
    torch.cuda.synchronize(dev)
    bits = api.check(ws)
    if bits:
        raise SystemExit(f"device table check failed: {bits:#x}")
    splits_used = api.splits_used(ws)

    # --- device-resident timed region ---------------------------------------
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for a, b in evs:  # torch creates the CUDA event on first record
        a.record(stream)
        b.record(stream)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(physical_gpu_index(local)) if rank == 0 else None
    if sampler:
        sampler.start()
    barrier(dist)
    torch.cuda.synchronize(dev)
    t_start.record(stream)
    for k in range(args.steps):
        api.verify_attn(di, out=out, lse=lse, num_splits=args.num_splits, algo=algo, workspace=ws, check=False)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(dist)
    clocks = sampler.stop() if sampler else None
    elapsed_ms = t_start.elapsed_time(t_end)
    elapsed_ms = max_over_ranks(dist, elapsed_ms, device=dev)
    # the attention kernel alone: the same calls with events around it (the
    # events keep its launch from overlapping the neighbouring kernels)
    barrier(dist)
    torch.cuda.synchronize(dev)
    for k in range(args.steps):
        api.verify_attn(di, out=out, lse=lse, num_splits=args.num_splits, algo=algo, workspace=ws,
                        profile_events=evs[k], check=False)
    torch.cuda.synchronize(dev)
    attn_ms = [a.elapsed_time(b) for a, b in evs]
    attn_avg_ms = max_over_ranks(dist, float(np.mean(attn_ms)), device=dev)

    # --- the same calls with L2 flushed between them --------------------------
    l2_flushed = None
    if not args.no_l2_flush:
        flush = torch.empty((L2_FLUSH_BYTES,), dtype=torch.uint8, device=dev)
        f_steps = max(10, min(args.steps, 20))
        f_call, f_kernel = time_calls(di, p, dev, stream, dist, f_steps, args.warmup, algo, args.num_splits, flush)
        l2_flushed = {"us_per_call": job_us_per_call(f_call, world), "kernel_us": f_kernel * 1000.0,
                      "steps": f_steps, "flush_bytes": L2_FLUSH_BYTES,
                      "note": "a buffer larger than L2 written between calls, outside the timed events"}
        del flush
        torch.cuda.empty_cache()

    # --- end to end through the public API with host buffers ----------------
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, p, di, dev, stream, algo, dist)
    graph = None
    if not args.no_graph:
        graph = run_graph(args, p, di, dev, stream, algo, dist)
    compact = None
    if not args.no_compact:
        compact = run_compact(args, p, di, dev, stream, dist)
    workloads = None
    if not args.no_workloads:
        workloads = run_workloads(args, dev, stream, dist, world)
    ddtree = None
    if not args.no_ddtree:
        ddtree = run_ddtree(args, dev, stream, dist, with_oracle=(world == 1 and not args.no_cpu_baseline))

    if rank != 0:
        return 0

    ms_step = elapsed_ms / args.steps
    us_call = job_us_per_call(ms_step, world)
    kernel_s = attn_avg_ms / 1000.0
    eff_kv_gbs = cnt["kv_bytes"] / (ms_step / 1000.0) / 1e9
    resolved = "simt" if algo == "simt" else "tc"   # AUTO takes the tensor-core kernel for bf16
    if resolved == "tc":
        peak, src = peak_bf16_tflops()
        achieved = cnt["flops"] / kernel_s / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic_record("attn_tc.cu"),
                "peak_source": f"bf16 dense, {src}", "kernel": "attn_tc_kernel",
                "kernel_us": attn_avg_ms * 1000.0}
    else:
        sm = torch.cuda.get_device_properties(dev).multi_processor_count
        mhz = (clocks or {}).get("sm_max_mhz") or 2070.0
        peak = sm * 128 * 2 * mhz * 1e6 / 1e12
        achieved = cnt["flops"] / kernel_s / 1e12
        roof = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic_record("attn_simt.cu"),
                "peak_source": f"fp32 FFMA: {sm} SMs x 128 lanes x 2 x {mhz:.0f} MHz",
                "kernel": "attn_simt_kernel", "kernel_us": attn_avg_ms * 1000.0}
    hbm_peak, hsrc = peak_hbm_gbs()
    hbm_bytes = cnt["kv_bytes"] + cnt["q_bytes"] + cnt["o_bytes"]
    t_roof = max(hbm_bytes / (hbm_peak * 1e9), cnt["flops"] / (peak_bf16_tflops()[0] * 1e12))

    line = {
        "metric": METRIC, "value": us_call, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{args.workload}: {workload_desc(args.workload, p)}", "algo": resolved,
                   "num_splits": args.num_splits, "splits_used": splits_used,
                   "l2": "inputs larger than L2: 230 MB of KV read per call (129 MB L2)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "effective_kv_gbs": eff_kv_gbs,
        "tflops": cnt["flops"] / (ms_step / 1000.0) / 1e12,
        "roofline_fraction_of_call": t_roof / (ms_step / 1000.0),
        "hbm_fraction": (hbm_bytes / (ms_step / 1000.0) / 1e9) / hbm_peak,
        "hbm_peak_source": hsrc,
        "roofline": roof,
        "gpu_launches": KERNELS_PER_CALL * args.steps,
        "clocks": clocks,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if graph is not None:
        line["graph"] = graph
    if l2_flushed is not None:
        line["l2_flushed"] = l2_flushed
    if compact is not None:
        line["kv_compact"] = compact
    if workloads is not None:
        line["workloads"] = workloads
    if ddtree is not None:
        line["ddtree"] = ddtree
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(p)
    print(json.dumps(line), flush=True)
    return 0


L2_FLUSH_BYTES = 512 << 20  # written between calls of the L2-flushed timing: about four times the L2


def time_calls(di, p, dev, stream, dist, steps, warmup, algo="auto", num_splits=0, flush=None, info=None):
    """Device-resident timing of `steps` verify calls of one workload:
    per-call time (events around the back-to-back loop; with `flush`, events
    around each call and a buffer larger than L2 written between calls,
    outside the events) and the attention kernel alone (the call's
    profiling events).  `info`, when given, receives the split count the
    calls used ("splits_used")."""
    import torch
    from mla_tree_verify_absorbed_gb300 import api

    out = torch.empty((p.B, p.Q, p.H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((p.B, p.Q, p.H), dtype=torch.float32, device=dev)
    ws = api.alloc_workspace(api.workspace_size(di, num_splits, algo), dev)
    for _ in range(max(3, warmup)):
        api.verify_attn(di, out=out, lse=lse, num_splits=num_splits, algo=algo, workspace=ws)
    torch.cuda.synchronize(dev)
    if api.check(ws):
        raise RuntimeError(f"{p.name}: device table check failed")
    if info is not None:
        info["splits_used"] = api.splits_used(ws)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in evs:
        a.record(stream)
        b.record(stream)
    barrier(dist)
    torch.cuda.synchronize(dev)
    if flush is None:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            api.verify_attn(di, out=out, lse=lse, num_splits=num_splits, algo=algo, workspace=ws, check=False)
        b.record(stream)
        torch.cuda.synchronize(dev)
        call_ms = a.elapsed_time(b) / steps
    else:
        calls = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for k in range(steps):
            flush.zero_()
            calls[k][0].record(stream)
            api.verify_attn(di, out=out, lse=lse, num_splits=num_splits, algo=algo, workspace=ws, check=False)
            calls[k][1].record(stream)
        torch.cuda.synchronize(dev)
        call_ms = float(np.mean([x.elapsed_time(y) for x, y in calls]))
    barrier(dist)
    for k in range(steps):
        if flush is not None:
            flush.zero_()
        api.verify_attn(di, out=out, lse=lse, num_splits=num_splits, algo=algo, workspace=ws,
                        profile_events=evs[k], check=False)
    torch.cuda.synchronize(dev)
    kernel_ms = float(np.mean([x.elapsed_time(y) for x, y in evs]))
    return max_over_ranks(dist, call_ms, device=dev), max_over_ranks(dist, kernel_ms, device=dev)


def roofline_entry(p, call_ms, kernel_ms, world=1):
    cnt = workload_counts(p)
    peak, src = peak_bf16_tflops()
    achieved = cnt["flops"] / (kernel_ms / 1000.0) / 1e12
    return {"us_per_call": job_us_per_call(call_ms, world), "kernel_us": kernel_ms * 1000.0,
            "gflop": cnt["flops"] / 1e9, "kv_mb": cnt["kv_bytes"] / 1e6,
            "kernel_tflops": achieved, "frac": achieved / peak, "peak_source": f"bf16 dense, {src}",
            "effective_kv_gbs": cnt["kv_bytes"] / (call_ms / 1000.0) / 1e9}


def run_workloads(args, dev, stream, dist, world):
    """Short timing blocks of the other workloads (device-resident inputs):
    c6 (4-node chain over 200k, the small-Q regime), c2, c4 (ragged batch),
    c5 (128 heads, paged), and the L2-flushed variant of c2."""
    import torch
    from mla_tree_verify_absorbed_gb300 import api

    res = {}
    steps = max(10, min(args.steps, 20))
    flush = torch.empty((L2_FLUSH_BYTES,), dtype=torch.uint8, device=dev)
    for name in ("c6", "c2", "c4", "c5"):
        p = I.make_config(name)
        di = api.device_inputs(p, device=dev)
        info = {}
        call_ms, kernel_ms = time_calls(di, p, dev, stream, dist, steps, args.warmup, info=info)
        entry = roofline_entry(p, call_ms, kernel_ms, world)
        entry.update(workload=workload_desc(name, p), steps=steps, splits_used=info["splits_used"])
        if name == "c2":
            f_call, f_kernel = time_calls(di, p, dev, stream, dist, steps, args.warmup, flush=flush)
            entry["l2_flushed"] = {"us_per_call": f_call * 1000.0, "kernel_us": f_kernel * 1000.0,
                                   "flush_bytes": L2_FLUSH_BYTES}
        res[name] = entry
        del di
        torch.cuda.empty_cache()
    return res


def run_compact(args, p, di, dev, stream, dist):
    """KV compaction of the workload's rows into a contiguous destination:
    us per call and the HBM bandwidth it reaches (each row read once and
    written once)."""
    import torch
    from mla_tree_verify_absorbed_gb300 import api

    total = int(np.sum(np.asarray(p.prefix_lens, dtype=np.int64) + p.Q))
    dst = torch.empty((total, 576), dtype=torch.bfloat16, device=dev)
    new_idx = torch.empty((total,), dtype=torch.int32, device=dev)
    new_indptr = torch.empty((p.B + 1,), dtype=torch.int32, device=dev)
    ws = api.alloc_workspace(api.workspace_size(di, 1), dev)
    steps = max(10, min(args.steps, 50))
    for _ in range(max(1, args.warmup)):
        api.kv_compact_into(di, dst, new_idx, new_indptr, ws)
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist)
    a.record(stream)
    for _ in range(steps):
        api.kv_compact_into(di, dst, new_idx, new_indptr, ws)
    b.record(stream)
    torch.cuda.synchronize(dev)
    if api.check(ws) != 0:
        raise RuntimeError("kv compaction reported a device error")
    ms = max_over_ranks(dist, a.elapsed_time(b), device=dev) / steps
    moved = 2.0 * total * 576 * 2
    hbm_peak, src = peak_hbm_gbs()
    gbs = moved / (ms / 1000.0) / 1e9
    # the verify call on the compacted (contiguous) layout
    import dataclasses
    dc = dataclasses.replace(di, kv_c=dst[:, :512], k_pe=dst[:, 512:], pool=dst, page_size=1,
                             kv_indptr=new_indptr, kv_indices=new_idx, block_table=None)
    out = torch.empty((p.B, p.Q, p.H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((p.B, p.Q, p.H), dtype=torch.float32, device=dev)
    vws = api.alloc_workspace(api.workspace_size(dc, args.num_splits), dev)
    for _ in range(max(1, args.warmup)):
        api.verify_attn(dc, out=out, lse=lse, num_splits=args.num_splits, workspace=vws)
    torch.cuda.synchronize(dev)
    a.record(stream)
    for _ in range(steps):
        api.verify_attn(dc, out=out, lse=lse, num_splits=args.num_splits, workspace=vws, check=False)
    b.record(stream)
    torch.cuda.synchronize(dev)
    vms = max_over_ranks(dist, a.elapsed_time(b), device=dev) / steps
    # and on the scattered layout, timed the same way in the same block
    a.record(stream)
    for _ in range(steps):
        api.verify_attn(di, out=out, lse=lse, num_splits=args.num_splits, workspace=vws, check=False)
    b.record(stream)
    torch.cuda.synchronize(dev)
    sms = max_over_ranks(dist, a.elapsed_time(b), device=dev) / steps
    return {"us_per_call": ms * 1000.0, "rows": total, "bytes_moved": moved, "gbs": gbs,
            "hbm_frac": gbs / hbm_peak, "hbm_peak_source": src, "steps": steps,
            "verify_us_on_compacted": vms * 1000.0, "verify_us_on_scattered": sms * 1000.0}


def run_ddtree(args, dev, stream, dist, with_oracle: bool):
    """DDTree construction and greedy acceptance around the verify call: us per
    call at one sequence (the 64-node tree of the verify workload) and at 256
    sequences.  Both kernels are latency-bound (one warp per sequence, a chain
    of `budget` dependent selection steps), so the figure of merit is the
    per-call latency and the cycles per selection step."""
    import torch
    from mla_tree_verify_absorbed_gb300 import api
    from mla_tree_verify_absorbed_gb300 import draft_inputs as DI

    res = {}
    steps = max(20, args.steps)
    for name in ("tree_b1", "tree_b256"):
        d = DI.make_draft_config(name)
        root = torch.from_numpy(d.root_token).to(dev)
        ctok = torch.from_numpy(d.cand_token).to(dev)
        clp = torch.from_numpy(d.cand_logp).to(dev)
        i32 = dict(dtype=torch.int32, device=dev)
        parent, token = torch.empty((d.B, d.Q), **i32), torch.empty((d.B, d.Q), **i32)
        ws = api.alloc_workspace(api.DDTREE_WORKSPACE_BYTES, dev)
        api.ddtree_build_into(root, ctok, clp, d.budget, parent, token, ws)
        torch.cuda.synchronize(dev)
        tgt = torch.from_numpy(DI.make_targets(d, parent.cpu().numpy(), seed=5, p_follow=0.8)).to(dev)
        n_len, nodes, nxt = torch.empty((d.B,), **i32), torch.empty((d.B, d.Q), **i32), torch.empty((d.B,), **i32)
        ws_a = api.alloc_workspace(api.DDTREE_WORKSPACE_BYTES, dev)

        def timed(fn):
            for _ in range(max(3, args.warmup)):
                fn()
            torch.cuda.synchronize(dev)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            barrier(dist)
            a.record(stream)
            for _ in range(steps):
                fn()
            b.record(stream)
            torch.cuda.synchronize(dev)
            return max_over_ranks(dist, a.elapsed_time(b), device=dev) * 1000.0 / steps

        # the tensors are checked once; the timed loops skip the binding's checks
        api.ddtree_accept_into(parent, token, tgt, n_len, nodes, nxt, ws_a)
        build_us = timed(lambda: api.ddtree_build_into(root, ctok, clp, d.budget, parent, token, ws, check=False))
        accept_us = timed(lambda: api.ddtree_accept_into(parent, token, tgt, n_len, nodes, nxt, ws_a, check=False))
        if api.check(ws) or api.check(ws_a):
            raise RuntimeError("ddtree kernels reported a device error")
        # both calls replayed from one CUDA graph (a decode step's launch pattern)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            api.ddtree_build_into(root, ctok, clp, d.budget, parent, token, ws)
            api.ddtree_accept_into(parent, token, tgt, n_len, nodes, nxt, ws_a)
        graph_us = timed(g.replay)
        entry = {"B": d.B, "L": d.L, "K": d.K, "budget": d.budget, "build_us": build_us,
                 "accept_us": accept_us, "build_plus_accept_graph_us": graph_us,
                 "mean_accept_len": float(n_len.float().mean().item())}
        if with_oracle:
            t0 = time.perf_counter()
            from oracle import ddtree as odd  # CPU baseline leg only
            odd.build_tree(d.root_token, d.cand_token, d.cand_logp, d.budget)
            entry["cpu_baseline_build_us"] = (time.perf_counter() - t0) * 1e6
        res[name] = entry
    return res


def run_ddtree_only(args):
    import torch
    from mla_tree_verify_absorbed_gb300 import api

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    api.load()
    res = run_ddtree(args, dev, torch.cuda.current_stream(dev), dist, with_oracle=False)
    if rank == 0:
        print(json.dumps({"ddtree": res, "n_gpus": world, "steps": args.steps, "warmup": args.warmup}), flush=True)
    return 0


def run_graph(args, p, di, dev, stream, algo, dist):
    """The same call captured once in a CUDA graph and replayed K times
    (device-resident inputs): what a decode loop that captures its verify
    step pays per call."""
    import torch
    from mla_tree_verify_absorbed_gb300 import api

    out = torch.empty((p.B, p.Q, p.H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((p.B, p.Q, p.H), dtype=torch.float32, device=dev)
    ws = api.alloc_workspace(api.workspace_size(di, args.num_splits, algo), dev)
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        api.verify_attn(di, out=out, lse=lse, num_splits=args.num_splits, algo=algo, workspace=ws)
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        api.verify_attn(di, out=out, lse=lse, num_splits=args.num_splits, algo=algo, workspace=ws, check=False)
    for _ in range(max(1, args.warmup)):
        g.replay()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize(dev)
    a.record(stream)
    for _ in range(args.steps):
        g.replay()
    b.record(stream)
    torch.cuda.synchronize(dev)
    barrier(dist)
    ms = max_over_ranks(dist, a.elapsed_time(b), device=dev)
    world = dist.get_world_size() if dist is not None else 1
    return {"value": job_us_per_call(ms / args.steps, world), "unit": UNIT, "note": "CUDA graph replay"}


def _packed(tensors, device, pin):
    """One byte buffer holding each tensor at a 256-byte aligned offset, and
    typed views of it in the same order."""
    import torch
    offs, total = [], 0
    for t in tensors:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    buf = torch.empty((max(total, 256),), dtype=torch.uint8, device=device)
    if pin:
        buf = buf.pin_memory()
    views = [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for o, t in zip(offs, tensors)]
    return buf, views


def run_e2e(args, p, di, dev, stream, algo, dist):
    """Per step: one H2D copy of the step's queries, tree and index tables
    from a pinned host buffer (packed at 256-byte aligned offsets), the C-ABI
    call on views of the device copy, one D2H copy of out and lse.  The KV
    pool is the cache: resident on the device, not copied per step."""
    import dataclasses
    import torch
    from mla_tree_verify_absorbed_gb300 import api

    names = [n for n in ("q_lat", "q_pe", "prefix_lens", "tree_parent", "kv_indptr", "kv_indices", "block_table")
             if getattr(di, n) is not None]
    src = [getattr(di, n) for n in names]
    host_in, host_views = _packed([t.cpu() for t in src], "cpu", pin=True)
    for hv, t in zip(host_views, src):
        hv.copy_(t.cpu())
    dev_in, dev_views = _packed(src, dev, pin=False)
    de = dataclasses.replace(di, **dict(zip(names, dev_views)))
    out_shape, lse_shape = (p.B, p.Q, p.H, 512), (p.B, p.Q, p.H)
    protos = [torch.empty(out_shape, dtype=torch.bfloat16), torch.empty(lse_shape, dtype=torch.float32)]
    dev_out, (out, lse) = _packed(protos, dev, pin=False)
    host_out, (out_h, lse_h) = _packed(protos, "cpu", pin=True)
    h2d = host_in.numel()
    d2h = host_out.numel()
    ws = api.alloc_workspace(api.workspace_size(de, args.num_splits, algo), dev)

    def step():
        dev_in.copy_(host_in, non_blocking=True)
        api.verify_attn(de, out=out, lse=lse, num_splits=args.num_splits, algo=algo, workspace=ws, check=False)
        host_out.copy_(dev_out, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    # the packed path computes what the device-resident call computes
    ref_out, ref_lse = api.verify_attn(di, num_splits=args.num_splits, algo=algo)
    torch.cuda.synchronize(dev)
    if not (torch.equal(out_h, ref_out.cpu()) and torch.equal(lse_h, ref_lse.cpu())):
        raise RuntimeError("e2e: the packed host-buffer call differs from the device-resident call")
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize(dev)
    a.record(stream)
    for _ in range(args.steps):
        step()
    b.record(stream)
    torch.cuda.synchronize(dev)
    barrier(dist)
    ms = max_over_ranks(dist, a.elapsed_time(b), device=dev)
    world = dist.get_world_size() if dist is not None else 1
    return {"value": job_us_per_call(ms / args.steps, world), "unit": UNIT,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "copies_per_step": {"h2d": 1, "d2h": 1}}


def relaunch(n: int, argv) -> int:
    """Run this script as n local processes (one replica per GPU) under
    torch.distributed.run, rendezvous on 127.0.0.1; rank 0 prints the line."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *argv]
    return subprocess.call(cmd, cwd=ROOT)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=None,
                    help="GPUs (one replica each); without a launcher's WORLD_SIZE, N > 1 relaunches "
                         "this script under torch.distributed.run with N local processes")
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD, choices=list(I.CONFIG_NAMES))
    ap.add_argument("--num-splits", type=int, default=0)
    ap.add_argument("--algo", default="auto", choices=["auto", "simt", "tc"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-compact", action="store_true", help="skip the KV compaction timing")
    ap.add_argument("--no-workloads", action="store_true", help="skip the short blocks of the other workloads")
    ap.add_argument("--no-l2-flush", action="store_true", help="skip the L2-flushed timing")
    ap.add_argument("--no-ddtree", action="store_true", help="skip the DDTree construction / acceptance timing")
    ap.add_argument("--ddtree-only", action="store_true",
                    help="time only DDTree construction / acceptance and print that block as one JSON line")
    args = ap.parse_args(argv)
    env_world = os.environ.get("WORLD_SIZE")
    if env_world is None and args.gpus is not None and args.gpus > 1:
        return relaunch(args.gpus, sys.argv[1:] if argv is None else list(argv))
    if env_world is not None and args.gpus is not None and args.gpus != int(env_world):
        raise SystemExit(f"--gpus {args.gpus} disagrees with the launcher's WORLD_SIZE={env_world}")
    if args.warmup < 3:
        args.warmup = 3  # timing rule: at least three untimed warm-up steps
    if args.impl == "reference":
        return run_reference(args)
    if args.ddtree_only:
        return run_ddtree_only(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
