#!/usr/bin/env python3
"""Benchmark of the indexer top-k (Lightning TopK) on one GB300.

Headline (the metric the pages quote): top-k latency per row at batch size 1,
n = 262144 compressed positions (a 1M-token context at 4:1), k = 512, in
microseconds per row. One step = one lt_topk call on one row. Inputs rotate
over copies whose total exceeds twice the L2 size, so every step reads its row
from HBM.

Also reported on the same line: the batched workloads (64 ragged rows, the
4096-row prefill chunk, the 16-row two-level selection) as rows/s and HBM GB/s
against the measured copy bandwidth, the dominant kernel's roofline, the CPU
oracle timed on this host, torch.topk on the same row, an end-to-end number
through the public API with host buffers, and SM clocks sampled while timing.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With --gpus N > 1 (torchrun, one process per GPU) every rank runs its own
replica of the step (rows are independent; there is no collective on the
data path) and rank 0 prints the aggregate.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

HEADLINE = "c2_decode_262144"
METRIC = "top-k µs/row (n=262144,k=512,BS=1); batched rows/s and HBM GB/s vs roofline"
PUBLISHED_US = 15.0  # the pages' Lightning TopK figure at 1M context, BS=1 (hardware not stated)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-batched", action="store_true", help="headline only")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--trace", choices=sorted(workloads.CONFIGS), default=None,
                    help="print per-phase kernel timestamps (thread 0 of each CTA) for one workload")
    ap.add_argument("--force-threads", type=int, default=0)
    ap.add_argument("--force-cluster", type=int, default=0)
    ap.add_argument("--only", choices=sorted(workloads.CONFIGS) + sorted(workloads.COMPRESS_CONFIGS), default=None,
                    help="time one workload's kernel alone (for profilers); prints a short JSON line")
    ap.add_argument("--dtype", choices=["f32", "bf16"], default="f32", help="score type in --only / --trace runs")
    ap.add_argument("--kernel", choices=["auto", "resident", "stream"], default="auto",
                    help="force the top-k kernel in --only / --trace runs")
    return ap.parse_args()


# ------------------------------------------------------------------ distributed (replicas)

def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The slowest rank's time (every rank gets it)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_us_per_row(max_total_ms: float, steps: int, rows_per_rank: int, world: int) -> float:
    """Replicas: every rank runs `steps` steps of `rows_per_rank` rows; the job's
    time is the slowest rank's, so the whole-job figure is that time over all
    rows processed by all ranks."""
    return max_total_ms * 1000.0 / (steps * rows_per_rank * world)


# ------------------------------------------------------------------ clocks

class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons while the GPU works."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except FileNotFoundError:
            self.proc = None
        time.sleep(0.2)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            self.proc.wait(timeout=10)

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sms, mx, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sms.append(float(parts[0]))
                mx.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        busy = [s for s, p in zip(sms, power) if p > 1.2 * min(power)] or sms
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sms)}


# ------------------------------------------------------------------ timing helpers

def timed_steps(launch, steps: int, warmup: int, world: int) -> float:
    """The timed region: `warmup` untimed steps, then exactly `steps` steps
    launched back to back between two CUDA events on the launching stream,
    bracketed by a barrier and a device synchronize on both sides. A sleep
    kernel queued first keeps the GPU busy while the host enqueues the steps,
    so the events see GPU time only. Returns milliseconds for all steps."""
    for i in range(warmup):
        launch(i)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    torch.cuda._sleep(int(2e6 + steps * 1e5))  # covers the host-side enqueue of all steps
    a.record()
    for i in range(steps):
        launch(warmup + i)
    b.record()
    torch.cuda.synchronize()
    barrier(world)
    return a.elapsed_time(b)


def launch_durations(launch, steps: int, world: int, offset: int = 0):
    """Diagnostic pass: an event pair around every launch (each launch then
    also pays its own launch latency). Returns per-launch milliseconds."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    torch.cuda._sleep(int(2e6 + steps * 1e5))
    for i in range(steps):
        ev[i][0].record()
        launch(offset + i)
        ev[i][1].record()
    torch.cuda.synchronize()
    barrier(world)
    return [x.elapsed_time(y) for x, y in ev]


def l2_bytes():
    try:
        return int(torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size)
    except Exception:
        return 128 << 20


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def profile_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it matches the current source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        with open(path) as fh:
            d = json.load(fh)
        e = d.get(f"{kernel}:{workload}")
        if not e:
            return None
        from sparse_attention_indexer_lt_gb300 import build as b
        if e.get("source_hash") != b.source_hash():
            return None
        return float(e["dram_bytes_per_launch"])
    except Exception:
        return None


# ------------------------------------------------------------------ our arm

def headline_config(world: int) -> dict:
    """The headline workload, printed identically by both arms."""
    w = workloads.CONFIGS[HEADLINE]
    return {"workload": HEADLINE, "rows": w.rows, "n": w.row_stride, "k": w.k,
            "l2": "inputs rotate over copies totalling more than twice the L2 (GPU arm)",
            "parallelism": "replicas" if world > 1 else "single GPU"}


def bench_ours(args, world, rank):
    import sparse_attention_indexer_lt_gb300 as lt
    from sparse_attention_indexer_lt_gb300 import build as ltb
    ltb.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    peak, peak_kind = measured_peaks()
    L2 = l2_bytes()
    result = {}

    # ---- headline: BS=1, n=262144, k=512
    S, _, w = workloads.make(HEADLINE)
    row_bytes = 4 * w.row_stride
    ncopies = workloads.l2_rotation_copies(row_bytes, L2)
    base = S.to(dev)
    copies = [base.clone() for _ in range(ncopies)]
    oi = torch.empty(w.rows, w.k, dtype=torch.int32, device=dev)
    ov = torch.empty(w.rows, w.k, dtype=torch.float32, device=dev)

    def step(i):
        lt.topk(copies[i % ncopies], None, w.k, out_idx=oi, out_val=ov)

    with Clocks(dev.index) as clk:
        total_ms = timed_steps(step, args.steps, args.warmup, world)
        per = launch_durations(step, args.steps, world, offset=args.warmup + args.steps)
        # warm-L2 latency (the indexer that produced the row has just written it)
        warm_ms = timed_steps(lambda i: lt.topk(base, None, w.k, out_idx=oi, out_val=ov),
                              args.steps, args.warmup, world)
        batched = [] if args.no_batched else bench_batched(lt, dev, args, world, peak, L2)
        compress = [] if args.no_batched else bench_compress(lt, dev, args, world, peak)
        ttk = bench_torch_topk(base, w.k, args, world)
    clocks = clk.summary()
    total_ms = max_over_ranks(total_ms, world)
    us_per_row = whole_job_us_per_row(total_ms, args.steps, w.rows, world)
    kern_ms = total_ms / args.steps  # average launch duration over the timed region
    achieved = (4 * w.row_stride * w.rows) / (kern_ms * 1e-3) / 1e9
    traffic = profile_traffic("topk_kernel", HEADLINE)
    plan = lt.plan(w.rows, w.row_stride, w.k)

    # ---- end to end through the public API: pinned host row -> device, top-k, results -> host
    e2e = bench_e2e(lt, S, w, dev, args, world)

    line = {
        "metric": METRIC,
        "value": round(us_per_row, 3),
        "unit": "µs/row",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 6),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": round(us_per_row / PUBLISHED_US, 4),
        "dtype": "u32",
        "data": "synthetic (seeded N(0,1)->bf16 + U(2,6) tail on 1%, no dataset)",
        "config": headline_config(world),
        "headline_detail": {
            "l2_copies": f"{ncopies} rotating input copies ({ncopies * row_bytes >> 20} MiB > 2x L2)",
            "plan": plan, "timing": "events around the back-to-back launches of the timed steps",
            "warm_l2_us_per_row": round(warm_ms * 1000.0 / args.steps, 3),
            "isolated_launch_us_median": round(statistics.median(per) * 1000.0, 3)},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 5), "traffic": traffic,
                     "peak_kind": f"{peak_kind} copy bandwidth (burst)",
                     "kernel": "lt::topk_kernel", "algorithmic_bytes_per_launch": 4 * w.row_stride * w.rows},
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clocks,
        "torch_topk_us": ttk,
        "batched": batched,
        "compress": compress,
        "published_context": {"lightning_topk_us": PUBLISHED_US, "plain_pytorch_us": 100.0,
                              "hardware": "not stated on the pages"},
    }
    if rank == 0 and world == 1 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(S, w, args.cpu_seconds)
    return line


BATCHED = [("c3_ragged_64", "f32"), ("c4_prefill_4096", "f32"), ("c5_blocked_16", "f32"),
           ("c6_listed_16", "f32"), ("c4_prefill_4096", "bf16"), ("c2_decode_262144", "bf16"),
           ("c5_blocked_16", "bf16")]


def bench_batched(lt, dev, args, world, peak, L2):
    out = []
    steps = max(3, min(args.steps, 50))
    for name, dtype in BATCHED:
        S, L, w = workloads.make(name)
        if dtype == "bf16":  # the same scores handed over as bf16: half the bytes per position
            S = workloads.to_bf16(S)
        esize = S.element_size()
        listed = name.startswith("c6")
        nbytes = workloads.read_bytes(L, w.rows, w.row_stride) * esize // 4
        # copies rotate over what a step touches (whole rows, for every kernel here)
        ncopies = workloads.l2_rotation_copies(nbytes, L2) if nbytes < 4 * L2 else 1
        cand = workloads.listed_blocks(name).to(dev) if listed else None
        if listed:  # the method reads the listed blocks' scores and the list, not the whole row
            nbytes = esize * cand.numel() * w.block + 4 * cand.numel()
        base = S.to(dev)
        copies = [base] + [base.clone() for _ in range(ncopies - 1)]
        ld = None if L is None else L.to(dev)
        oi = torch.empty(w.rows, w.k, dtype=torch.int32, device=dev)
        ov = torch.empty(w.rows, w.k, dtype=torch.float32, device=dev)
        ob = torch.empty(w.rows, w.k_blocks, dtype=torch.int32, device=dev) if w.blocked else None
        if w.blocked:
            def step(i, c=copies, n=ncopies):
                lt.topk_blocked(c[i % n], ld, w.block, w.k_blocks, w.k, out_idx=oi, out_val=ov, out_blocks=ob)
        elif listed:
            def step(i, c=copies, n=ncopies):
                lt.topk_candidates(c[i % n], cand, ld, w.block, w.k, out_idx=oi, out_val=ov)
        else:
            def step(i, c=copies, n=ncopies):
                lt.topk(c[i % n], ld, w.k, out_idx=oi, out_val=ov)
        total_ms = timed_steps(step, steps, max(3, args.warmup), world)
        total_ms = max_over_ranks(total_ms, world)
        step_ms = total_ms / steps
        kern_ms = step_ms
        gbs = nbytes / (kern_ms * 1e-3) / 1e9
        out.append({
            "workload": name, "dtype": dtype, "rows": w.rows, "read_bytes": nbytes,
            "rows_per_s": round(w.rows * world / (step_ms * 1e-3), 1),
            "us_per_row": round(step_ms * 1000.0 / w.rows, 4),
            "kernel_us": round(kern_ms * 1000.0, 2),
            "hbm_gbs": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
            "l2": f"{ncopies} rotating copies" if ncopies > 1 else "input larger than 4x L2",
            "plan": lt.plan(w.rows, w.row_stride, w.k, blocked=w.blocked or listed,
                            k_blocks=1 if listed else w.k_blocks),
        })
        if w.rows == 1:
            out[-1]["us_per_row_note"] = "one row: latency per call, back to back"
        if listed:
            out[-1]["bytes"] = "listed blocks' scores + the list"
            out[-1]["plan"] = lt.plan_candidates(w.rows, w.row_stride, w.block, cand.shape[1], w.k, dtype=S.dtype)
        kname = "listed_kernel" if listed else ("blocked_kernel" if w.blocked else "topk_kernel")
        key = name if dtype == "f32" else f"{name}:{dtype}"
        # DRAM bytes per launch from the committed ncu capture (null when none
        # matches the built sources)
        out[-1]["traffic"] = profile_traffic(kname, key)
        if not args.no_cpu and world == 1 and dtype == "f32":
            out[-1]["cpu_baseline"] = cpu_batched(name, S, L, w, None if cand is None else cand.cpu())
        del copies, base
        torch.cuda.empty_cache()
    return out


def compress_bytes(w, esize: int) -> int:
    """Algorithmic bytes of one compressor launch: kv and score read once, one
    entry per block written, the bias read once."""
    nblk = w.tokens // w.ratio
    return w.rows * (nblk * w.ratio * w.dim * 2 * esize + nblk * w.dim * esize) + w.ratio * w.dim * 4


def bench_compress(lt, dev, args, world, peak):
    """The fused KV compressor at a million-token context (bf16 kv and scores,
    inputs larger than the L2, drawn on the device)."""
    out = []
    steps = max(3, min(args.steps, 20))
    for name in sorted(workloads.COMPRESS_CONFIGS):
        w = workloads.COMPRESS_CONFIGS[name]
        kv, sc, bias = workloads.compress_inputs(w.rows, w.tokens, w.dim, w.ratio, seed=0, device=dev,
                                                 dtype=torch.bfloat16)
        y = torch.empty(w.rows, w.tokens // w.ratio, w.dim, dtype=torch.bfloat16, device=dev)
        nbytes = compress_bytes(w, 2)
        total_ms = timed_steps(lambda i: lt.compress(kv, sc, bias, w.ratio, out=y), steps, max(3, args.warmup),
                               world)
        step_ms = max_over_ranks(total_ms, world) / steps
        gbs = nbytes / (step_ms * 1e-3) / 1e9
        out.append({"workload": name, "dtype": "bf16", "tokens": w.tokens, "dim": w.dim, "ratio": w.ratio,
                    "bytes": nbytes, "kernel_us": round(step_ms * 1000.0, 2), "hbm_gbs": round(gbs, 1),
                    "frac_of_peak": round(gbs / peak, 4),
                    "tokens_per_s": round(w.rows * w.tokens * world / (step_ms * 1e-3), 1),
                    "l2": f"inputs {2 * kv.numel() * 2 >> 20} MiB, larger than the L2",
                    "traffic": profile_traffic("compress_ring_kernel", name)})
        del kv, sc, bias, y
        torch.cuda.empty_cache()
    return out


KERNEL_IDS = {"auto": 0, "resident": 1, "stream": 2}


def bench_only(args, world):
    """One workload, one kernel: warmup + steps launches on rotating copies."""
    import sparse_attention_indexer_lt_gb300 as lt
    from sparse_attention_indexer_lt_gb300 import build as ltb
    ltb.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    if args.only in workloads.COMPRESS_CONFIGS:
        w = workloads.COMPRESS_CONFIGS[args.only]
        kv, sc, bias = workloads.compress_inputs(w.rows, w.tokens, w.dim, w.ratio, seed=0, device=dev,
                                                 dtype=torch.bfloat16)
        y = torch.empty(w.rows, w.tokens // w.ratio, w.dim, dtype=torch.bfloat16, device=dev)
        total_ms = timed_steps(lambda i: lt.compress(kv, sc, bias, w.ratio, out=y), args.steps, args.warmup, world)
        kern = total_ms / args.steps
        nbytes = compress_bytes(w, 2)
        return {"workload": args.only, "dtype": "bf16", "steps": args.steps, "step_us": round(kern * 1000, 3),
                "bytes": nbytes, "hbm_gbs": round(nbytes / (kern * 1e-3) / 1e9, 1)}
    S, L, w = workloads.make(args.only)
    if args.dtype == "bf16":
        S = workloads.to_bf16(S)
    nbytes = workloads.read_bytes(L, w.rows, w.row_stride) * S.element_size() // 4
    L2 = l2_bytes()
    ncopies = workloads.l2_rotation_copies(nbytes, L2) if nbytes < 4 * L2 else 1
    base = S.to(dev)
    copies = [base] + [base.clone() for _ in range(ncopies - 1)]
    ld = None if L is None else L.to(dev)
    oi = torch.empty(w.rows, w.k, dtype=torch.int32, device=dev)
    ov = torch.empty(w.rows, w.k, dtype=torch.float32, device=dev)
    ob = torch.empty(w.rows, w.k_blocks, dtype=torch.int32, device=dev) if w.blocked else None
    listed = args.only.startswith("c6")
    cand = workloads.listed_blocks(args.only).to(dev) if listed else None
    if listed:
        nbytes = S.element_size() * cand.numel() * w.block + 4 * cand.numel()

    def step(i):
        c = copies[i % ncopies]
        if w.blocked:
            lt.topk_blocked(c, ld, w.block, w.k_blocks, w.k, out_idx=oi, out_val=ov, out_blocks=ob,
                            force_cluster=args.force_cluster, force_threads=args.force_threads)
        elif listed:
            lt.topk_candidates(c, cand, ld, w.block, w.k, out_idx=oi, out_val=ov,
                               force_cluster=args.force_cluster, force_threads=args.force_threads)
        else:
            lt.topk(c, ld, w.k, out_idx=oi, out_val=ov, force_kernel=KERNEL_IDS[args.kernel],
                    force_cluster=args.force_cluster, force_threads=args.force_threads)

    total_ms = timed_steps(step, args.steps, args.warmup, world)
    kern = total_ms / args.steps
    return {"workload": args.only, "dtype": args.dtype, "steps": args.steps, "step_us": round(kern * 1000, 3),
            "read_bytes": nbytes,
            "hbm_gbs": round(nbytes / (kern * 1e-3) / 1e9, 1), "copies": ncopies,
            "plan": (lt.plan_candidates(w.rows, w.row_stride, w.block, cand.shape[1], w.k, dtype=S.dtype) if listed else
                     lt.plan(w.rows, w.row_stride, w.k, blocked=w.blocked, k_blocks=w.k_blocks,
                             force_kernel=0 if w.blocked else KERNEL_IDS[args.kernel],
                             force_cluster=args.force_cluster, force_threads=args.force_threads))}


TRACE_NAMES = ["start", "hist", "merge", "estimate", "filter", "exchange", "exact", "output",
               "B.start", "B.hist", "B.merge", "B.estimate", "B.filter", "B.exchange", "B.exact", "B.unused"]


def bench_trace(args):
    """Phase timestamps of one launch: per phase, the median and max over CTAs of
    the time since that CTA started, and the median time since the first CTA started."""
    import sparse_attention_indexer_lt_gb300 as lt
    from sparse_attention_indexer_lt_gb300 import build as ltb
    ltb.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    S, L, w = workloads.make(args.trace)
    if args.dtype == "bf16":
        S = workloads.to_bf16(S)
    base = S.to(dev)
    # as many rotating copies as the timed bench uses, so the traced launch reads cold rows
    nbytes = workloads.read_bytes(L, w.rows, w.row_stride)
    L2 = l2_bytes()
    ncopies = workloads.l2_rotation_copies(nbytes, L2) if nbytes < 4 * L2 else 1
    copies = [base] + [base.clone() for _ in range(max(1, ncopies) - 1)]
    ld = None if L is None else L.to(dev)
    listed = args.trace.startswith("c6")
    cand = workloads.listed_blocks(args.trace).to(dev) if listed else None
    kid = 0 if (w.blocked or listed) else KERNEL_IDS[args.kernel]
    if listed:
        pl = lt.plan_candidates(w.rows, w.row_stride, w.block, cand.shape[1], w.k, dtype=S.dtype,
                                force_cluster=args.force_cluster, force_threads=args.force_threads)
    else:
        pl = lt.plan(w.rows, w.row_stride, w.k, blocked=w.blocked or listed, k_blocks=1 if listed else w.k_blocks,
                     force_cluster=args.force_cluster, force_threads=args.force_threads, force_kernel=kid)
    ctas = pl["grid"]  # persistent kernels: the first row of each CTA is traced
    tr = torch.full((ctas, 16), -1, dtype=torch.int64, device=dev)
    kw = dict(force_cluster=args.force_cluster, force_threads=args.force_threads)
    for i in range(max(3, args.warmup) + 1):
        tr.fill_(-1)
        c = copies[i % len(copies)]
        if w.blocked:
            lt.topk_blocked(c, ld, w.block, w.k_blocks, w.k, trace=tr, **kw)
        elif listed:
            lt.topk_candidates(c, cand, ld, w.block, w.k, trace=tr, **kw)
        else:
            lt.topk(c, ld, w.k, trace=tr, force_kernel=kid, **kw)
        torch.cuda.synchronize()
    t = tr.cpu()
    t = t[t[:, 0] >= 0]  # CTAs that ran (the buffer may hold more slots than the launch has CTAs)
    start = t[:, 0]
    t0 = int(start.min())
    out = {"workload": args.trace, "plan": pl, "ctas": ctas, "phases_us": {}}
    for i, name in enumerate(TRACE_NAMES):
        col = t[:, i]
        ok = col >= 0
        if i == 0 or int(ok.sum()) == 0:
            continue
        rel = (col[ok] - start[ok]).double() / 1000.0
        glob = (col[ok] - t0).double() / 1000.0
        out["phases_us"][name] = {"median": round(float(rel.median()), 3), "max": round(float(rel.max()), 3),
                                  "since_first_start_median": round(float(glob.median()), 3)}
    out["start_spread_us"] = round(float((start - t0).double().max()) / 1000.0, 3)
    return out


def bench_torch_topk(x, k, args, world):
    steps = max(3, min(args.steps, 50))
    ms = timed_steps(lambda i: torch.topk(x, k, dim=1, sorted=True), steps, 3, world)
    return round(ms * 1000.0 / steps, 3)


def bench_e2e(lt, S, w, dev, args, world):
    """The headline step through the public API with host buffers: the row from
    pinned host memory, the selection, and indices and values in pinned host
    memory. The kernel reads the pinned row and writes the pinned outputs in
    place over the host link (NVLink-C2C on this Grace host); the same step
    with the row first copied into device memory and the outputs copied back
    (one copy: both share one device buffer) is timed too and reported beside
    it. Each step is captured once in a
    CUDA graph and replayed, as a decode loop would run it; if capture fails,
    the same calls run eagerly."""
    host = S.pin_memory()
    dev_in = torch.empty_like(S, device=dev)
    out = torch.empty(2, w.rows, w.k, dtype=torch.int32, device=dev)
    oi, ov = out[0], out[1].view(torch.float32)
    hout = torch.empty(2, w.rows, w.k, dtype=torch.int32).pin_memory()

    hoi, hov = hout[0], hout[1].view(torch.float32)

    def in_place(_):
        # the kernel reads the pinned row and writes the pinned outputs in place
        lt.topk(host, None, w.k, out_idx=hoi, out_val=hov)

    def staged(_):
        dev_in.copy_(host, non_blocking=True)
        lt.topk(dev_in, None, w.k, out_idx=oi, out_val=ov)
        hout.copy_(out, non_blocking=True)

    def timed(step):
        mode = "eager"
        run = step
        try:
            side = torch.cuda.Stream(dev)
            side.wait_stream(torch.cuda.current_stream(dev))
            with torch.cuda.stream(side):
                for i in range(3):
                    step(i)  # plans and attributes are cached before capture
            torch.cuda.current_stream(dev).wait_stream(side)
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                step(0)
            torch.cuda.synchronize()
            run = lambda _: graph.replay()  # noqa: E731
            mode = "CUDA graph"
        except Exception as e:  # pragma: no cover - reported, not hidden
            mode = f"eager (graph capture failed: {type(e).__name__})"
            torch.cuda.synchronize()
        for i in range(args.warmup):
            run(i)
        torch.cuda.synchronize()
        barrier(world)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for i in range(args.steps):
            run(i)
        b.record()
        torch.cuda.synchronize()
        barrier(world)
        ms = max_over_ranks(a.elapsed_time(b), world)
        return round(ms * 1000.0 / (args.steps * w.rows * world), 3), mode

    us, mode = timed(in_place)
    ref_i = hout[0].clone()
    us_staged, mode_staged = timed(staged)
    if not torch.equal(ref_i, hout[0]):  # both ways must give the same row
        raise RuntimeError("in-place and staged end-to-end steps disagree")
    return {"value": us, "unit": "µs/row",
            "h2d_bytes_per_step": host.numel() * 4, "d2h_bytes_per_step": 8 * w.rows * w.k,
            "staged_copy_value": us_staged,
            "note": f"lt.topk reading the pinned host row and writing indices and values to pinned host "
                    f"memory in place over the host link; {mode}; host launch overhead included. "
                    f"staged_copy_value: the row copied to device memory and the results copied back "
                    f"({mode_staged})"}


def cpu_baseline(S, w, seconds):
    import oracle
    oracle.build()
    x = S.numpy()
    oracle.topk(x, None, w.k, nthreads=1)
    n, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        oracle.topk(x, None, w.k, nthreads=1)
        n += 1
    dt = time.perf_counter() - t0
    return {"value": round(dt / (n * w.rows) * 1e6, 1), "unit": "µs/row", "cores": 1, "kind": "oracle",
            "sample": f"{n} repetitions of the {HEADLINE} row (std::stable_sort, one thread: batch size 1)",
            "cpu": cpu_name()}


def cpu_batched(name, S, L, w, cand, seconds: float = 2.0):
    """The oracle on a batched workload, rows spread over every host core this
    process may use; whole batches repeated for about `seconds`."""
    import oracle
    oracle.build()
    nt = oracle.default_threads()
    x = S.numpy()
    ln = None if L is None else L.numpy()

    def run():
        if w.blocked:
            oracle.topk_blocked(x, ln, w.block, w.k_blocks, w.k, nthreads=nt)
        elif cand is not None:
            oracle.topk_candidates(x, ln, cand.numpy(), w.block, w.k, nthreads=nt)
        else:
            oracle.topk(x, ln, w.k, nthreads=nt)

    n, t0 = 0, time.perf_counter()
    while n == 0 or time.perf_counter() - t0 < seconds:
        run()
        n += 1
    dt = time.perf_counter() - t0
    return {"value": round(dt / (n * w.rows) * 1e6, 2), "unit": "µs/row", "cores": nt, "kind": "oracle",
            "sample": f"{n} whole batches of {name} ({w.rows} rows), rows spread over {nt} threads",
            "cpu": cpu_name()}


def cpu_name():
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part", "hardware")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


# ------------------------------------------------------------------ reference arm (the CPU oracle)

def bench_reference(args, world, rank):
    import oracle
    oracle.build()
    S, _, w = workloads.make(HEADLINE)
    x = S.numpy()
    for _ in range(args.warmup):
        oracle.topk(x, None, w.k, nthreads=1)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.topk(x, None, w.k, nthreads=1)
    dt = time.perf_counter() - t0
    v = round(dt / (args.steps * w.rows) * 1e6, 1)
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "µs/row", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1000.0 / args.steps, 4),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded)", "config": headline_config(1),
        "cpu_baseline": {"value": v, "unit": "µs/row", "cores": 1, "kind": "oracle",
                         "sample": f"{args.steps} timed steps of the {HEADLINE} row, one thread",
                         "cpu": cpu_name()},
        "e2e": {"value": v, "unit": "µs/row", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    if args.impl == "reference":
        # the reference arm is the CPU oracle: rank 0 runs it, other ranks exit without work
        if int(os.environ.get("RANK", "0")) == 0:
            print(json.dumps(bench_reference(args, 1, 0)), flush=True)
        return
    world, rank, local = dist_setup(args.gpus)
    if args.trace:
        line = bench_trace(args)
        if rank == 0:
            print(json.dumps(line), flush=True)
        return
    if args.only:
        line = bench_only(args, world)
        if rank == 0:
            print(json.dumps(line), flush=True)
        return
    line = bench_ours(args, world, rank)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
