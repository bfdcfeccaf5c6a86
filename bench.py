#!/usr/bin/env python3
"""Benchmark of the paged-KV decode step on GB300.

Default workload (N=1): LLaMA-7B-shaped single-layer decode -- 64 sequences,
32 heads MHA, head_dim 128, block size 16, context lengths U[512, 4096],
bf16 K/V, physical blocks shuffled across a pool of the needed blocks + 10 %.
One step = the append of one new token per sequence (into its last page, the
slot of a freshly allocated block where the page was full) followed by the
decode over the context including that token, in one call
(paged_attn_decode_append: the decode CTA of each sequence's last split
writes the token's rows before it loads the pages).  The metric is KV
bytes read per second (logical K+V bytes of every sequence's context) and
sequence-steps per second.  The end-to-end figure (`e2e`) times the same
step from pinned host buffers, one library call per step (a HostStep
prepared once; paged_attn_decode_append_host: the step's packed inputs
copied in, append + decode, the output copied back, the stream
synchronised).

Under torchrun each rank runs its own replica (own sequences, own pools):
decode is data-parallel by sequence with no exchange, so scaling is weak and
the value is the bytes all ranks read divided by the slowest rank's time.

--impl reference times the fp64 CPU oracle on the host cores instead (the
reference arm of this benchmark): the same workload's whole step, or an
equal share of its sequences when the run would take more than about two
minutes.

On one GPU with the default workload the line also carries `per_config`:
the other stated workloads (tiny per launch and as 1100 problems in one
batched launch, gqa_prefix, long_context, continuous with its block copies)
measured the same way, each with the oracle's GB/s on the same inputs.

Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attention KV-read GB/s vs ~8 TB/s HBM; seq-steps/sec"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_traffic.txt")
KERNEL_SOURCES = ["paged_kv_decode_26_gb300/csrc/decode_kernel.cuh",
                  "paged_kv_decode_26_gb300/csrc/pkv_device.cuh",
                  "paged_kv_decode_26_gb300/csrc/capi.cu",
                  "paged_kv_decode_26_gb300/csrc/decode_inst.inc"]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=2, help="workload 1..5 (default 2)")
    ap.add_argument("--split", type=int, default=0, help="split_tokens (0 = automatic)")
    ap.add_argument("--seqs", type=int, default=0,
                    help="override the number of sequences (smaller cases for profiling)")
    ap.add_argument("--lens", default="",
                    help="override the context-length mix (profiling cases), e.g. "
                         "const:32768, uniform:512:4096, loguniform:128:32768")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--graph", action="store_true",
                    help="replay each step as one CUDA graph")
    ap.add_argument("--replicas", type=int, default=1,
                    help="independent copies of the workload (own pools) per GPU, one graph")
    ap.add_argument("--batched", action="store_true",
                    help="run the replicas as one batched launch (pkv_decode_batched_plan once, "
                         "paged_attn_decode_batched per step) instead of a graph")
    ap.add_argument("--multi-query", type=int, default=0,
                    help="time paged_attn_multi_query with this many new tokens per sequence")
    ap.add_argument("--graph-streams", type=int, default=32,
                    help="parallel branches of the replica graph")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the other stated workloads after the headline one")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds (wall) of threaded oracle work for the CPU baseline")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers

def kernel_source_hash() -> str:
    """Digest of the decode kernel's code: its sources with comments and
    whitespace removed, so that a comment edit keeps the committed traffic
    figure valid while any change to the code itself invalidates it."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def committed_traffic(workload: str):
    """Per-launch DRAM bytes of the decode kernel from the committed ncu
    summary, if it was taken on the current kernel sources and workload."""
    try:
        text = open(TRAFFIC_FILE).read()
    except OSError:
        return None
    src = re.search(r"^source_sha256:\s*(\S+)", text, re.M)
    wl = re.search(r"^workload:\s*(.+)$", text, re.M)
    tb = re.search(r"^traffic_bytes_per_launch:\s*(\d+)", text, re.M)
    if not (src and wl and tb) or src.group(1) != kernel_source_hash() or wl.group(1).strip() != workload:
        return None
    return int(tb.group(1))


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons (100 ms)."""
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, device_id: str):
        self.device_id = device_id
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.out = open("/tmp/pkv_clocks_%d.csv" % os.getpid(), "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.device_id, "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.out.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) == len(self.FIELDS):
                    rows.append(parts)
        os.unlink(self.out.name)
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        reasons = set()
        for r in rows:
            for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                  "sw_power_cap"), r[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


def gpu_id_for_smi(torch, dev: int) -> str:
    try:
        p = torch.cuda.get_device_properties(dev)
        return "%08x:%02x:%02x.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
    except Exception:
        return str(dev)


def workload_name(case, config, lens_override: str = "") -> str:
    from paged_kv_decode_26_gb300 import workloads as wl
    spec = wl.CONFIGS[config]
    lens = tuple(lens_override.split(":")) if lens_override else spec["lens"]
    return (f"{case.name}: {case.S} seqs, {case.H} q / {case.Hk} kv heads, d={case.D}, "
            f"block_size={case.B}, lens {lens[0]}{list(lens[1:])}, "
            f"{str(case.dtype).replace('torch.', '')} K/V, {case.num_blocks} pool blocks, seed {case.seed}")


# ------------------------------------------------------------- CPU oracle

def oracle_step_seconds(case, lens, tables, budget_s, threads=None):
    """The fp64 oracle on the whole decode step of `case` (every sequence,
    every head), threaded over the host cores (oracle.parallel), repeated
    while the total stays under about `budget_s` seconds of wall time.
    Returns (kv_bytes per run, seconds per run, runs, threads); the bytes are
    the logical K+V bytes of the step, the unit of the GPU figures."""
    from oracle import parallel
    threads = threads or parallel.host_threads()
    import torch
    row = case.Hk * case.D * case.k_pool.element_size() * 2
    kv = int(lens.to(torch.int64).sum()) * row
    times = []
    while True:
        t0 = time.perf_counter()
        parallel.decode_two_pass(case.q, case.k_pool, case.v_pool, tables, lens, case.scale,
                                 threads=threads)
        times.append(time.perf_counter() - t0)
        if sum(times) + times[-1] > budget_s or len(times) >= 50:
            break
    return kv, statistics.median(times), len(times), threads


def run_reference(args):
    """The reference arm: the fp64 oracle timed on the host cores (threaded
    over sequences and heads), each step the whole decode step of the
    workload, or an equal share of its sequences when K + W whole steps
    would not end within about two minutes."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import torch
    from oracle import build as ob
    from oracle import parallel
    from paged_kv_decode_26_gb300 import workloads as wl
    ob.build()
    threads = parallel.host_threads()
    case = wl.make_case(args.config, **({"pool_extra": 0.01} if args.config == 4 else {}))
    lens = case.context_lens
    row = case.Hk * case.D * case.k_pool.element_size() * 2
    t0 = time.perf_counter()
    parallel.decode_two_pass(case.q, case.k_pool, case.v_pool, case.block_tables, lens,
                             case.scale, threads=threads)
    t_full = time.perf_counter() - t0
    n_runs = max(1, args.steps + args.warmup)
    frac = min(1.0, 120.0 / (n_runs * max(t_full, 1e-6)))
    n_seq = max(1, int(round(case.S * frac)))
    # every step takes the next n_seq sequences (cyclically), so the steps
    # together cover the workload's length mix
    order = list(range(case.S))

    def seqs_of(i):
        return [order[(i * n_seq + k) % case.S] for k in range(n_seq)]

    for i in range(args.warmup):
        parallel.decode_two_pass(case.q, case.k_pool, case.v_pool, case.block_tables, lens,
                                 case.scale, seq_ids=seqs_of(i), threads=threads)
    total_b, total_t = 0, 0.0
    for i in range(args.steps):
        sel = seqs_of(args.warmup + i)
        t0 = time.perf_counter()
        parallel.decode_two_pass(case.q, case.k_pool, case.v_pool, case.block_tables, lens,
                                 case.scale, seq_ids=sel, threads=threads)
        total_t += time.perf_counter() - t0
        total_b += int(lens[sel].to(torch.int64).sum()) * row
    ms = total_t / max(1, args.steps) * 1e3
    value = total_b / max(total_t, 1e-9) / 1e9
    sample = (f"per step: {n_seq} of {case.S} sequences of the step (all {case.H} heads), "
              f"fp64 two-pass oracle on {threads} host threads" +
              ("" if n_seq == case.S else "; consecutive steps take consecutive sequences"))
    line = {"metric": METRIC, "value": value, "unit": "GB/s", "impl": "reference",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_name(case, args.config, args.lens)},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------- multi-rank helpers

def rank_seed(config: int, rank: int, replica: int = 0) -> int:
    """Seed of one rank's replica: every rank decodes its own sequences."""
    return (config - 1) + 1000 * rank + 7919 * replica


def reduce_over_ranks(values, op: str, dist, world: int, device):
    """Element-wise max or sum of a list of floats over all ranks."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return [float(v) for v in t.tolist()]


def job_gbs(total_bytes: float, ms: float) -> float:
    """Whole-job throughput: bytes of all ranks over the slowest rank's time."""
    return total_bytes / (ms / 1e3) / 1e9


# ------------------------------------------------------------------ ours

def build_replicas(args, rank, dev, pkv, wl, torch, np):
    """R independent copies of the workload (own pools, own sequences), with
    the per-step inputs of all copies packed in contiguous buffers (so that
    the end-to-end step moves them with one copy each)."""
    R = max(1, args.replicas)
    extra = {"pool_extra": 0.01} if args.config == 4 else {}
    if args.seqs:
        extra["S"] = args.seqs
    if args.lens:
        kind, *nums = args.lens.split(":")
        extra["lens"] = (kind, *[float(x) if "." in x else int(x) for x in nums])
    reps = []
    for r in range(R):
        seed = rank_seed(args.config, rank, r)
        case = wl.make_case(args.config, seed=seed, **extra)
        S = case.S
        bm = pkv.BlockManager(case.num_blocks, case.B, free_ids=case.free_ids)
        bt_h = case.block_tables.clone()
        lens_h = case.context_lens.clone()
        slots_h = torch.empty(S, dtype=torch.int64)
        if case.k_new is None:
            case.k_new = wl._normal(np.random.default_rng(seed + 7), (S, case.Hk, case.D), case.dtype)
            case.v_new = wl._normal(np.random.default_rng(seed + 8), (S, case.Hk, case.D), case.dtype)
        need_cols = int(((lens_h + 1 + case.B - 1) // case.B).max())
        if need_cols > bt_h.shape[1]:
            bt_h = torch.cat([bt_h, torch.full((S, need_cols - bt_h.shape[1]), -1,
                                               dtype=torch.int32)], 1)
        if bm.append_slots(bt_h, lens_h, slots_h) != 0:
            raise RuntimeError("pool has no room for the appended tokens")
        reps.append({"case": case, "bt_h": bt_h, "lens_h": lens_h, "slots_h": slots_h})
    S = reps[0]["case"].S
    mb = max(r["bt_h"].shape[1] for r in reps)
    host = {
        "q": torch.cat([r["case"].q for r in reps]).pin_memory(),
        "k_new": torch.cat([r["case"].k_new for r in reps]).pin_memory(),
        "v_new": torch.cat([r["case"].v_new for r in reps]).pin_memory(),
        "bt": torch.stack([torch.nn.functional.pad(r["bt_h"], (0, mb - r["bt_h"].shape[1]),
                                                   value=-1) for r in reps]).pin_memory(),
        "lens": torch.cat([r["lens_h"] for r in reps]).pin_memory(),
        "slots": torch.cat([r["slots_h"] for r in reps]).pin_memory(),
    }
    # One pinned staging buffer and one device buffer hold every per-step
    # input (256-byte aligned sections), so a step's inputs cross in one copy.
    offs, total = {}, 0
    for k, v in host.items():
        nbytes = v.numel() * v.element_size()
        offs[k] = (total, nbytes)
        total = (total + nbytes + 255) // 256 * 256
    hbuf = torch.empty(total, dtype=torch.uint8).pin_memory()
    dbuf = torch.empty(total, dtype=torch.uint8, device=dev)
    devb = {}
    for k in list(host):
        o, nbytes = offs[k]
        hv = hbuf[o:o + nbytes].view(host[k].dtype).view(host[k].shape)
        hv.copy_(host[k])
        host[k] = hv
        devb[k] = dbuf[o:o + nbytes].view(hv.dtype).view(hv.shape)
    dbuf.copy_(hbuf)
    host["inputs"], devb["inputs"] = hbuf, dbuf
    c0 = reps[0]["case"]
    out_all = torch.empty(R * S, c0.H, c0.D, dtype=c0.out_dtype, device=dev)
    host["out"] = torch.empty(out_all.shape, dtype=out_all.dtype).pin_memory()
    devb["out"] = out_all
    for i, r in enumerate(reps):
        case = r["case"]
        sl = slice(i * S, (i + 1) * S)
        r["q"], r["k_new"], r["v_new"] = devb["q"][sl], devb["k_new"][sl], devb["v_new"][sl]
        r["bt"], r["lens"], r["slots"] = devb["bt"][i], devb["lens"][sl], devb["slots"][sl]
        r["out"] = out_all[sl]
        r["k_pool"], r["v_pool"] = case.k_pool.to(dev), case.v_pool.to(dev)
        r["max_ctx"] = int(r["lens_h"].max())
        r["ws"] = pkv.alloc_decode_workspace(r["q"], r["k_pool"], r["max_ctx"], args.split)
        if case.d2d_pairs is not None:
            r["d2d"] = case.d2d_pairs.to(dev)
            r["h2d"] = case.h2d_pairs.pin_memory()
            r["hk"], r["hv"] = case.host_k_pool.pin_memory(), case.host_v_pool.pin_memory()
    return reps, host, devb


def run_multi_query(args):
    """Causal attention of a chunk of `--multi-query` new tokens per sequence
    over the workload's paged context (the prefill / verification side of the
    decode path).  Prints one JSON line with TFLOP/s of algorithmic work
    (4 * head_dim flops per key per query row and head)."""
    import torch
    from paged_kv_decode_26_gb300 import build as lib_build
    lib_build.build()
    import paged_kv_decode_26_gb300 as pkv
    from paged_kv_decode_26_gb300 import workloads as wl
    case = wl.make_case(args.config, seed=rank_seed(args.config, 0),
                        **({"S": args.seqs} if args.seqs else {}))
    q, qs = wl.multi_query_inputs(case, ("const", args.multi_query))
    dev = torch.device("cuda", 0)
    t = {k: getattr(case, k).to(dev) for k in ("k_pool", "v_pool", "block_tables", "context_lens")}
    qd, qsd = q.to(dev), qs.to(dev)
    out = torch.empty(q.shape[0], case.H, case.D, dtype=case.out_dtype, device=dev)
    ql = (qs[1:] - qs[:-1]).numpy()
    lens = case.context_lens.numpy()
    keys = sum(int(ql[s]) * (int(lens[s]) - int(ql[s])) + int(ql[s]) * (int(ql[s]) + 1) // 2
               for s in range(case.S))
    flops = 4.0 * case.H * case.D * keys
    kv_bytes, kv_unique = wl.kv_bytes(case)

    def call():
        pkv.paged_attn_multi_query(out, qd, qsd, t["k_pool"], t["v_pool"], t["block_tables"],
                                   t["context_lens"], case.scale, int(ql.max()),
                                   case.max_context_len)
    for _ in range(max(3, args.warmup)):
        call()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for a, b in evs:
        a.record()
        call()
        b.record()
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    if pkv.device_errors(clear=True):
        raise RuntimeError("device error flags raised")
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        pass
    peak = float(peaks.get("bf16_tflops", 1900.0))
    tflops = flops / (ms / 1e3) / 1e12
    print(json.dumps({
        "metric": "paged multi-query attention TFLOP/s (causal chunk per sequence)",
        "value": tflops, "unit": "TFLOP/s", "ms_per_call": ms, "steps": args.steps,
        "config": {"workload": workload_name(case, args.config, args.lens), "q_len": args.multi_query,
                   "query_rows": int(qs[-1]), "keys_attended": keys},
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                     "frac": tflops / peak, "peak_kind": "measured cuBLAS bf16 burst "
                     "(MEASURED_PEAKS.json bf16_tflops)",
                     "kv_gbs_unique": kv_unique / (ms / 1e3) / 1e9},
        "dtype": "bf16 in, f32 accumulate"}), flush=True)


def measure(args, rank, world, dev, pkv, wl, *, full):
    """Times one workload (args.config, args.replicas, args.batched, ...):
    the step, then the decode call alone; with `full` also the clock record,
    the end-to-end step through the public API and (continuous-batching
    workload) the device-side allocation.  The block copies of the
    continuous-batching workload are timed either way.  Returns a dict of
    figures; rank 0 holds the job-wide ones."""
    import numpy as np
    import torch
    import torch.distributed as dist

    reps, host, devb = build_replicas(args, rank, dev, pkv, wl, torch, np)
    R = len(reps)
    case = reps[0]["case"]
    S = case.S
    with_swaps = case.d2d_pairs is not None
    stream = torch.cuda.current_stream()
    use_graph = (args.graph or R > 1) and not args.batched
    if args.batched and with_swaps:
        raise SystemExit("--batched does not cover the block copies of the continuous workload")

    def decode(r):
        pkv.paged_attn_decode(r["out"], r["q"], r["k_pool"], r["v_pool"], r["bt"], r["lens"],
                              case.scale, r["max_ctx"], split_tokens=args.split, workspace=r["ws"])

    # The block copies of the continuous-batching step touch only blocks
    # that neither the append nor the decode uses (free targets, read-only
    # sources), and the two copies have disjoint targets and the host copy
    # writes no source of the device copy: each runs on its own side stream,
    # overlapped with the decode and with each other (the step is then bound
    # by the pinned-host copy alone).
    side = (torch.cuda.Stream(), torch.cuda.Stream()) if with_swaps else None

    def step_one(r):
        if with_swaps:
            fork = torch.cuda.Event()
            fork.record(torch.cuda.current_stream())
            for st in side:
                st.wait_event(fork)
            with torch.cuda.stream(side[0]):
                pkv.swap_blocks_kv(r["k_pool"], r["v_pool"], r["hk"], r["hv"], r["h2d"])
            with torch.cuda.stream(side[1]):
                pkv.swap_blocks_kv(r["k_pool"], r["v_pool"], r["k_pool"], r["v_pool"], r["d2d"])
        # append the step's token and decode, in one launch
        pkv.paged_attn_decode_append(r["out"], r["q"], r["k_pool"], r["v_pool"], r["bt"],
                                     r["lens"], case.scale, r["max_ctx"], r["k_new"],
                                     r["v_new"], r["slots"], split_tokens=args.split,
                                     workspace=r["ws"])
        if with_swaps:
            for st in side:
                join = torch.cuda.Event()
                join.record(st)
                torch.cuda.current_stream().wait_event(join)

    def step_eager():
        for r in reps:
            step_one(r)

    def decode_eager():
        for r in reps:
            decode(r)

    # ---- bytes per step (all replicas of this rank)
    es = 2
    kv_read = kv_unique = io_bytes = 0
    launches_per_step = 0
    for r in reps:
        lo, un = wl.kv_bytes(r["case"], r["lens_h"].numpy(), r["bt_h"].numpy())
        kv_read += lo
        kv_unique += un
        io_bytes += (S * case.H * case.D * (es + devb["out"].element_size()) +
                     r["bt"].numel() * 4 + S * 4)
        split_r = args.split or pkv.decode_split_tokens(S, case.H, case.Hk, case.D, case.B,
                                                        r["max_ctx"])
        launches_per_step += 1 + (1 if (r["max_ctx"] + split_r - 1) // split_r > 1 else 0) + \
            (2 if with_swaps else 0)
    split_used = args.split or pkv.decode_split_tokens(S, case.H, case.Hk, case.D, case.B,
                                                       reps[0]["max_ctx"])
    if args.batched:
        # one launch (and one merge if any context splits) for all replicas
        split_b = args.split or pkv.decode_split_tokens(R * S, case.H, case.Hk, case.D, case.B,
                                                        max(r["max_ctx"] for r in reps))
        split_used = split_b
        launches_per_step = 1 + (1 if any((r["max_ctx"] + split_b - 1) // split_b > 1
                                          for r in reps) else 0)
    decode_alg_bytes = kv_unique + io_bytes       # shared prefix rows counted once
    bb = case.B * case.Hk * case.D * es
    swap_bytes = 0
    if with_swaps:
        n_d2d, n_h2d = case.d2d_pairs.shape[0], case.h2d_pairs.shape[0]
        swap_bytes = R * 2 * 2 * bb * (n_d2d + n_h2d)
    # Workloads whose bytes fit in L2 are timed step by step with an L2
    # flush between steps, outside the timed events: a read of a 512 MB
    # buffer, which leaves the L2 holding clean lines of that buffer only (a
    # flush by writing would leave dirty lines whose write-back the timed
    # step would pay for).
    flush_mode = with_swaps or kv_read < 4 * L2_BYTES
    flush_buf = torch.zeros(512 * 1024 * 1024 // 8, dtype=torch.int64, device=dev) \
        if flush_mode else None

    def flush_l2():
        flush_buf.sum()

    def ev():
        return torch.cuda.Event(enable_timing=True)

    pkv.device_errors(clear=True)
    for _ in range(max(3, args.warmup)):
        step_eager()
    torch.cuda.synchronize()

    def fan_out(body):
        """Capture body(r) for every replica on `graph_streams` parallel
        branches (independent replicas need no ordering between them)."""
        cap = torch.cuda.current_stream()
        n_br = max(1, min(args.graph_streams, R))
        branches = [torch.cuda.Stream() for _ in range(n_br)]
        fork = torch.cuda.Event()
        fork.record(cap)
        for b in branches:
            b.wait_event(fork)
        for i, r in enumerate(reps):
            with torch.cuda.stream(branches[i % n_br]):
                body(r)
        for b in branches:
            join = torch.cuda.Event()
            join.record(b)
            cap.wait_event(join)

    if args.batched:
        # every replica is one problem of a single batched launch
        max_ctx_all = max(r["max_ctx"] for r in reps)

        def problem(r, append):
            d = dict(out=r["out"], q=r["q"], k_pool=r["k_pool"], v_pool=r["v_pool"],
                     block_tables=r["bt"], context_lens=r["lens"])
            if append:
                d.update(k_new=r["k_new"], v_new=r["v_new"], slot_mapping=r["slots"])
            return d
        batch_step = pkv.DecodeBatch([problem(r, True) for r in reps], case.scale, max_ctx_all,
                                     split_tokens=args.split)
        batch_dec = pkv.DecodeBatch([problem(r, False) for r in reps], case.scale, max_ctx_all,
                                    split_tokens=args.split)
        run_step, run_decode = batch_step.run, batch_dec.run
        for _ in range(3):
            run_step()
        torch.cuda.synchronize()
    elif use_graph:
        g_step, g_dec = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_step):
            fan_out(step_one)
        with torch.cuda.graph(g_dec):
            fan_out(decode)
        run_step, run_decode = g_step.replay, g_dec.replay
        for _ in range(3):
            run_step()
        torch.cuda.synchronize()
        stream = torch.cuda.current_stream()
    else:
        run_step, run_decode = step_eager, decode_eager

    sampler = ClockSampler(gpu_id_for_smi(torch, dev.index or 0)) if full else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    step_events = [(ev(), ev()) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    if flush_mode:
        for i in range(args.steps):
            flush_l2()
            step_events[i][0].record(stream)
            run_step()
            step_events[i][1].record(stream)
        torch.cuda.synchronize()
        ms = statistics.mean(a.elapsed_time(b) for a, b in step_events)
    else:
        t_start, t_end = ev(), ev()
        t_start.record(stream)
        for i in range(args.steps):
            run_step()
        t_end.record(stream)
        torch.cuda.synchronize()
        ms = t_start.elapsed_time(t_end) / max(1, args.steps)
    if world > 1:
        dist.barrier()
    clocks = None
    if sampler:
        # keep the GPU under the same load until the sampler has ~1.5 s of samples
        while time.perf_counter() - wall0 < 1.5:
            for _ in range(20):
                run_step()
            torch.cuda.synchronize()
        clocks = sampler.stop()

    # ---- the decode call alone (the dominant kernel), timed per launch
    dec_events = [(ev(), ev()) for _ in range(args.steps)]
    for i in range(args.steps):
        if flush_mode:
            flush_l2()
        dec_events[i][0].record(stream)
        run_decode()
        dec_events[i][1].record(stream)
    torch.cuda.synchronize()
    dec_ms = statistics.mean(a.elapsed_time(b) for a, b in dec_events)

    ms, dec_ms = reduce_over_ranks([ms, dec_ms], "max", dist, world, dev)
    total_kv, = reduce_over_ranks([kv_read], "sum", dist, world, dev)
    errors = pkv.device_errors(clear=True)
    if errors:
        raise RuntimeError(f"device error flags 0x{errors:x} raised during the benchmark")

    # ---- swap_blocks alone (continuous-batching workload), with copy references
    swap = None
    if with_swaps and rank == 0:
        r0 = reps[0]
        d2d_t, h2d_t, d2d_ref_t, h2d_ref_t, d2d_two_t = [], [], [], [], []
        n_ref_d2d, n_ref_h2d = n_d2d * bb, n_h2d * bb
        src_d = torch.empty(n_ref_d2d, dtype=torch.uint8, device=dev)
        dst_d = torch.empty(n_ref_d2d, dtype=torch.uint8, device=dev)
        src_h = torch.empty(n_ref_h2d, dtype=torch.uint8).pin_memory()
        dst_h = torch.empty(n_ref_h2d, dtype=torch.uint8, device=dev)
        for i in range(max(20, min(args.steps, 200))):
            for fn, acc in (
                    (lambda: pkv.swap_blocks_kv(r0["k_pool"], r0["v_pool"], r0["k_pool"],
                                                r0["v_pool"], r0["d2d"]), d2d_t),
                    (lambda: (pkv.swap_blocks(r0["k_pool"], r0["k_pool"], r0["d2d"]),
                              pkv.swap_blocks(r0["v_pool"], r0["v_pool"], r0["d2d"])), d2d_two_t),
                    (lambda: pkv.swap_blocks_kv(r0["k_pool"], r0["v_pool"], r0["hk"], r0["hv"],
                                                r0["h2d"]), h2d_t),
                    (lambda: (dst_d.copy_(src_d, non_blocking=True),
                              dst_d.copy_(src_d, non_blocking=True)), d2d_ref_t),
                    (lambda: (dst_h.copy_(src_h, non_blocking=True),
                              dst_h.copy_(src_h, non_blocking=True)), h2d_ref_t)):
                flush_l2()
                a, b = ev(), ev()
                a.record(stream)
                fn()
                b.record(stream)
                torch.cuda.synchronize()
                acc.append(a.elapsed_time(b))
        peak_copy, _ = measured_peak()
        moved_d2d, moved_h2d = 2 * n_d2d * bb, 2 * n_h2d * bb       # K and V
        d2d_ms, h2d_ms = statistics.median(d2d_t), statistics.median(h2d_t)
        d2d_ref_ms, h2d_ref_ms = statistics.median(d2d_ref_t), statistics.median(h2d_ref_t)
        # the asymptote: 8192 pairs of the same block size (1 GB moved)
        n_big = 8192
        big_k = torch.empty(2 * n_big, bb, dtype=torch.uint8, device=dev)
        big_v = torch.empty(2 * n_big, bb, dtype=torch.uint8, device=dev)
        perm = torch.randperm(2 * n_big, generator=torch.Generator().manual_seed(5))
        big_pairs = torch.stack([perm[:n_big], perm[n_big:]], 1).to(dev)
        big_src = torch.empty(2 * n_big * bb, dtype=torch.uint8, device=dev)
        big_dst = torch.empty_like(big_src)
        big_t, big_ref_t = [], []
        for i in range(20):
            for fn, acc in ((lambda: pkv.swap_blocks_kv(big_k, big_v, big_k, big_v, big_pairs),
                             big_t),
                            (lambda: big_dst.copy_(big_src, non_blocking=True), big_ref_t)):
                flush_l2()
                a, b = ev(), ev()
                a.record(stream)
                fn()
                b.record(stream)
                torch.cuda.synchronize()
                acc.append(a.elapsed_time(b))
        big_ms, big_ref_ms = statistics.median(big_t), statistics.median(big_ref_t)
        moved_big = 2 * 2 * n_big * bb                             # K and V, read + write
        del big_k, big_v, big_src, big_dst
        swap = {
            "d2d_8192_pairs": {"pairs": n_big, "block_bytes": bb, "ms_k_and_v": big_ms,
                               "gbs_read_write": moved_big / (big_ms / 1e3) / 1e9,
                               "vs_measured_copy_peak":
                                   moved_big / (big_ms / 1e3) / 1e9 / peak_copy,
                               "contiguous_copy_same_bytes_gbs_read_write":
                                   moved_big / (big_ref_ms / 1e3) / 1e9},
            "d2d": {"pairs": n_d2d, "block_bytes": bb, "ms_k_and_v": d2d_ms,
                    "gbs_read_write": 2 * moved_d2d / (d2d_ms / 1e3) / 1e9,
                    "vs_measured_copy_peak": 2 * moved_d2d / (d2d_ms / 1e3) / 1e9 / peak_copy,
                    "contiguous_copy_same_bytes_gbs_read_write":
                        2 * moved_d2d / (d2d_ref_ms / 1e3) / 1e9,
                    "vs_contiguous_copy": d2d_ref_ms / d2d_ms,
                    "ms_two_calls_swap_blocks": statistics.median(d2d_two_t)},
            "h2d": {"pairs": n_h2d, "ms_k_and_v": h2d_ms,
                    "gbs": moved_h2d / (h2d_ms / 1e3) / 1e9,
                    "memcpy_h2d_same_bytes_gbs": moved_h2d / (h2d_ref_ms / 1e3) / 1e9,
                    "vs_memcpy": h2d_ref_ms / h2d_ms},
            "timing": "median of per-call CUDA events, L2 flushed (512 MB read) before each; "
                      "K and V in one swap_blocks_kv launch",
        }
        del src_d, dst_d, src_h, dst_h

    # ---- the step's allocation on the device (continuous-batching workload):
    # pkv_device_append_slots from the pre-step state, restored before each
    # timed call
    dev_alloc = None
    if full and with_swaps and rank == 0:
        r0 = reps[0]
        c0 = r0["case"]
        refs = torch.zeros(c0.num_blocks, dtype=torch.int32)
        bt0 = c0.block_tables
        mbd = r0["bt_h"].shape[1]
        bt_init = torch.full((S, mbd), -1, dtype=torch.int32)
        bt_init[:, :bt0.shape[1]] = bt0
        refs.index_add_(0, bt0[bt0 >= 0].long(), torch.ones(int((bt0 >= 0).sum()),
                                                            dtype=torch.int32))
        dm = pkv.DeviceBlockManager(refs, c0.B)
        saved = (dm.ref_counts.clone(), dm.free_ids.clone(), dm.state.clone())
        bt_d0, lens_d0 = bt_init.to(dev), c0.context_lens.to(dev)
        bt_d, lens_d = bt_d0.clone(), lens_d0.clone()
        slots_d = torch.empty(S, dtype=torch.int64, device=dev)
        times = []
        for i in range(50):
            dm.ref_counts.copy_(saved[0])
            dm.free_ids.copy_(saved[1])
            dm.state.copy_(saved[2])
            bt_d.copy_(bt_d0)
            lens_d.copy_(lens_d0)
            a, b = ev(), ev()
            a.record(stream)
            dm.append_slots(bt_d, lens_d, slots_d)
            b.record(stream)
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b))
        same = torch.equal(slots_d.cpu(), reps[0]["slots_h"]) and \
            torch.equal(bt_d.cpu(), reps[0]["bt_h"])
        dev_alloc = {"us": statistics.median(times) * 1e3, "sequences": S,
                     "timing": "events around one eager call, launch latency included",
                     "matches_host_manager": bool(same)}

    # ---- end to end through the public API with host buffers
    e2e = None
    if full:
        h2d_bytes = host["inputs"].numel()        # the staging buffer, copied whole
        d2h_bytes = host["out"].numel() * host["out"].element_size()

        if R == 1 and not with_swaps and not use_graph and not args.batched:
            # the library's one-call step from host memory: the staging
            # buffer in, append + decode, the output back, the stream synced
            r0, e2e_call = reps[0], "HostStep.run (paged_attn_decode_append_host)"
            host_step = pkv.HostStep(
                [(host["inputs"], devb["inputs"])], host["out"], r0["out"], r0["q"],
                r0["k_pool"], r0["v_pool"], r0["bt"], r0["lens"], case.scale, r0["max_ctx"],
                r0["k_new"], r0["v_new"], r0["slots"], split_tokens=args.split,
                workspace=r0["ws"], stream=stream)
            e2e_step = host_step.run
        else:
            e2e_call = "copy in, the step, copy out, stream synchronize"

            def e2e_step():
                devb["inputs"].copy_(host["inputs"], non_blocking=True)
                run_step()
                host["out"].copy_(devb["out"], non_blocking=True)
                stream.synchronize()

        for _ in range(3):
            e2e_step()
        n_e2e = max(1, min(args.e2e_steps, args.steps))
        if world > 1:
            dist.barrier()
        e2e_times = []
        for i in range(n_e2e):
            if flush_mode:
                flush_l2()
            a, b = ev(), ev()
            a.record(stream)
            e2e_step()
            b.record(stream)
            torch.cuda.synchronize()
            e2e_times.append(a.elapsed_time(b))
        e2e_ms = statistics.mean(e2e_times)
        e2e_ms, = reduce_over_ranks([e2e_ms], "max", dist, world, dev)
        e2e = {"value": job_gbs(total_kv, e2e_ms), "unit": "GB/s",
               "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
               "ms_per_step": e2e_ms, "steps": n_e2e, "call": e2e_call}

    return dict(case=case, reps=reps, R=R, S=S, ms=ms, dec_ms=dec_ms, kv_read=kv_read,
                kv_unique=kv_unique, io_bytes=io_bytes, total_kv=total_kv,
                decode_alg_bytes=decode_alg_bytes, split_used=split_used,
                launches_per_step=launches_per_step, flush_mode=flush_mode, use_graph=use_graph,
                with_swaps=with_swaps, swap_bytes=swap_bytes, swap=swap, dev_alloc=dev_alloc,
                clocks=clocks, e2e=e2e)


def release(res):
    """Drops a measured workload's device and pinned buffers."""
    import gc
    import torch
    res.pop("reps", None)
    gc.collect()
    torch.cuda.empty_cache()


# Other stated workloads measured after the headline one, each as
# (label, config, replicas, batched).  The tiny workload reads 0.9 MB per
# step, so it is reported per launch and as 1100 independent problems in
# one batched launch (~1 GB of distinct pools per step).
PER_CONFIG = [("tiny_per_launch", 1, 1, False), ("tiny_batched_x1100", 1, 1100, True),
              ("gqa_prefix", 3, 1, False), ("long_context", 4, 1, False),
              ("continuous", 5, 1, False)]


def per_config_entry(args, res, peak, cpu_budget):
    """Summary of one extra workload: decode GB/s and roofline fraction,
    step GB/s, sequence-steps per second, and the threaded oracle's GB/s on
    the same inputs (one replica's whole step)."""
    case = res["case"]
    dec_gbs = res["decode_alg_bytes"] / (res["dec_ms"] / 1e3) / 1e9
    e = {"workload": workload_name(case, args.config),
         "replicas": res["R"], "launch": ("batched" if args.batched else
                                          "graph" if res["use_graph"] else "eager"),
         "decode_ms": res["dec_ms"], "decode_gbs": dec_gbs,
         "roofline_frac": dec_gbs / peak,
         "decode_bytes": res["decode_alg_bytes"],
         "step_ms": res["ms"], "step_gbs": job_gbs(res["total_kv"], res["ms"]),
         "seq_steps_per_s": res["R"] * res["S"] / (res["ms"] / 1e3),
         "split_tokens": res["split_used"],
         "l2": "flushed before every step" if res["flush_mode"] else "inputs larger than L2"}
    if res["swap"]:
        e["swap_blocks"] = res["swap"]
    if cpu_budget > 0:
        r0 = res["reps"][0]
        kv, secs, runs, thr = oracle_step_seconds(case, r0["lens_h"], r0["bt_h"], cpu_budget)
        e["oracle"] = {"gbs": kv / secs / 1e9, "threads": thr, "runs": runs,
                       "sample": "one replica's whole step, fp64 two-pass oracle"}
    return e


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
        return
    if args.multi_query:
        run_multi_query(args)
        return

    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from paged_kv_decode_26_gb300 import build as lib_build
    if rank == 0:
        lib_build.build()
    if world > 1:
        dist.barrier()
    import paged_kv_decode_26_gb300 as pkv
    from paged_kv_decode_26_gb300 import workloads as wl

    res = measure(args, rank, world, dev, pkv, wl, full=True)
    case, R, S = res["case"], res["R"], res["S"]

    # ---- CPU baseline: the oracle on the step (rank 0, N=1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle import build as ob
        ob.build()
        r0 = res["reps"][0]
        kv, secs, runs, thr = oracle_step_seconds(case, r0["lens_h"], r0["bt_h"],
                                                  args.cpu_budget)
        cpu = {"value": kv / secs / 1e9, "unit": "GB/s", "cores": thr, "kind": "oracle",
               "sample": f"the whole step ({S} sequences, all {case.H} heads, "
                         f"{kv / 1e6:.1f} MB of K/V), fp64 two-pass oracle threaded over "
                         f"{thr} host threads, median of {runs} runs"}

    peak, peak_kind = measured_peak()
    name = workload_name(case, args.config, args.lens)
    value = job_gbs(res["total_kv"], res["ms"])
    achieved = res["decode_alg_bytes"] / (res["dec_ms"] / 1e3) / 1e9
    logical_gbs = (res["kv_read"] + res["io_bytes"]) / (res["dec_ms"] / 1e3) / 1e9
    line = None
    if rank == 0:
        line = {
            "metric": METRIC,
            "value": value,
            "unit": "GB/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": res["ms"],
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f32",
            "data": "synthetic",
            "seq_steps_per_s": R * S * world / (res["ms"] / 1e3),
            "kv_bytes_per_step_all_gpus": res["total_kv"],
            "config": {
                "workload": name,
                "step": "paged_attn_decode_append (append 1 token/seq, then decode: one call)" +
                        (" + swap_blocks_kv D2D and pinned-H2D on two side streams, overlapped"
                         if res["with_swaps"] else ""),
                "replicas_per_gpu": R,
                "launch": ("one batched launch per step for all replicas "
                           "(paged_attn_decode_batched)" if args.batched else
                           f"one CUDA graph per step, replicas on {min(args.graph_streams, R)} "
                           "parallel branches" if res["use_graph"] else "eager"),
                "num_seqs_per_gpu": R * S,
                "kv_bytes_per_step_per_gpu": res["kv_read"],
                "kv_unique_bytes_per_step_per_gpu": res["kv_unique"],
                "split_tokens": res["split_used"],
                "storage_dtype": str(case.dtype).replace("torch.", ""),
                "out_dtype": str(case.out_dtype).replace("torch.", ""),
                "l2": ("inputs larger than L2 (%.2f GB of K/V vs 129 MB), no flush"
                       % (res["kv_read"] / 1e9) if not res["flush_mode"] else
                       "L2 flushed (512 MB read) before every step, outside the timed events"),
                "parallelism": f"replicas x{world} (sequences per GPU independent)",
            },
            "roofline": {
                "bound": "hbm",
                "achieved": achieved,
                "peak": peak,
                "unit": "GB/s",
                "frac": achieved / peak,
                "traffic": committed_traffic(name) if R == 1 else None,
                "kernel": "paged_attn_decode (decode kernel + split merge), CUDA events per call" +
                          (" (all replicas, one graph)" if res["use_graph"] else ""),
                "bytes": "unique K/V rows read (shared prefix rows once) + q + out + tables",
                "logical_gbs": logical_gbs,
                "algorithmic_bytes_per_launch": res["decode_alg_bytes"],
                "ms_per_launch": res["dec_ms"],
                "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                if peak_kind == "measured" else "fallback 6.8 TB/s",
            },
            "clocks": res["clocks"],
            "e2e": res["e2e"],
            "gpu_launches": res["launches_per_step"] * args.steps,
            "cpu_baseline": cpu,
        }
        if res["with_swaps"]:
            line["config"]["swap_bytes_per_step"] = res["swap_bytes"]
            line["swap_blocks"] = res["swap"]
            line["device_append_slots"] = res["dev_alloc"]
    release(res)

    # ---- the other stated workloads (single GPU, headline workload only)
    if world == 1 and not args.no_per_config and args.config == 2 and not args.seqs \
            and not args.lens and R == 1 and not args.batched and not args.graph:
        per = {}
        for label, cfg, reps_n, batched in PER_CONFIG:
            sub = argparse.Namespace(**vars(args))
            sub.config, sub.replicas, sub.batched, sub.graph = cfg, reps_n, batched, False
            sub.split = 0
            sub.steps = min(args.steps, 200)
            r = measure(sub, rank, world, dev, pkv, wl, full=False)
            per[label] = per_config_entry(sub, r, peak,
                                          0.0 if args.no_cpu_baseline else min(args.cpu_budget,
                                                                               6.0))
            release(r)
        line["per_config"] = per
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
