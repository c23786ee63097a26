#!/usr/bin/env python3
"""Decode-attention benchmark: KV-cache GB/s read and decode-attention calls/s.

One step = one ifa_run call (split-KV partial kernel + combine kernel) over one
batch of the workload.  Default workload: GQA decode against a padded cache,
B=16, N=32, KV_N=8, D=128, BSH bf16, Smax=4096, lengths ~ U{1..4096}, bool mask
(B,1,1,S) true past each length.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Prints one JSON line on rank 0.  ``value`` is algorithmic bytes (valid-token K
and V, query, output, mask over the valid windows, block-table entries used,
antiquant parameters) per step divided by the device time per step, summed over
ranks (weak scaling: every rank runs its own copy of the workload).
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from kv_cache_incremental_split_gb300 import inputs as gen  # noqa: E402

METRIC = "KV-cache GB/s read (% of GB300 HBM peak); decode attention calls/sec"
UNIT = "GB/s"
L2_BYTES = 129 * 1024 * 1024

WORKLOADS = {
    "gqa_padded": ("GQA decode, padded cache: B=16 N=32 KV_N=8 D=128 BSH bf16 Smax=4096, "
                   "lengths U{1..4096}, bool mask (B,1,1,S) true past each length, scale 1/sqrt(128)"),
    "tiny_mha": "MHA decode: B=1 N=KV_N=8 D=64 BNSD fp16 S=128, length 128, scale 1/8",
    "paged_gqa": ("paged GQA decode: B=64 N=32 KV_N=8 D=128 bf16, blockSize 128, cache (blocknum,KV_N,128,D), "
                  "random block table, lengths U{512..32768}"),
    "int8_leftpad": ("int8 KV antiquant + left padding: B=32 N=64 KV_N=8 D=128 fp16 query, BNSD int8 K/V, "
                     "per-channel scale/offset, Smax=8192, lengths U{256..8192}, pad Smax-len-U{0..64}"),
    "paged_gqa_small": ("paged GQA decode, profiling size: B=64 N=32 KV_N=8 D=128 bf16, blockSize 128, "
                        "random block table, lengths U{512..4096}"),
}


def make_case(name: str, seed: int) -> gen.IfaCase:
    if name == "paged_gqa_small":
        return gen.paged_gqa(seed, len_hi=4096)
    return {"gqa_padded": gen.gqa_padded, "tiny_mha": gen.tiny_mha, "paged_gqa": gen.paged_gqa,
            "int8_leftpad": gen.int8_leftpad}[name](seed)


# ------------------------------------------------------------------------ algorithmic bytes

def windows(case: gen.IfaCase):
    """(start, length) of every batch's valid window, as the pages define it."""
    B = case.B
    lens = case.actual_seq_lengths if case.actual_seq_lengths is not None else np.full(B, case.max_seq_len)
    out = []
    for b in range(B):
        L = int(lens[b])
        if case.kv_padding_size is not None:
            pads = case.kv_padding_size.reshape(-1)
            pad = max(int(pads[0 if pads.size == 1 else b]), 0)
            st, en = case.max_seq_len - pad - L, case.max_seq_len - pad
            out.append((0, 0) if (st < 0 or en < 0) else (st, L))
        else:
            out.append((0, L))
    return out


def algorithmic_bytes(case: gen.IfaCase) -> int:
    kv_es = 1 if case.kv_dtype == "int8" else 2
    kvn = case.num_kv_heads or case.num_heads
    toks = sum(L for _, L in windows(case))
    total = 2 * toks * kvn * case.D * kv_es                 # K and V of valid tokens
    total += 2 * case.B * case.num_heads * case.D * 2       # query and output
    if case.atten_mask is not None:
        mN = case.atten_mask.shape[1]
        total += toks * mN if case.atten_mask.shape[0] > 1 else max(L for _, L in windows(case)) * mN
    if case.block_table is not None:
        total += sum(-(-L // case.block_size) for _, L in windows(case)) * 4
    if case.antiquant_scale is not None:
        total += 2 * case.antiquant_scale.nbytes
    return int(total)


# ------------------------------------------------------------------------ clocks

CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu=timestamp,{CLOCK_QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self):
        rows = []
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(f[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                rows.append((ts, float(f[2]), float(f[3]), f[6:10]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        t0 = (self.t0 or 0) - 1.0
        t1 = (self.t1 or 0) + 1.0
        inside = [r for r in rows if t0 <= r[0] <= t1] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside)}


# ------------------------------------------------------------------------ helpers

def kernel_sources_digest() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "kv_cache_incremental_split_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh")):
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(f.encode())
                h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch of the partial kernel from a committed ncu summary,
    valid only while the kernel sources are unchanged since the capture."""
    path = os.path.join(ROOT, "profiles", f"decode_kernel_{workload}.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("kernel_sources_digest") != kernel_sources_digest():
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(local_elapsed_ms: float, local_bytes: float, world: int):
    """Max time over ranks and total bytes over ranks (identity when world == 1)."""
    if world == 1:
        return local_elapsed_ms, local_bytes
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([local_elapsed_ms], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    b = torch.tensor([local_bytes], dtype=torch.float64, device=dev)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return float(t.item()), float(b.item())


# ------------------------------------------------------------------------ CPU oracle baseline

def oracle_sample(case: gen.IfaCase, budget_s: float, start_batch: int = 0):
    """Time the CPU oracle, batch by batch, for about `budget_s` seconds."""
    import oracle  # test infrastructure: only the CPU-baseline leg of the benchmark uses it
    from copy import copy
    fmt = {"contig": oracle.CONTIG, "paged_nbsd": oracle.PAGED_NBSD, "paged_bsh": oracle.PAGED_BSH}
    aq = {"none": oracle.AQ_NONE, "per_channel": oracle.AQ_PER_CHANNEL, "per_tensor": oracle.AQ_PER_TENSOR}
    done, nbytes, t_used = [], 0, 0.0
    b = start_batch % case.B
    while True:
        c = copy(case)
        sel = np.array([b])
        c.query = case.query[sel]
        if case.kv_format == "contig":
            c.key, c.value = case.key[sel], case.value[sel]
        if case.block_table is not None:
            c.block_table = case.block_table[sel]
        if case.atten_mask is not None and case.atten_mask.shape[0] > 1:
            c.atten_mask = case.atten_mask[sel]
        if case.actual_seq_lengths is not None:
            c.actual_seq_lengths = case.actual_seq_lengths[sel]
        if case.kv_padding_size is not None and case.kv_padding_size.size > 1:
            c.kv_padding_size = case.kv_padding_size[sel]
        t = time.perf_counter()
        oracle.ifa_ref(c.query, c.key, c.value, num_heads=c.num_heads, num_kv_heads=c.num_kv_heads,
                       scale=c.scale, layout=c.layout, kv_format=fmt[c.kv_format], block_size=c.block_size,
                       block_table=c.block_table, atten_mask=c.atten_mask,
                       actual_seq_lengths=c.actual_seq_lengths, kv_padding_size=c.kv_padding_size,
                       antiquant=aq[c.antiquant], antiquant_scale=c.antiquant_scale,
                       antiquant_offset=c.antiquant_offset)
        t_used += time.perf_counter() - t
        nbytes += algorithmic_bytes(c)
        done.append(b)
        b = (b + 1) % case.B
        if t_used >= budget_s or len(done) >= case.B:
            break
    return nbytes, t_used, done


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    case = make_case(args.workload, args.seed)
    per_step = args.ref_step_seconds
    for w in range(args.warmup):
        oracle_sample(case, per_step, start_batch=w)
    total_b, total_t, batches = 0, 0.0, 0
    for s in range(args.steps):
        nb, t, done = oracle_sample(case, per_step, start_batch=args.warmup + s)
        total_b += nb
        total_t += t
        batches += len(done)
    value = total_b / total_t / 1e9
    sample = (f"each step: the oracle on whole batches of the workload for about {per_step} s "
              f"({batches} batch rows over {args.steps} steps, {total_b / 1e6:.1f} MB algorithmic)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / max(1, args.steps),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOADS[args.workload], "seed": args.seed},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------------------ GPU arm

def run_gpu(args):
    import torch

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    from kv_cache_incremental_split_gb300 import build as libbuild
    libbuild.build()
    from kv_cache_incremental_split_gb300.ifa import IncreFlashAttention

    case = make_case(args.workload, args.seed + rank)
    alg = algorithmic_bytes(case)

    def dev_t(a):
        if a is None:
            return None
        t = torch.from_numpy(np.ascontiguousarray(a))
        return (t.view(torch.bfloat16) if a.dtype == np.uint16 else t).to(dev)

    m = case.atten_mask
    op = IncreFlashAttention(
        batch=case.B, num_heads=case.num_heads, num_kv_heads=case.num_kv_heads, head_dim=case.D,
        max_seq_len=case.max_seq_len, dtype=case.q_dtype, kv_dtype=case.kv_dtype, layout=case.layout,
        kv_format=case.kv_format, block_size=case.block_size,
        block_num=case.key.shape[0] if case.kv_format != "contig" else 0,
        block_table_cols=case.block_table.shape[1] if case.block_table is not None else 0,
        mask_shape=None if m is None else m.shape, mask_dtype="bool", antiquant=case.antiquant,
        kv_padding=case.kv_padding_size is not None, scale=case.scale, device=dev)

    q, k, v = dev_t(case.query), dev_t(case.key), dev_t(case.value)
    mask, bt = dev_t(case.atten_mask), dev_t(case.block_table)
    sc, of = dev_t(case.antiquant_scale), dev_t(case.antiquant_offset)
    kv_bytes = k.numel() * k.element_size() + v.numel() * v.element_size()
    # Rotate through enough key/value copies that the valid bytes streamed between two
    # uses of one copy exceed L2 several times (inputs larger than L2: no flush needed).
    copies = max(1, min(8, math.ceil(6 * L2_BYTES / max(1, alg))))
    ks = [k] + [k.clone() for _ in range(copies - 1)]
    vs = [v] + [v.clone() for _ in range(copies - 1)]
    outs = [torch.empty_like(q) for _ in range(copies)]
    stream = torch.cuda.Stream(device=dev)

    def call(i):
        return op(q, ks[i], vs[i], atten_mask=mask, actual_seq_lengths=case.actual_seq_lengths,
                  kv_padding_size=case.kv_padding_size, block_table=bt, antiquant_scale=sc,
                  antiquant_offset=of, out=outs[i], stream=stream)

    with torch.cuda.stream(stream):
        for w in range(max(args.warmup, 3)):
            call(w % copies)
        stream.synchronize()
        launches_per_call = op.last_launch_count()
        graphs = []
        for i in range(copies):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                call(i)
            graphs.append(g)
        for i in range(copies):
            graphs[i].replay()
        stream.synchronize()

    # eager calls/s (host-launched, no graph), for reference only
    with torch.cuda.stream(stream):
        n_eager = min(args.steps, 200)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        stream.synchronize()
        e0.record(stream)
        for i in range(n_eager):
            call(i % copies)
        e1.record(stream)
        e1.synchronize()
        eager_ms = e0.elapsed_time(e1) / n_eager

    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    smi_index = vis.split(",")[local] if vis and len(vis.split(",")) > local else str(local)
    sampler = ClockSampler(smi_index)
    with sampler:
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        sampler.mark_start()
        start.record(stream)
        with torch.cuda.stream(stream):
            for s in range(args.steps):
                graphs[s % copies].replay()
        end.record(stream)
        end.synchronize()
        torch.cuda.synchronize()
        sampler.mark_end()
    elapsed = start.elapsed_time(end)
    max_elapsed, total_bytes = aggregate(elapsed, float(alg) * args.steps, world)
    ms_per_step = max_elapsed / args.steps
    value = total_bytes / (max_elapsed * 1e-3) / 1e9
    local_gbs = alg / (elapsed / args.steps * 1e-3) / 1e9

    # ---- end to end through the public API: pinned host inputs -> device -> ifa_run -> host output
    host = {n: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
            for n, a in (("q", case.query), ("k", case.key), ("v", case.value), ("mask", case.atten_mask),
                         ("bt", case.block_table), ("sc", case.antiquant_scale), ("of", case.antiquant_offset))
            if a is not None}
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d_in = {n: torch.empty(t.shape, dtype=t.dtype, device=dev) for n, t in host.items()}
    out_host = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    d2h = out_host.numel() * out_host.element_size()
    n_e2e = max(3, min(args.steps, 20))

    def e2e_step():
        for n, t in host.items():
            d_in[n].copy_(t, non_blocking=True)
        qq = d_in["q"].view(torch.bfloat16) if case.query.dtype == np.uint16 else d_in["q"]
        kk = d_in["k"].view(torch.bfloat16) if case.key.dtype == np.uint16 else d_in["k"]
        vv = d_in["v"].view(torch.bfloat16) if case.value.dtype == np.uint16 else d_in["v"]
        sc_ = d_in.get("sc")
        of_ = d_in.get("of")
        if sc_ is not None and case.antiquant_scale.dtype == np.uint16:
            sc_, of_ = sc_.view(torch.bfloat16), of_.view(torch.bfloat16)
        o = op(qq, kk, vv, atten_mask=d_in.get("mask"), actual_seq_lengths=case.actual_seq_lengths,
               kv_padding_size=case.kv_padding_size, block_table=d_in.get("bt"), antiquant_scale=sc_,
               antiquant_offset=of_, stream=stream)
        out_host.copy_(o, non_blocking=True)

    with torch.cuda.stream(stream):
        e2e_step()
        stream.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        a1.record(stream)
        a1.synchronize()
    e2e_ms = a0.elapsed_time(a1) / n_e2e
    e2e_max, e2e_bytes = aggregate(e2e_ms, float(alg), world)
    e2e_value = e2e_bytes / (e2e_max * 1e-3) / 1e9

    # ---- CPU oracle baseline on a bounded sample (rank 0, single GPU runs only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        nb, t, done = oracle_sample(case, args.cpu_seconds)
        cpu = {"value": nb / t / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"batch rows {done} of the same workload ({nb / 1e6:.1f} MB algorithmic, "
                         f"{t:.1f} s, single-threaded C, float64)"}

    peak, peak_kind = measured_peaks()
    clocks = sampler.summary()
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": case.q_dtype if case.kv_dtype != "int8" else "int8-kv/" + case.q_dtype,
            "data": "synthetic",
            "config": {"workload": WORKLOADS[args.workload], "seed": args.seed,
                       "algorithmic_bytes_per_step": alg,
                       "l2": f"inputs larger than L2: {copies} rotating key/value copies "
                             f"({copies * kv_bytes / 1e6:.0f} MB) ",
                       "launch": "CUDA graph replay of one ifa_run call per step",
                       "parallelism": f"replica x{world}" if world > 1 else "single GPU"},
            "calls_per_sec": world * 1e3 / ms_per_step,
            "calls_per_sec_eager": 1e3 / eager_ms,
            "pct_of_hbm_peak": 100.0 * local_gbs / peak,
            "roofline": {"bound": "hbm", "achieved": local_gbs, "peak": peak, "unit": "GB/s",
                         "frac": local_gbs / peak, "peak_kind": peak_kind,
                         "timed": "ifa_run (split-KV partial kernel + combine kernel) per step, CUDA events",
                         "traffic": recorded_traffic(args.workload)},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": args.steps * launches_per_call,
            "clocks": clocks,
        }
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


def parse(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="gqa_padded", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-step-seconds", type=float, default=0.5)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args(argv)


def main(argv=None):
    args = parse(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
