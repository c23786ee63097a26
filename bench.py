#!/usr/bin/env python3
"""Decode-attention benchmark: KV-cache GB/s read and decode-attention calls/s.

One step = one library call (ifa_run, or sfa_run for the sparse workloads) over
one batch of the workload.  Default workload: paged GQA decode, B=64, N=32,
KV_N=8, D=128, bf16, blockSize 128, cache (blocknum, KV_N, 128, D) through a
random block table, lengths ~ U{512..32768} (about 4.4 GB of keys and values
per call: the largest single-GPU workload).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Prints one JSON line on rank 0.  ``value`` is algorithmic bytes per step
(key/value rows of the valid tokens, query, output, mask over the valid
windows, block-table entries and sparse indices used, antiquant parameters)
divided by the device time per step, summed over ranks (weak scaling: every
rank runs its own rank-seeded copy of the workload).  The K timed steps are
timed as one region, R times over (at least --repeats, and at least
--min-timed-seconds of regions in all); ``ms_per_step`` is the median region
time / K, with the 10th and 90th percentiles beside it.  With --gpus N > 1 and
no WORLD_SIZE in the environment, the script relaunches itself under
torch.distributed.run with N ranks, one per GPU.
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
    "gqa_tensorlist": ("GQA decode, key/value as one tensor per batch: B=16 N=32 KV_N=8 D=128 BSH bf16, "
                       "tensor b of batch 1 holding len_b + U{0..256} tokens, lengths U{1..4096}, bool mask "
                       "(B,1,1,4096) true past each length, scale 1/sqrt(128)"),
    "paged_gqa_small": ("paged GQA decode, profiling size: B=64 N=32 KV_N=8 D=128 bf16, blockSize 128, "
                        "random block table, lengths U{512..4096}"),
    "sfa_mla": ("sparse MLA-absorb decode: B=32 Q_N=128 KV_N=1 D=512+rope 64 bf16, PA_BSND block 64, "
                "KV length 32768, sparse_indices (B,1,1,2048) with U{1024..2048} valid then -1, scale 1/sqrt(576)"),
    "sfa_mla_small": ("sparse MLA-absorb decode, profiling size: B=8 Q_N=128 D=512+64 bf16, block 64, "
                      "KV length 8192, 2048 indices with U{1024..2048} valid"),
    "sfa_mla_vk": ("sparse MLA-absorb decode with value = key (one cache tensor serves both): B=32 Q_N=128 KV_N=1 "
                   "D=512+rope 64 bf16, PA_BSND block 64, KV length 32768, sparse_indices (B,1,1,2048) with "
                   "U{1024..2048} valid then -1, scale 1/sqrt(576)"),
    "sfa_mla_blockwise": ("sparse MLA-absorb decode, block-wise: B=32 Q_N=128 D=512+64 bf16, PA_BSND block 64, "
                          "KV length 32768, sparse_block_size 16, 128 block indices with U{64..128} valid then -1"),
    "sfa_mla_mtp": ("sparse MLA-absorb decode, two query tokens (multi-token prediction): B=32 Q_S=2 Q_N=128 "
                    "D=512+64 bf16, PA_BSND block 64, KV length 32768, sparse_mode 3 (right-down causal), "
                    "sparse_indices (B,2,1,2048) with U{1024..2048} valid per row then -1"),
    "kv_append_paged": ("KV-cache append (the step before the attention): B=64 KV_N=8 D=128 bf16 new token rows into "
                        "a paged (blocknum, 8, 128, 128) cache through a random block table, at each batch's "
                        "length U{512..4096} minus the step number mod 8"),
    "kv_append_int8": ("KV-cache append with int8 quantisation: B=32 KV_N=8 D=128 fp16 new token rows into a BNSD "
                       "int8 cache (Smax 8192) with per-channel scale U[0.005,0.02] and offset U[-4,4], at "
                       "positions U{256..8191} minus the step number mod 8"),
}


def make_case(name: str, seed: int):
    if name == "paged_gqa_small":
        return gen.paged_gqa(seed, len_hi=4096)
    if name == "sfa_mla":
        return gen.sfa_mla(seed)
    if name == "sfa_mla_small":
        return gen.sfa_mla(seed, B=8, kv_len=8192)
    if name == "sfa_mla_vk":
        c = gen.sfa_mla(seed)
        c.value = c.key  # the same array: the call receives one tensor as key and value
        return c
    if name == "sfa_mla_blockwise":
        return gen.sfa_mla(seed, sparse_size=128, nvalid_lo=64, nvalid_hi=128, sparse_block_size=16)
    if name == "sfa_mla_mtp":
        return gen.sfa_mla(seed, Q_S=2, sparse_mode=3)
    if name == "gqa_tensorlist":
        return gen.tensorlist_from(gen.gqa_padded(seed), seed, extra_hi=256)
    if name == "kv_append_paged":
        return gen.kv_append_paged(seed)
    if name == "kv_append_int8":
        return gen.kv_append_int8(seed)
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


def sfa_valid_counts(case: gen.SfaCase):
    """Selected tokens per (batch, query token) row, shape (B * Q_S,): each index covers
    sparse_block_size tokens; those below the row's key limit count (the length, cut to
    len - qlen + s + 1 under sparse_mode 3, none for query tokens at or past qlen)."""
    sbs = case.sparse_block_size
    B, Q_S = case.query.shape[0], case.query.shape[1]
    idx = case.sparse_indices.reshape(B, Q_S, -1).astype(np.int64)
    lens = case.actual_seq_lengths_kv.astype(np.int64).reshape(B, 1)
    qlen = (np.full((B, 1), Q_S, dtype=np.int64) if case.actual_seq_lengths_query is None
            else case.actual_seq_lengths_query.astype(np.int64).reshape(B, 1))
    s = np.arange(Q_S, dtype=np.int64)[None, :]
    limit = lens - qlen + s + 1 if case.sparse_mode == 3 else np.broadcast_to(lens, (B, Q_S))
    limit = np.where(s < qlen, limit, 0)
    tok = idx[..., None] * sbs + np.arange(sbs)
    ok = (idx[..., None] >= 0) & (tok < limit[:, :, None, None])
    return ok.reshape(B * Q_S, -1).sum(axis=1)


def algorithmic_bytes(case) -> int:
    if isinstance(case, gen.AppendCase):
        rows = case.key_new.size                               # B * KV_N * D elements per tensor
        es = 1 if case.kv_dtype == "int8" else 2
        total = 2 * rows * 2 + 2 * rows * es                   # new key/value rows read, cache rows written
        total += case.positions.nbytes
        if case.block_table is not None:
            total += case.B * 4                                # the block-table entry of each position
        if case.antiquant_scale is not None:
            total += case.antiquant_scale.nbytes + case.antiquant_offset.nbytes
        return int(total)
    if isinstance(case, gen.SfaCase):
        n = int(sfa_valid_counts(case).sum())
        QN = case.query.shape[2]
        # key, key_rope and value rows of selected tokens; with value = key a row serves both
        total = n * (512 + 64 + (0 if case.value is case.key else 512)) * 2
        rows = case.B * case.query.shape[1]                    # (batch, query token) rows
        total += rows * QN * (512 + 64) * 2                    # query and query_rope
        total += rows * QN * 512 * 2                           # output
        total += case.sparse_indices.nbytes + n * 4            # indices and block-table entries used
        return int(total)
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
    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.t0 = self.t1 = None
        self.lines = []

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

def kernel_sources_digest(family: str) -> str:
    """Digest of the sources that decide one kernel family's DRAM traffic: "decode" (the
    split-KV decode kernel, its planner and API) or "sfa" (the sparse tile-count, decode and combine
    kernels, their API, and the shared constants and PTX helpers)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "kv_cache_incremental_split_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if not f.endswith((".cu", ".cuh")):
            continue
        sfa_file = f.startswith("sfa")
        shared = f in ("decode.cuh", "ptx.cuh")
        if (family == "sfa" and (sfa_file or shared)) or (family == "decode" and not sfa_file):
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(f.encode())
                h.update(fh.read())
    return h.hexdigest()[:16]


def kernel_family(workload: str) -> str:
    return "sfa" if workload.startswith("sfa") else "decode"


def recorded_traffic(workload: str):
    """DRAM bytes per launch of the dominant kernel from a committed ncu summary,
    valid only while that kernel family's sources are unchanged since the capture."""
    path = os.path.join(ROOT, "profiles", f"traffic_{workload}.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("kernel_sources_digest") != kernel_sources_digest(kernel_family(workload)):
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

def _batch_subset(case, b):
    """The same problem restricted to batch b (shared paged caches stay whole)."""
    from copy import copy
    c = copy(case)
    sel = np.array([b])
    if isinstance(case, gen.AppendCase):
        c.key_new, c.value_new, c.positions = case.key_new[sel], case.value_new[sel], case.positions[sel]
        if case.block_table is None:
            c.key_cache, c.value_cache = case.key_cache[sel], case.value_cache[sel]
        else:  # only batch b's blocks, renumbered
            blocks = case.block_table[b][case.block_table[b] >= 0]
            c.key_cache, c.value_cache = case.key_cache[blocks], case.value_cache[blocks]
            c.block_table = np.where(case.block_table[sel] >= 0, np.arange(case.block_table.shape[1])[None], -1)
            c.block_table = c.block_table.astype(np.int32)
        return c
    if isinstance(case, gen.SfaCase):
        c.query, c.query_rope = case.query[sel], case.query_rope[sel]
        c.sparse_indices, c.block_table = case.sparse_indices[sel], case.block_table[sel]
        c.actual_seq_lengths_kv = case.actual_seq_lengths_kv[sel]
        if case.actual_seq_lengths_query is not None:
            c.actual_seq_lengths_query = case.actual_seq_lengths_query[sel]
        return c
    c.query = case.query[sel]
    if case.kv_format == "contig":
        c.key, c.value = case.key[sel], case.value[sel]
    elif case.kv_format == "tensorlist":
        c.key, c.value = [case.key[b]], [case.value[b]]
    if case.block_table is not None:
        c.block_table = case.block_table[sel]
    if case.atten_mask is not None and case.atten_mask.shape[0] > 1:
        c.atten_mask = case.atten_mask[sel]
    if case.actual_seq_lengths is not None:
        c.actual_seq_lengths = case.actual_seq_lengths[sel]
    if case.kv_padding_size is not None and case.kv_padding_size.size > 1:
        c.kv_padding_size = case.kv_padding_size[sel]
    return c


def _run_oracle(c):
    """One run of the CPU oracle on case c (test infrastructure: only the CPU-baseline and
    reference legs of the benchmark call it)."""
    import oracle
    fmt = {"contig": oracle.CONTIG, "paged_nbsd": oracle.PAGED_NBSD, "paged_bsh": oracle.PAGED_BSH}
    aq = {"none": oracle.AQ_NONE, "per_channel": oracle.AQ_PER_CHANNEL, "per_tensor": oracle.AQ_PER_TENSOR}
    if isinstance(c, gen.AppendCase):
        oracle.kv_append_ref(c.key_new, c.value_new, c.positions, c.key_cache, c.value_cache, layout=c.layout,
                             kv_format=fmt[c.kv_format], block_size=c.block_size, block_table=c.block_table,
                             antiquant=aq[c.antiquant], antiquant_scale=c.antiquant_scale,
                             antiquant_offset=c.antiquant_offset)
    elif isinstance(c, gen.SfaCase):
        oracle.sfa_ref(c.query, c.query_rope, c.key, c.key_rope, c.value, c.sparse_indices, c.block_table,
                       c.actual_seq_lengths_kv, scale=c.scale, sparse_block_size=c.sparse_block_size,
                       sparse_mode=c.sparse_mode, actual_seq_lengths_query=c.actual_seq_lengths_query)
    elif c.kv_format == "tensorlist":
        oracle.ifa_ref_tensorlist(c.query, c.key, c.value, num_heads=c.num_heads, num_kv_heads=c.num_kv_heads,
                                  scale=c.scale, layout=c.layout, atten_mask=c.atten_mask,
                                  actual_seq_lengths=c.actual_seq_lengths, antiquant=aq[c.antiquant],
                                  antiquant_scale=c.antiquant_scale, antiquant_offset=c.antiquant_offset)
    else:
        oracle.ifa_ref(c.query, c.key, c.value, num_heads=c.num_heads, num_kv_heads=c.num_kv_heads,
                       scale=c.scale, layout=c.layout, kv_format=fmt[c.kv_format], block_size=c.block_size,
                       block_table=c.block_table, atten_mask=c.atten_mask,
                       actual_seq_lengths=c.actual_seq_lengths, kv_padding_size=c.kv_padding_size,
                       antiquant=aq[c.antiquant], antiquant_scale=c.antiquant_scale,
                       antiquant_offset=c.antiquant_offset)


def host_threads() -> int:
    """Host cores this process may run on."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except (AttributeError, OSError):
        return max(1, os.cpu_count() or 1)


ORACLE_MAX_PASSES = 64  # a small workload's sample stops after this many passes over its rows


def oracle_sample(case, budget_s: float, threads: int = 1, start_batch: int = 0):
    """Time the CPU oracle on whole batch rows of the workload for about `budget_s` seconds of
    wall time (or ORACLE_MAX_PASSES passes over the rows), `threads` threads taking rows in
    turn (the C oracle runs without the GIL).
    Returns (algorithmic bytes done, wall seconds, rows done in order)."""
    import threading
    from concurrent.futures import ThreadPoolExecutor
    lock = threading.Lock()
    state = {"next": start_batch, "bytes": 0, "done": []}
    t0 = time.perf_counter()

    def worker():
        first = True
        while True:
            with lock:
                if not first and (time.perf_counter() - t0 >= budget_s or
                                  len(state["done"]) >= ORACLE_MAX_PASSES * case.B):
                    return
                b = state["next"] % case.B
                state["next"] += 1
            first = False
            c = _batch_subset(case, b)
            _run_oracle(c)
            nb = algorithmic_bytes(c)
            with lock:
                state["bytes"] += nb
                state["done"].append(b)

    with ThreadPoolExecutor(max_workers=threads) as ex:
        for f in [ex.submit(worker) for _ in range(threads)]:
            f.result()
    return state["bytes"], time.perf_counter() - t0, state["done"]


def cpu_baseline_legs(case, budget_s: float):
    """The oracle at one thread and at every host core: the baseline object of the JSON line
    (its value and cores are the all-core leg's)."""
    legs = {}
    for th in sorted({1, host_threads()}):
        nb, t, done = oracle_sample(case, budget_s, threads=th)
        legs[th] = (nb / t / 1e9, nb, t, len(done))
    nmax = max(legs)
    v, nb, t, rows = legs[nmax]
    return {"value": v, "unit": UNIT, "cores": nmax, "kind": "oracle",
            "sample": (f"whole batch rows of the same workload, taken in turn by {nmax} threads until about "
                       f"{budget_s:.0f} s or {ORACLE_MAX_PASSES} passes over the batch rows, whichever comes "
                       f"first ({rows} rows, {nb / 1e6:.1f} MB algorithmic, {t:.2f} s wall); plain C, float64"),
            "by_threads": {str(th): {"value": lv, "rows": lr, "seconds": round(lt, 2)}
                           for th, (lv, _, lt, lr) in legs.items()}}


_ROWS = {}


def _truncated(case, b, frac):
    """Batch b of the workload with its work cut to about `frac` (0 < frac <= 1): fewer
    tokens (attention), fewer selected indices (sparse), or the whole row (append).  The
    batch rows are cut out of the workload once and reused."""
    from copy import copy
    key = (id(case), b)
    if key not in _ROWS:
        _ROWS[key] = _batch_subset(case, b)
    c = copy(_ROWS[key])
    if frac >= 1.0 or isinstance(c, gen.AppendCase):
        return c
    if isinstance(c, gen.SfaCase):
        n = max(1, int(c.sparse_indices.shape[-1] * frac))
        c.sparse_indices = np.ascontiguousarray(c.sparse_indices[..., :n])
        return c
    if c.actual_seq_lengths is not None:
        c.actual_seq_lengths = np.maximum(1, (c.actual_seq_lengths * frac).astype(np.int64))
    return c


def oracle_unit(case, b, frac):
    """Bytes and seconds of one oracle run on batch b cut to `frac` of its work."""
    c = _truncated(case, b, frac)
    t = time.perf_counter()
    _run_oracle(c)
    return algorithmic_bytes(c), time.perf_counter() - t


def input_copies(args, alg):
    """Input copies the device arm rotates through: enough that the bytes streamed between two
    uses of one copy exceed L2 several times (inputs larger than L2: no flush between steps)."""
    return args.copies or max(1, min(8, math.ceil(6 * L2_BYTES / max(1, alg))))


def l2_method(args, case):
    """How the device arm keeps L2 from serving repeated inputs, stated for `config`."""
    if isinstance(case, gen.AppendCase):
        return "no flush: the append caches stay resident (launch-bound calls)"
    alg = algorithmic_bytes(case)
    copies = input_copies(args, alg)
    if copies * alg >= L2_BYTES:
        return (f"inputs larger than L2, no flush: {copies} input cop{'y' if copies == 1 else 'ies'} in "
                f"rotation, {copies * alg / 1e6:.0f} MB of algorithmic bytes between two uses of a copy")
    return (f"inputs resident in L2 ({copies} input copies in rotation, {copies * alg / 1e6:.1f} MB): "
            f"a latency-bound workload")


def line_config(args, case, world):
    """The `config` object both arms print: the workload, its seed, algorithmic bytes and the
    device arm's L2 method."""
    return {"workload": WORKLOADS[args.workload], "name": args.workload, "seed": args.seed,
            "algorithmic_bytes_per_step": algorithmic_bytes(case),
            "parallelism": f"replica x{world}" if world > 1 else "single GPU",
            "l2": l2_method(args, case)}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    case = make_case(args.workload, args.seed)
    threads = args.ref_threads or host_threads()
    # The whole run takes about --ref-total-seconds: each of the W + K steps runs the oracle on
    # `threads` batch rows at once, each cut to the fraction of its work that fits the per-step
    # share (calibrated on a full row first).
    per_step = args.ref_total_seconds / max(1, args.warmup + args.steps)
    _, t_full = oracle_unit(case, 0, 1.0)
    frac = min(1.0, per_step / max(t_full, 1e-9))
    from concurrent.futures import ThreadPoolExecutor
    total_b, total_t, rows = 0, 0.0, 0
    with ThreadPoolExecutor(max_workers=threads) as ex:
        for step in range(args.warmup + args.steps):
            t = time.perf_counter()
            futs = [ex.submit(oracle_unit, case, (step * threads + i) % case.B, frac) for i in range(threads)]
            nb = sum(f.result()[0] for f in futs)
            t = time.perf_counter() - t
            if step >= args.warmup:
                total_b += nb
                total_t += t
                rows += threads
    value = total_b / total_t / 1e9
    sample = (f"each step: the oracle on {threads} batch rows of the workload at once ({threads} threads), each "
              f"cut to {100 * frac:.1f}% of its work ({rows} rows over {args.steps} steps, "
              f"{total_b / 1e6:.1f} MB algorithmic, {total_t:.1f} s wall)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / max(1, args.steps),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": line_config(args, case, world),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------------------ GPU arm

def _to_dev(a, dev):
    import torch
    if a is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(a))
    return (t.view(torch.bfloat16) if a.dtype == np.uint16 else t).to(dev)


class IfaWorkload:
    """One incremental-attention problem on the device, with rotating key/value copies.  With
    key/value as one tensor per batch each copy has its own op (plan), so the per-batch tensor
    maps of every copy are encoded once, before the graphs are captured."""

    def __init__(self, case: gen.IfaCase, dev, copies_for):
        from kv_cache_incremental_split_gb300.ifa import IncreFlashAttention
        self.case, self.dev = case, dev
        m = case.atten_mask
        self.tensorlist = case.kv_format == "tensorlist"
        paged = case.kv_format.startswith("paged")

        def new_op():
            return IncreFlashAttention(
                batch=case.B, num_heads=case.num_heads, num_kv_heads=case.num_kv_heads, head_dim=case.D,
                max_seq_len=case.max_seq_len, dtype=case.q_dtype, kv_dtype=case.kv_dtype, layout=case.layout,
                kv_format=case.kv_format, block_size=case.block_size,
                block_num=case.key.shape[0] if paged else 0,
                block_table_cols=case.block_table.shape[1] if case.block_table is not None else 0,
                mask_shape=None if m is None else m.shape, mask_dtype="bool", antiquant=case.antiquant,
                kv_padding=case.kv_padding_size is not None, scale=case.scale, device=dev)

        self.copies = copies_for
        self.ops = [new_op() for _ in range(self.copies if self.tensorlist else 1)]
        self.op = self.ops[0]
        self.e2e_op = new_op() if self.tensorlist else self.op
        self.q = _to_dev(case.query, dev)
        self.mask, self.bt = _to_dev(case.atten_mask, dev), _to_dev(case.block_table, dev)
        self.sc, self.of = _to_dev(case.antiquant_scale, dev), _to_dev(case.antiquant_offset, dev)
        if self.tensorlist:
            k = [_to_dev(t, dev) for t in case.key]
            v = [_to_dev(t, dev) for t in case.value]
            self.rotating_bytes = sum(t.numel() * t.element_size() for t in k + v)
            self.ks = [k] + [[t.clone() for t in k] for _ in range(self.copies - 1)]
            self.vs = [v] + [[t.clone() for t in v] for _ in range(self.copies - 1)]
        else:
            k, v = _to_dev(case.key, dev), _to_dev(case.value, dev)
            self.rotating_bytes = k.numel() * k.element_size() + v.numel() * v.element_size()
            self.ks = [k] + [k.clone() for _ in range(self.copies - 1)]
            self.vs = [v] + [v.clone() for _ in range(self.copies - 1)]
        self.outs = [self.q.new_empty(self.q.shape) for _ in range(self.copies)]
        self.dtype = case.q_dtype if case.kv_dtype != "int8" else "int8-kv/" + case.q_dtype
        self.call_name = "ifa_run_tensorlist" if self.tensorlist else "ifa_run"
        self.launch_note = "; programmatic dependent launch lets each kernel start its prologue as the previous one drains"

    def call(self, i, stream):
        c = self.case
        op = self.ops[i] if self.tensorlist else self.op
        return op(self.q, self.ks[i], self.vs[i], atten_mask=self.mask, actual_seq_lengths=c.actual_seq_lengths,
                  kv_padding_size=c.kv_padding_size, block_table=self.bt, antiquant_scale=self.sc,
                  antiquant_offset=self.of, out=self.outs[i], stream=stream)

    def launches_per_call(self):
        return self.op.last_launch_count()

    def host_inputs(self):
        c = self.case
        named = [("q", c.query), ("mask", c.atten_mask), ("bt", c.block_table), ("sc", c.antiquant_scale),
                 ("of", c.antiquant_offset)]
        if self.tensorlist:
            named += [(f"k{b}", t) for b, t in enumerate(c.key)] + [(f"v{b}", t) for b, t in enumerate(c.value)]
        else:
            named += [("k", c.key), ("v", c.value)]
        return {n: a for n, a in named if a is not None}

    def call_on(self, d, stream):
        c = self.case
        if self.tensorlist:
            k, v = [d[f"k{b}"] for b in range(c.B)], [d[f"v{b}"] for b in range(c.B)]
        else:
            k, v = d["k"], d["v"]
        return self.e2e_op(d["q"], k, v, atten_mask=d.get("mask"), actual_seq_lengths=c.actual_seq_lengths,
                           kv_padding_size=c.kv_padding_size, block_table=d.get("bt"), antiquant_scale=d.get("sc"),
                           antiquant_offset=d.get("of"), stream=stream)


class SfaWorkload:
    """One sparse MLA-absorb problem on the device, with rotating cache copies."""

    def __init__(self, case: gen.SfaCase, dev, copies_for):
        from kv_cache_incremental_split_gb300.ifa import SparseFlashAttention
        self.case, self.dev = case, dev
        self.op = SparseFlashAttention(batch=case.B, num_heads=case.query.shape[2], block_size=case.key.shape[1],
                                       block_num=case.key.shape[0], block_table_cols=case.block_table.shape[1],
                                       sparse_size=case.sparse_indices.shape[-1], dtype=case.dtype,
                                       scale=case.scale, sparse_block_size=case.sparse_block_size,
                                       sparse_mode=case.sparse_mode, q_seq_len=case.query.shape[1], device=dev)
        self.q, self.qr = _to_dev(case.query, dev), _to_dev(case.query_rope, dev)
        self.idx, self.bt = _to_dev(case.sparse_indices, dev), _to_dev(case.block_table, dev)
        self.lens = _to_dev(case.actual_seq_lengths_kv, dev)
        self.lq = None if case.actual_seq_lengths_query is None else _to_dev(case.actual_seq_lengths_query, dev)
        self.aliased = case.value is case.key  # one tensor passed as key and as value
        k, kr = _to_dev(case.key, dev), _to_dev(case.key_rope, dev)
        v = k if self.aliased else _to_dev(case.value, dev)
        self.copies = copies_for
        self.rotating_bytes = sum(t.numel() * t.element_size() for t in ((k, kr) if self.aliased else (k, kr, v)))

        def clone3():
            k2, kr2 = k.clone(), kr.clone()
            return k2, kr2, (k2 if self.aliased else v.clone())

        self.caches = [(k, kr, v)] + [clone3() for _ in range(self.copies - 1)]
        self.outs = [self.q.new_empty(self.q.shape) for _ in range(self.copies)]
        self.dtype = case.dtype
        self.call_name = "sfa_run"
        self.launch_note = ": tile-count kernel + decode kernel + combine kernel"

    def call(self, i, stream):
        k, kr, v = self.caches[i]
        return self.op(self.q, self.qr, k, kr, v, self.idx, self.bt, self.lens, actual_seq_lengths_query=self.lq,
                       out=self.outs[i], stream=stream)

    def launches_per_call(self):
        return 3  # tile-count kernel, decode kernel (CTA pairs), combine kernel

    def host_inputs(self):
        c = self.case
        return {"q": c.query, "qr": c.query_rope, "k": c.key, "kr": c.key_rope,
                **({} if self.aliased else {"v": c.value}),
                "idx": c.sparse_indices, "bt": c.block_table, "lens": c.actual_seq_lengths_kv,
                **({} if c.actual_seq_lengths_query is None else {"lq": c.actual_seq_lengths_query})}

    def call_on(self, d, stream):
        return self.op(d["q"], d["qr"], d["k"], d["kr"], d["k"] if self.aliased else d["v"], d["idx"], d["bt"],
                       d["lens"], actual_seq_lengths_query=d.get("lq"), stream=stream)


class AppendWorkload:
    """One decode step's KV-cache append on the device: the caches stay resident and are
    written in place; step i writes at the positions minus i mod 8, so the rows written
    differ from one step to the next."""

    def __init__(self, case: gen.AppendCase, dev, copies_for):
        import torch
        from kv_cache_incremental_split_gb300.ifa import KvCacheAppend
        self.case, self.dev = case, dev
        paged = case.kv_format != "contig"
        KVN, D = case.key_new.shape[1], case.key_new.shape[2]
        self.op = KvCacheAppend(batch=case.B, num_kv_heads=KVN, head_dim=D,
                                max_seq_len=0 if paged else case.key_cache.shape[2], dtype=case.dtype,
                                kv_dtype=case.kv_dtype, layout=case.layout, kv_format=case.kv_format,
                                block_size=case.block_size, block_num=case.key_cache.shape[0] if paged else 0,
                                block_table_cols=case.block_table.shape[1] if paged else 0,
                                antiquant=case.antiquant, device=dev)
        self.kn, self.vn = _to_dev(case.key_new, dev), _to_dev(case.value_new, dev)
        self.kc, self.vc = _to_dev(case.key_cache, dev), _to_dev(case.value_cache, dev)
        self.bt = _to_dev(case.block_table, dev)
        self.sc, self.of = _to_dev(case.antiquant_scale, dev), _to_dev(case.antiquant_offset, dev)
        self.copies = copies_for
        # earlier positions of the same sequences: still inside the cache and the block table
        self.pos = [_to_dev(case.positions - (i % 8), dev) for i in range(self.copies)]
        self.q = self.op.errors  # the step's result read back end to end: the device error word
        self.rotating_bytes = 0
        self.l2_note = (f"the caches ({2 * self.kc.numel() * self.kc.element_size() / 1e6:.0f} MB) stay resident; "
                        f"positions shift by the step number mod {self.copies}")
        self.dtype = case.dtype if case.kv_dtype != "int8" else "int8-kv/" + case.dtype
        self.call_name = "ifa_kv_append"
        self.launch_note = ""

    def call(self, i, stream):
        self.op(self.kn, self.vn, self.pos[i], self.kc, self.vc, block_table=self.bt, antiquant_scale=self.sc,
                antiquant_offset=self.of, stream=stream)
        return self.op.errors

    def launches_per_call(self):
        return 1

    def host_inputs(self):
        c = self.case
        d = {"kn": c.key_new, "vn": c.value_new, "pos": c.positions}
        if c.block_table is not None:
            d["bt"] = c.block_table
        if c.antiquant_scale is not None:
            d["sc"], d["of"] = c.antiquant_scale, c.antiquant_offset
        return d

    def call_on(self, d, stream):
        self.op(d["kn"], d["vn"], d["pos"], self.kc, self.vc, block_table=d.get("bt"), antiquant_scale=d.get("sc"),
                antiquant_offset=d.get("of"), stream=stream)
        return self.op.errors


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

    case = make_case(args.workload, args.seed + rank)
    alg = algorithmic_bytes(case)
    copies = input_copies(args, alg)
    if isinstance(case, gen.AppendCase):
        wl = AppendWorkload(case, dev, copies)
    elif isinstance(case, gen.SfaCase):
        wl = SfaWorkload(case, dev, copies)
    else:
        wl = IfaWorkload(case, dev, copies)
    stream = torch.cuda.Stream(device=dev)

    with torch.cuda.stream(stream):
        # every copy is called at least once before the capture (a tensorlist plan encodes its
        # per-batch descriptors on its first call, outside the graph)
        for w in range(max(args.warmup, 3, copies)):
            wl.call(w % copies, stream)
        stream.synchronize()
        launches_per_call = wl.launches_per_call()
        # Consecutive calls are captured together, as a decode step's layers would be: one graph
        # of `chunk` calls (a multiple of the copy count, so step s always reads copy s % copies)
        # replayed K // chunk times, plus one graph for the remaining K % chunk calls.
        chunk = max(1, 64 // copies) * copies
        n_chunks, rem = divmod(args.steps, chunk)
        graphs = []
        for n_calls in (chunk, rem):
            if n_calls == 0:
                graphs.append(None)
                continue
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(n_calls):
                    wl.call(i % copies, stream)
            graphs.append(g)
        for g in graphs:
            if g is not None:
                g.replay()
        stream.synchronize()

    # eager calls/s (host-launched, no graph), for reference only
    with torch.cuda.stream(stream):
        n_eager = min(args.steps, 200)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        stream.synchronize()
        e0.record(stream)
        for i in range(n_eager):
            wl.call(i % copies, stream)
        e1.record(stream)
        e1.synchronize()
        eager_ms = e0.elapsed_time(e1) / n_eager

    # ---- timed: the K steps as one region (graph replays), R times over; each region is
    # bracketed by a barrier (multi-rank) and a device synchronisation
    def region_ms():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        start.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(n_chunks):
                graphs[0].replay()
            if graphs[1] is not None:
                graphs[1].replay()
        end.record(stream)
        end.synchronize()
        return start.elapsed_time(end)

    if world > 1:
        import torch.distributed as dist
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    est = region_ms()  # untimed: sizes the repeat count
    reps = max(args.repeats, min(args.max_repeats, math.ceil(args.min_timed_seconds * 1e3 / max(est, 1e-3))))
    if world > 1:  # every rank runs the same number of regions
        rt = torch.tensor([reps], dtype=torch.int64, device=dev)
        dist.all_reduce(rt, op=dist.ReduceOp.MAX)
        reps = int(rt.item())
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    smi_index = vis.split(",")[local] if vis and len(vis.split(",")) > local else str(local)
    sampler = ClockSampler(smi_index)
    with sampler:
        sampler.mark_start()
        regions = [region_ms() for _ in range(reps)]
        torch.cuda.synchronize()
        sampler.mark_end()
    q10, q50, q90 = (float(x) for x in np.percentile(regions, [10, 50, 90]))
    # max over ranks of each statistic; bytes summed over ranks
    max_elapsed, total_bytes = aggregate(q50, float(alg) * args.steps, world)
    p10_elapsed, _ = aggregate(q10, 0.0, world)
    p90_elapsed, _ = aggregate(q90, 0.0, world)
    ms_per_step = max_elapsed / args.steps
    value = total_bytes / (max_elapsed * 1e-3) / 1e9
    local_gbs = alg / (q50 / args.steps * 1e-3) / 1e9

    # ---- end to end through the public API: pinned host inputs -> device -> call -> host output
    host = {n: torch.from_numpy(np.ascontiguousarray(a)).pin_memory() for n, a in wl.host_inputs().items()}
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    bf_names = {n for n, a in wl.host_inputs().items() if a.dtype == np.uint16}
    d_raw = {n: torch.empty(t.shape, dtype=t.dtype, device=dev) for n, t in host.items()}
    d_in = {n: (t.view(torch.bfloat16) if n in bf_names else t) for n, t in d_raw.items()}
    out_host = torch.empty(wl.q.shape, dtype=wl.q.dtype).pin_memory()
    d2h = out_host.numel() * out_host.element_size()
    n_e2e = max(3, min(args.steps, 20))

    def e2e_step():
        for n, t in host.items():
            d_raw[n].copy_(t, non_blocking=True)
        o = wl.call_on(d_in, stream)
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
        cpu = cpu_baseline_legs(case, args.cpu_seconds)

    peak, peak_kind = measured_peaks()
    clocks = sampler.summary()
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
            "config": line_config(args, case, world),
            "timing": {"regions": reps, "ms_per_step_p10": p10_elapsed / args.steps,
                       "ms_per_step_p90": p90_elapsed / args.steps,
                       "statistic": f"median over {reps} timed regions of the {args.steps} steps",
                       "l2": getattr(wl, "l2_note", None) or (f"inputs larger than L2: {copies} rotating cache "
                                                              f"copies ({copies * wl.rotating_bytes / 1e6:.0f} MB)"),
                       "launch": f"CUDA graphs of {chunk} consecutive {wl.call_name} calls (one call per step"
                                 f"{wl.launch_note}), replayed {n_chunks} times + {rem} calls per region"},
            "calls_per_sec": world * 1e3 / ms_per_step,
            "calls_per_sec_eager": 1e3 / eager_ms,
            "pct_of_hbm_peak": 100.0 * local_gbs / peak,
            "roofline": {"bound": "hbm", "achieved": local_gbs, "peak": peak, "unit": "GB/s",
                         "frac": local_gbs / peak, "peak_kind": peak_kind,
                         "timed": f"{wl.call_name} per step ({launches_per_call} kernel launch"
                                  f"{'es' if launches_per_call > 1 else ''}), CUDA events on its stream",
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
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="paged_gqa", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--copies", type=int, default=0,
                    help="rotating input copies (0: enough that > 6x L2 streams between two uses of one)")
    ap.add_argument("--repeats", type=int, default=5, help="timed regions of K steps, at least")
    ap.add_argument("--min-timed-seconds", type=float, default=1.0,
                    help="more regions until their estimated total reaches this")
    ap.add_argument("--max-repeats", type=int, default=5000)
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="wall seconds of each CPU-baseline leg")
    ap.add_argument("--ref-total-seconds", type=float, default=120.0,
                    help="reference arm: about this many seconds of oracle time over all steps")
    ap.add_argument("--ref-threads", type=int, default=0, help="reference arm threads (0: every host core)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--launch-check", action="store_true",
                    help="check the multi-rank launch and reduction on CPU (gloo): each rank reports its "
                         "workload's bytes and a stand-in time of rank + 1 ms; measures nothing")
    return ap.parse_args(argv)


def _free_port() -> int:
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def relaunch(args, argv) -> int:
    """--gpus N > 1 without a launcher: run this script under torch.distributed.run with N ranks
    on this node (one per GPU), the same arguments, rendezvous on 127.0.0.1."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), os.path.abspath(__file__)]
    cmd += list(sys.argv[1:] if argv is None else argv)
    return subprocess.call(cmd)


def run_launch_check(args) -> int:
    """The multi-rank path without a GPU: process group over gloo, each rank's rank-seeded case,
    the max/sum reduction, one line from rank 0 (value null: nothing is measured)."""
    import torch.distributed as dist
    world, rank, _ = dist_env()
    if world > 1:
        dist.init_process_group("gloo")
    case = make_case(args.workload, args.seed + rank)
    alg = float(algorithmic_bytes(case))
    t, b = aggregate(float(rank + 1), alg * args.steps, world)
    if rank == 0:
        print(json.dumps({"launch_check": True, "metric": METRIC, "value": None, "n_gpus": world,
                          "steps": args.steps, "max_rank_ms": t, "bytes_all_ranks": b,
                          "config": line_config(args, case, world)}))
    if world > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse(argv)
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        return relaunch(args, argv)
    if args.launch_check:
        return run_launch_check(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
