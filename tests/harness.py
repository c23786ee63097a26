"""Helpers shared by the tests: run an ``IfaCase`` / ``SfaCase`` through the CUDA
library (via the C-ABI binding) or through the CPU oracle, and compare."""
from __future__ import annotations

import numpy as np

import oracle
from kv_cache_incremental_split_gb300 import inputs as gen

# Output tolerances (max abs error against the float64 oracle).
TOL = {"fp16": 2e-3, "bf16": 1.5e-2}

_AQ = {"none": oracle.AQ_NONE, "per_channel": oracle.AQ_PER_CHANNEL, "per_tensor": oracle.AQ_PER_TENSOR}
_FMT = {"contig": oracle.CONTIG, "paged_nbsd": oracle.PAGED_NBSD, "paged_bsh": oracle.PAGED_BSH}


def subset(case: gen.IfaCase, batches) -> gen.IfaCase:
    """The same problem restricted to some batches (paged caches are shared)."""
    import copy
    c = copy.copy(case)
    bs = np.asarray(batches)
    c.query = case.query[bs]
    if case.kv_format == "contig":
        c.key, c.value = case.key[bs], case.value[bs]
    if case.block_table is not None:
        c.block_table = case.block_table[bs]
    if case.atten_mask is not None and case.atten_mask.shape[0] > 1:
        c.atten_mask = case.atten_mask[bs]
    if case.actual_seq_lengths is not None:
        c.actual_seq_lengths = case.actual_seq_lengths[bs]
    if case.kv_padding_size is not None and case.kv_padding_size.size > 1:
        c.kv_padding_size = case.kv_padding_size[bs]
    return c


def oracle_ifa(case: gen.IfaCase, batches=None) -> np.ndarray:
    c = case if batches is None else subset(case, batches)
    return oracle.ifa_ref(c.query, c.key, c.value, num_heads=c.num_heads, num_kv_heads=c.num_kv_heads,
                          scale=c.scale, layout=c.layout, kv_format=_FMT[c.kv_format],
                          block_size=c.block_size, block_table=c.block_table, atten_mask=c.atten_mask,
                          actual_seq_lengths=c.actual_seq_lengths, kv_padding_size=c.kv_padding_size,
                          antiquant=_AQ[c.antiquant], antiquant_scale=c.antiquant_scale,
                          antiquant_offset=c.antiquant_offset)


def to_device(a, device="cuda"):
    import torch
    if a is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        t = t.view(torch.bfloat16)
    return t.to(device)


def out_to_f64(t) -> np.ndarray:
    import torch
    return t.detach().to(torch.float64).cpu().numpy()


def make_op(case: gen.IfaCase, split_tiles=0, **kw):
    from kv_cache_incremental_split_gb300.ifa import IncreFlashAttention
    m = case.atten_mask
    return IncreFlashAttention(
        batch=case.B, num_heads=case.num_heads, num_kv_heads=case.num_kv_heads, head_dim=case.D,
        max_seq_len=case.max_seq_len, dtype=case.q_dtype, kv_dtype=case.kv_dtype, layout=case.layout,
        kv_format=case.kv_format, block_size=case.block_size,
        block_num=case.key.shape[0] if case.kv_format in ("paged_nbsd", "paged_bsh") else 0,
        block_table_cols=case.block_table.shape[1] if case.block_table is not None else 0,
        mask_shape=None if m is None else m.shape,
        mask_dtype="bool" if m is None or m.dtype == np.bool_ else ("int8" if m.dtype == np.int8 else "uint8"),
        antiquant=case.antiquant, kv_padding=case.kv_padding_size is not None, scale=case.scale,
        split_tiles=split_tiles, **kw)


class DeviceCase:
    """Device copies of a case's tensors, created once and reused across calls."""

    def __init__(self, case: gen.IfaCase):
        self.case = case
        self.q = to_device(case.query)
        self.k = to_device(case.key)
        self.v = to_device(case.value)
        self.mask = to_device(case.atten_mask)
        self.bt = to_device(case.block_table)
        self.sc = to_device(case.antiquant_scale)
        self.of = to_device(case.antiquant_offset)

    def run(self, op, out=None, **kw):
        c = self.case
        return op(self.q, self.k, self.v, atten_mask=self.mask, actual_seq_lengths=c.actual_seq_lengths,
                  kv_padding_size=c.kv_padding_size, block_table=self.bt, antiquant_scale=self.sc,
                  antiquant_offset=self.of, out=out, **kw)


def gpu_ifa(case: gen.IfaCase, split_tiles=0) -> np.ndarray:
    import torch
    dc = DeviceCase(case)
    op = make_op(case, split_tiles)
    out = dc.run(op)
    torch.cuda.synchronize()
    return out_to_f64(out).reshape(case.B, case.num_heads, case.D)


def max_abs_err(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    if a.size == 0:
        return 0.0
    return float(np.max(np.abs(a - b)))
