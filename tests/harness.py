"""Helpers shared by the tests: run an ``IfaCase`` / ``SfaCase`` through the CUDA
library (via the C-ABI binding) or through the CPU oracle, and compare."""
from __future__ import annotations

import math

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


# ---------------------------------------------------------------- sparse decode probes

_PROBE_BITS = 12  # token-index bits the softmax_sum fingerprint covers


def sfa_live_tiles(idx_rows):
    """Live 128-position tiles of each index row: up to the last entry that holds an index >= 0."""
    ok = idx_rows >= 0
    last = np.where(ok.any(axis=1), idx_rows.shape[1] - 1 - np.argmax(ok[:, ::-1], axis=1), -1)
    return np.where(last < 0, 0, (last + 1 + 127) // 128)


def sfa_pieces_per_row(idx_rows, sms):
    """CTA pairs that hold a part of each index row, under the library's split: pairs take equal
    contiguous shares (floor(c W / Pa)) of the rows' live tiles in row order, with at most one pair
    per two SMs and shares of at least one tile (the library's smallest share)."""
    eff = sfa_live_tiles(idx_rows).astype(np.int64)
    tps = -(-idx_rows.shape[1] // 128)
    share = 1
    launched = max(1, min(min(256, sms) // 2, -(-(len(eff) * tps) // share)))
    W = int(eff.sum())
    Pa = max(1, min(launched, -(-W // share)))
    pre = np.concatenate([[0], np.cumsum(eff)])
    first = ((pre[:-1] + 1) * Pa - 1) // W
    last = ((pre[:-1] + eff) * Pa - 1) // W
    bounds = {c * W // Pa for c in range(1, Pa)}
    ends_on_boundary = np.array([eff[r] > 0 and int(pre[r] + eff[r]) in bounds for r in range(len(eff))])
    return np.where(eff > 0, last - first + 1, 0), ends_on_boundary


def sfa_selected_tokens(c, r):
    """Tokens row r (batch b, query token s) attends to, for token-wise indices with every query
    token valid: its indices in [0, limit), the limit being the length, or len - Q_S + s + 1 under
    the right-down causal mode."""
    Q_S = c.query.shape[1]
    b, s = divmod(r, Q_S)
    idx = c.sparse_indices[b, s, 0].astype(np.int64)
    ln = int(c.actual_seq_lengths_kv[b])
    lim = ln - Q_S + s + 1 if c.sparse_mode == 3 else ln
    return idx[(idx >= 0) & (idx < lim)]


def sfa_bit_probe(c):
    """Query 0 except query_rope[head n] = -1 at channel n mod 12; key_rope of token t = the bits
    of t; scale ln 2.  Every score of head n is -bit_{n mod 12}(t), every probability exactly 1 or
    1/2, so softmax_sum is exact: (count with bit 0) + (count with bit 1) / 2, or the count when no
    selected token has bit 0.  It pins the selected set, not only its size."""
    B, Q_S, Q_N = c.query.shape[0], c.query.shape[1], c.query.shape[2]
    bs = c.key.shape[1]
    c.query = np.zeros_like(c.query)
    qr = np.zeros(c.query_rope.shape, dtype=np.float32)
    for n in range(Q_N):
        qr[:, :, n, n % _PROBE_BITS] = -1.0
    c.query_rope = gen.to_storage(qr, c.dtype)
    cols = c.block_table.shape[1]
    col_of_block = np.empty(c.key.shape[0], dtype=np.int64)
    col_of_block[c.block_table.reshape(-1)] = np.tile(np.arange(cols), B)
    tok = col_of_block[:, None] * bs + np.arange(bs)[None, :]            # (block, slot) -> token
    kr = np.zeros(c.key_rope.shape, dtype=np.float32)
    for j in range(_PROBE_BITS):
        kr[:, :, 0, j] = (tok >> j) & 1
    c.key_rope = gen.to_storage(kr, c.dtype)
    c.scale = math.log(2.0)
    exp_sum = np.zeros((B * Q_S, Q_N))
    exp_max = np.full((B * Q_S, Q_N), -np.inf)
    for r in range(B * Q_S):
        t = sfa_selected_tokens(c, r)
        for n in range(Q_N):
            bit = (t >> (n % _PROBE_BITS)) & 1
            n1 = int(bit.sum())
            n0 = len(t) - n1
            exp_sum[r, n] = n0 + 0.5 * n1 if n0 > 0 else float(n1)
            if len(t):
                exp_max[r, n] = 0.0 if n0 > 0 else -math.log(2.0)
    return c, exp_sum, exp_max
