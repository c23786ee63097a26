"""Seeded synthetic inputs for decode attention, shared by the tests, the
benchmark and the smoke check.

This module holds no attention arithmetic: it only draws random numbers,
rounds them to the device storage types and lays them out in the shapes the
IncreFlashAttention / SparseFlashAttention pages define.  Host arrays use
``numpy.float16`` for fp16, ``numpy.uint16`` bit patterns for bf16 and
``numpy.int8`` for int8.

Workload recipes (value distributions and structure follow the decode
workloads this library is measured on):

* ``tiny_mha``      B=1, N=KV_N=8, D=64, BNSD fp16, S=128, lengths [128]
* ``gqa_padded``    B=16, N=32, KV_N=8, D=128, BSH bf16, Smax=4096,
                    lengths ~ U{1..4096}, bool mask (B,1,1,S) true past each length
* ``paged_gqa``     B=64, N=32, KV_N=8, D=128, bf16, blockSize=128,
                    cache (blocknum, KV_N, 128, D), blockTable a random permutation
                    of the physical blocks, lengths ~ U{512..32768}
* ``int8_leftpad``  B=32, N=64, KV_N=8, D=128, fp16 query, BNSD int8 K/V ~ U{-127..127},
                    per-channel scale ~ U[0.005,0.02], offset ~ U[-4,4], Smax=8192,
                    lengths ~ U{256..8192}, kvPaddingSize = Smax - length - U{0..64}
* ``sfa_mla``       B=32, Q_N=128, KV_N=1, D=512 + rope 64, bf16, PA_BSND block 64,
                    KV length 32768, sparse_indices (B,1,1,2048): U{1024..2048} distinct
                    indices < length in random order, then a -1 tail

Every generator takes shrink arguments so tests can build the same structure
at sizes the CPU oracle finishes in seconds.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Any, Dict, Optional

import numpy as np

_CHUNK = 1 << 22  # elements per independently seeded chunk (fixed: results do not depend on threads)


def _pool_map(fn, n):
    workers = max(1, min(32, os.cpu_count() or 1))
    if n <= 1 or workers == 1:
        return [fn(i) for i in range(n)]
    with ThreadPoolExecutor(max_workers=workers) as ex:
        return list(ex.map(fn, range(n)))


def _children(seed: int, tag: int, n: int):
    return np.random.SeedSequence(entropy=int(seed), spawn_key=(int(tag),)).spawn(n)


def normal_f32(seed: int, tag: int, shape) -> np.ndarray:
    """N(0,1) float32 array, filled in fixed-size chunks with spawned seeds."""
    size = int(np.prod(shape))
    out = np.empty(size, dtype=np.float32)
    n = max(1, math.ceil(size / _CHUNK))
    kids = _children(seed, tag, n)

    def fill(i):
        lo, hi = i * _CHUNK, min(size, (i + 1) * _CHUNK)
        np.random.default_rng(kids[i]).standard_normal(out=out[lo:hi], dtype=np.float32)

    _pool_map(fill, n)
    return out.reshape(shape)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (round to nearest even), returned as uint16 bits."""
    flat = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    out = np.empty(flat.size, dtype=np.uint16)
    n = max(1, math.ceil(flat.size / _CHUNK))

    def conv(i):
        lo, hi = i * _CHUNK, min(flat.size, (i + 1) * _CHUNK)
        u = flat[lo:hi].view(np.uint32)
        r = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
        out[lo:hi] = ((u + r) >> np.uint32(16)).astype(np.uint16)

    _pool_map(conv, n)
    return out.reshape(x.shape)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "fp16":
        return x.astype(np.float16)
    if dtype == "bf16":
        return f32_to_bf16_bits(x)
    raise ValueError(dtype)


def random_storage(seed: int, tag: int, shape, dtype: str) -> np.ndarray:
    return to_storage(normal_f32(seed, tag, shape), dtype)


def uniform_int8(seed: int, tag: int, shape, lo: int = -127, hi: int = 127) -> np.ndarray:
    size = int(np.prod(shape))
    out = np.empty(size, dtype=np.int8)
    n = max(1, math.ceil(size / _CHUNK))
    kids = _children(seed, tag, n)

    def fill(i):
        a, b = i * _CHUNK, min(size, (i + 1) * _CHUNK)
        out[a:b] = np.random.default_rng(kids[i]).integers(lo, hi + 1, size=b - a, dtype=np.int8)

    _pool_map(fill, n)
    return out.reshape(shape)


@dataclass
class IfaCase:
    """One incremental-attention problem: host arrays plus the call attributes."""
    name: str
    query: np.ndarray
    key: np.ndarray
    value: np.ndarray
    num_heads: int
    num_kv_heads: int
    scale: float
    layout: str = "BNSD"          # query layout (and contiguous key/value layout)
    kv_format: str = "contig"     # contig | paged_nbsd | paged_bsh
    q_dtype: str = "bf16"
    kv_dtype: str = "bf16"        # bf16 | fp16 | int8
    max_seq_len: int = 0          # contiguous S (Smax)
    block_size: int = 0
    block_table: Optional[np.ndarray] = None
    atten_mask: Optional[np.ndarray] = None
    actual_seq_lengths: Optional[np.ndarray] = None
    kv_padding_size: Optional[np.ndarray] = None
    antiquant: str = "none"       # none | per_channel | per_tensor
    antiquant_scale: Optional[np.ndarray] = None
    antiquant_offset: Optional[np.ndarray] = None
    meta: Dict[str, Any] = field(default_factory=dict)

    @property
    def B(self) -> int:
        return self.query.shape[0]

    @property
    def D(self) -> int:
        return self.query.size // (self.B * self.num_heads)


@dataclass
class SfaCase:
    name: str
    query: np.ndarray           # (B, Q_S, Q_N, D)
    query_rope: np.ndarray      # (B, Q_S, Q_N, Dr)
    key: np.ndarray             # (block_num, block_size, 1, D)
    key_rope: np.ndarray        # (block_num, block_size, 1, Dr)
    value: np.ndarray           # (block_num, block_size, 1, D)
    sparse_indices: np.ndarray  # (B, Q_S, 1, sparse_size) int32
    block_table: np.ndarray     # (B, cols) int32
    actual_seq_lengths_kv: np.ndarray  # (B,) int32
    scale: float
    dtype: str = "bf16"
    sparse_block_size: int = 1  # > 1: each index selects that many consecutive tokens
    sparse_mode: int = 0        # 3: right-down causal over the Q_S query tokens
    actual_seq_lengths_query: Optional[np.ndarray] = None  # (B,) int32, None: every query token valid
    layout_query: str = "BSND"  # "TND": query (Q_T, Q_N, D), prefix-sum actual_seq_lengths_query
    layout_kv: str = "PA_BSND"  # "BSND": key (B, KV_S, 1, D); "TND": key (KV_T, 1, D), prefix-sum lengths
    meta: Dict[str, Any] = field(default_factory=dict)

    @property
    def B(self) -> int:
        return self.query.shape[0]


def _lengths(rng, B, lo, hi):
    return rng.integers(lo, hi + 1, size=B, dtype=np.int64)


def _block_table(rng, lens, block_size, cols):
    """Random permutation of exactly the blocks the lengths need; -1 elsewhere."""
    need = [(int(l) + block_size - 1) // block_size for l in lens]
    blocknum = max(1, sum(need))
    perm = rng.permutation(blocknum).astype(np.int32)
    bt = np.full((len(lens), cols), -1, dtype=np.int32)
    off = 0
    for b, nb in enumerate(need):
        bt[b, :nb] = perm[off:off + nb]
        off += nb
    return bt, blocknum


def query_shape(layout, B, N, D):
    if layout == "BNSD":
        return (B, N, 1, D)
    if layout == "BSND":
        return (B, 1, N, D)
    return (B, 1, N * D)


def kv_shape(layout, B, KV_N, S, D):
    if layout == "BNSD":
        return (B, KV_N, S, D)
    if layout == "BSND":
        return (B, S, KV_N, D)
    return (B, S, KV_N * D)


def tiny_mha(seed: int = 0, B=1, N=8, D=64, S=128, dtype="fp16") -> IfaCase:
    lens = np.full(B, S, dtype=np.int64)
    return IfaCase("tiny_mha", random_storage(seed, 1, query_shape("BNSD", B, N, D), dtype),
                   random_storage(seed, 2, kv_shape("BNSD", B, N, S, D), dtype),
                   random_storage(seed, 3, kv_shape("BNSD", B, N, S, D), dtype),
                   num_heads=N, num_kv_heads=N, scale=1.0 / math.sqrt(D), layout="BNSD",
                   q_dtype=dtype, kv_dtype=dtype, max_seq_len=S, actual_seq_lengths=lens)


def gqa_padded(seed: int = 0, B=16, N=32, KV_N=8, D=128, Smax=4096, layout="BSH", dtype="bf16",
               mask=True, len_lo=1, len_hi=None) -> IfaCase:
    rng = np.random.default_rng(seed)
    lens = _lengths(rng, B, len_lo, Smax if len_hi is None else len_hi)
    m = None
    if mask:
        m = (np.arange(Smax)[None, :] >= lens[:, None]).reshape(B, 1, 1, Smax)
    return IfaCase("gqa_padded", random_storage(seed, 1, query_shape(layout, B, N, D), dtype),
                   random_storage(seed, 2, kv_shape(layout, B, KV_N, Smax, D), dtype),
                   random_storage(seed, 3, kv_shape(layout, B, KV_N, Smax, D), dtype),
                   num_heads=N, num_kv_heads=KV_N, scale=1.0 / math.sqrt(D), layout=layout,
                   q_dtype=dtype, kv_dtype=dtype, max_seq_len=Smax, atten_mask=m,
                   actual_seq_lengths=lens)


def paged_gqa(seed: int = 0, B=64, N=32, KV_N=8, D=128, block_size=128, len_lo=512,
              len_hi=32768, dtype="bf16", kv_format="paged_nbsd", bt_cols=None) -> IfaCase:
    rng = np.random.default_rng(seed)
    lens = _lengths(rng, B, len_lo, len_hi)
    cols = bt_cols or (len_hi + block_size - 1) // block_size
    bt, blocknum = _block_table(rng, lens, block_size, cols)
    if kv_format == "paged_nbsd":
        shape = (blocknum, KV_N, block_size, D)
    else:
        shape = (blocknum, block_size, KV_N * D)
    return IfaCase("paged_gqa", random_storage(seed, 1, (B, N, 1, D), dtype),
                   random_storage(seed, 2, shape, dtype), random_storage(seed, 3, shape, dtype),
                   num_heads=N, num_kv_heads=KV_N, scale=1.0 / math.sqrt(D), layout="BNSD",
                   kv_format=kv_format, q_dtype=dtype, kv_dtype=dtype, block_size=block_size,
                   block_table=bt, actual_seq_lengths=lens, meta={"blocknum": blocknum})


def int8_paged(seed: int = 0, B=4, N=16, KV_N=4, D=128, block_size=64, len_lo=1, len_hi=1024,
               kv_format="paged_nbsd", q_dtype="fp16") -> IfaCase:
    """int8 key/value in a paged cache (per-channel antiquant), blocks a random permutation."""
    rng = np.random.default_rng(seed)
    lens = _lengths(rng, B, len_lo, len_hi)
    cols = (len_hi + block_size - 1) // block_size
    bt, blocknum = _block_table(rng, lens, block_size, cols)
    shape = (blocknum, KV_N, block_size, D) if kv_format == "paged_nbsd" else (blocknum, block_size, KV_N * D)
    scale = to_storage(rng.uniform(0.005, 0.02, size=(2, KV_N, 1, D)).astype(np.float32), q_dtype)
    offset = to_storage(rng.uniform(-4.0, 4.0, size=(2, KV_N, 1, D)).astype(np.float32), q_dtype)
    return IfaCase("int8_paged", random_storage(seed, 1, (B, N, 1, D), q_dtype),
                   uniform_int8(seed, 2, shape), uniform_int8(seed, 3, shape),
                   num_heads=N, num_kv_heads=KV_N, scale=1.0 / math.sqrt(D), layout="BNSD",
                   kv_format=kv_format, q_dtype=q_dtype, kv_dtype="int8", block_size=block_size,
                   block_table=bt, actual_seq_lengths=lens, antiquant="per_channel",
                   antiquant_scale=scale, antiquant_offset=offset, meta={"blocknum": blocknum})


def int8_leftpad(seed: int = 0, B=32, N=64, KV_N=8, D=128, Smax=8192, len_lo=256, len_hi=8192,
                 pad_extra=64, per_tensor=False, q_dtype="fp16") -> IfaCase:
    rng = np.random.default_rng(seed)
    lens = _lengths(rng, B, len_lo, len_hi)
    u = rng.integers(0, pad_extra + 1, size=B, dtype=np.int64)
    pads = Smax - lens - u  # may be negative near Smax; the operator clamps it
    pshape = (2,) if per_tensor else (2, KV_N, 1, D)
    scale = to_storage(rng.uniform(0.005, 0.02, size=pshape).astype(np.float32), q_dtype)
    offset = to_storage(rng.uniform(-4.0, 4.0, size=pshape).astype(np.float32), q_dtype)
    return IfaCase("int8_leftpad", random_storage(seed, 1, (B, N, 1, D), q_dtype),
                   uniform_int8(seed, 2, (B, KV_N, Smax, D)),
                   uniform_int8(seed, 3, (B, KV_N, Smax, D)),
                   num_heads=N, num_kv_heads=KV_N, scale=1.0 / math.sqrt(D), layout="BNSD",
                   q_dtype=q_dtype, kv_dtype="int8", max_seq_len=Smax, actual_seq_lengths=lens,
                   kv_padding_size=pads, antiquant="per_tensor" if per_tensor else "per_channel",
                   antiquant_scale=scale, antiquant_offset=offset)


def sfa_mla(seed: int = 0, B=32, Q_N=128, D=512, Dr=64, block_size=64, kv_len=32768,
            sparse_size=2048, nvalid_lo=1024, nvalid_hi=2048, dtype="bf16", sparse_block_size=1, Q_S=1,
            sparse_mode=0, q_lens=None) -> SfaCase:
    """Indices of each (batch, query token) row are distinct and valid first, then -1; with
    sparse_block_size > 1 they are block indices below kv_len / sparse_block_size.  Q_S query
    tokens per batch (multi-token prediction); q_lens: valid query tokens per batch, or None."""
    rng = np.random.default_rng(seed)
    cols = (kv_len + block_size - 1) // block_size
    block_num = B * cols
    bt = rng.permutation(block_num).astype(np.int32).reshape(B, cols)
    idx = np.full((B, Q_S, 1, sparse_size), -1, dtype=np.int32)
    n_units = kv_len // sparse_block_size
    for b in range(B):
        for s in range(Q_S):
            nv = int(rng.integers(nvalid_lo, nvalid_hi + 1))
            idx[b, s, 0, :nv] = rng.choice(n_units, size=nv, replace=False).astype(np.int32)
    lens = np.full(B, kv_len, dtype=np.int32)
    lq = None if q_lens is None else np.asarray(q_lens, dtype=np.int32).reshape(B)
    return SfaCase("sfa_mla", random_storage(seed, 1, (B, Q_S, Q_N, D), dtype),
                   random_storage(seed, 4, (B, Q_S, Q_N, Dr), dtype),
                   random_storage(seed, 2, (block_num, block_size, 1, D), dtype),
                   random_storage(seed, 5, (block_num, block_size, 1, Dr), dtype),
                   random_storage(seed, 3, (block_num, block_size, 1, D), dtype),
                   idx, bt, lens, scale=1.0 / math.sqrt(D + Dr), dtype=dtype,
                   sparse_block_size=sparse_block_size, sparse_mode=sparse_mode, actual_seq_lengths_query=lq)


def sfa_relayout(case: SfaCase, layout_query: str = "BSND", layout_kv: str = "PA_BSND") -> SfaCase:
    """The same problem with its query rows and/or key rows stored in another layout (data
    movement only).  Query TND: each batch's valid query rows (actual_seq_lengths_query, or
    all Q_S) packed in order, the lengths becoming prefix sums.  Key BSND: (B, KV_S, 1, d)
    with KV_S the longest length; key TND: each batch's tokens packed in order, the lengths
    becoming prefix sums.  Tokens are read from the paged caches through the block table."""
    from copy import copy
    c = copy(case)
    B, Q_S = case.query.shape[0], case.query.shape[1]
    if layout_query == "TND":
        qlen = (np.full(B, Q_S, dtype=np.int64) if case.actual_seq_lengths_query is None
                else case.actual_seq_lengths_query.astype(np.int64))
        rows = [(b, s) for b in range(B) for s in range(int(qlen[b]))]
        c.query = np.stack([case.query[b, s] for b, s in rows]) if rows else case.query[:0, 0]
        c.query_rope = np.stack([case.query_rope[b, s] for b, s in rows]) if rows else case.query_rope[:0, 0]
        c.sparse_indices = (np.stack([case.sparse_indices[b, s] for b, s in rows]) if rows
                            else case.sparse_indices[:0, 0])
        c.actual_seq_lengths_query = np.cumsum(qlen).astype(np.int32)
        c.layout_query = "TND"
    if layout_kv != "PA_BSND":
        bs = case.key.shape[1]
        lens = case.actual_seq_lengths_kv.astype(np.int64)

        def rows_of(b, n):
            t = np.arange(n)
            return case.block_table[b, t // bs].astype(np.int64) * bs + t % bs

        flat = [a.reshape(-1, a.shape[-1]) for a in (case.key, case.key_rope, case.value)]
        if layout_kv == "BSND":
            kv_s = int(lens.max()) if B else 1
            outs = [np.zeros((B, kv_s, 1, f.shape[-1]), dtype=f.dtype) for f in flat]
            for b in range(B):
                r = rows_of(b, int(lens[b]))
                for o, f in zip(outs, flat):
                    o[b, :len(r), 0] = f[r]
            c.key, c.key_rope, c.value = outs
        else:
            r = np.concatenate([rows_of(b, int(lens[b])) for b in range(B)]) if B else np.zeros(0, np.int64)
            c.key, c.key_rope, c.value = [f[r][:, None, :] for f in flat]
            c.actual_seq_lengths_kv = np.cumsum(lens).astype(np.int32)
        c.block_table = None
        c.layout_kv = layout_kv
    return c


@dataclass
class AppendCase:
    """One decode step's KV-cache append: the new token's rows of every batch and the caches."""
    name: str
    key_new: np.ndarray          # (B, KV_N, D), dtype
    value_new: np.ndarray
    positions: np.ndarray        # (B,) int64: token index of the new token
    key_cache: np.ndarray        # contiguous (B, KV_N, Smax, D) BNSD, or paged (blocknum, KV_N, bs, D)
    value_cache: np.ndarray
    layout: str = "BNSD"
    kv_format: str = "contig"
    block_size: int = 0
    block_table: Optional[np.ndarray] = None
    dtype: str = "bf16"
    kv_dtype: str = "bf16"
    antiquant: str = "none"
    antiquant_scale: Optional[np.ndarray] = None
    antiquant_offset: Optional[np.ndarray] = None
    meta: Dict[str, Any] = field(default_factory=dict)

    @property
    def B(self) -> int:
        return self.key_new.shape[0]


def kv_append_paged(seed: int = 0, B=64, KV_N=8, D=128, block_size=128, len_lo=512, len_hi=4096,
                    dtype="bf16") -> AppendCase:
    """Append at each batch's length into a paged (blocknum, KV_N, blockSize, D) cache whose
    block table (a random permutation of physical blocks) covers length + 1 tokens."""
    rng = np.random.default_rng(seed)
    lens = _lengths(rng, B, len_lo, len_hi)
    cols = (len_hi + 1 + block_size - 1) // block_size
    bt, blocknum = _block_table(rng, lens + 1, block_size, cols)
    shape = (blocknum, KV_N, block_size, D)
    return AppendCase("kv_append_paged", random_storage(seed, 1, (B, KV_N, D), dtype),
                      random_storage(seed, 2, (B, KV_N, D), dtype), lens.astype(np.int64),
                      np.zeros(shape, dtype=np.uint16 if dtype == "bf16" else np.float16),
                      np.zeros(shape, dtype=np.uint16 if dtype == "bf16" else np.float16),
                      layout="BNSD", kv_format="paged_nbsd", block_size=block_size, block_table=bt,
                      dtype=dtype, kv_dtype=dtype)


def kv_append_int8(seed: int = 0, B=32, KV_N=8, D=128, Smax=8192, dtype="fp16") -> AppendCase:
    """Append into a contiguous BNSD int8 cache with per-channel antiquant parameters (the
    int8 workload's shapes and parameter distributions), at positions U{256..Smax-1}."""
    rng = np.random.default_rng(seed)
    pos = rng.integers(256, Smax, size=B).astype(np.int64)
    scale = to_storage(rng.uniform(0.005, 0.02, size=(2, KV_N, 1, D)).astype(np.float32), dtype)
    offset = to_storage(rng.uniform(-4, 4, size=(2, KV_N, 1, D)).astype(np.float32), dtype)
    shape = (B, KV_N, Smax, D)
    return AppendCase("kv_append_int8", random_storage(seed, 1, (B, KV_N, D), dtype),
                      random_storage(seed, 2, (B, KV_N, D), dtype), pos, np.zeros(shape, dtype=np.int8),
                      np.zeros(shape, dtype=np.int8), layout="BNSD", kv_format="contig", dtype=dtype,
                      kv_dtype="int8", antiquant="per_channel", antiquant_scale=scale, antiquant_offset=offset)


def tensorlist_from(case: IfaCase, seed: int = 0, extra_hi: int = 0) -> IfaCase:
    """The same problem with key/value as one tensor per batch (data movement, plus random
    tokens past each length): tensor b holds batch b's first len_b + U{0..extra_hi} tokens of
    a contiguous case, in its layout, so S_b differs from batch to batch.  The case's
    key/value become lists and its kv_format "tensorlist"."""
    from copy import copy
    assert case.kv_format == "contig" and case.kv_padding_size is None
    rng = np.random.default_rng(seed)
    c = copy(case)
    s_axis = 2 if case.layout == "BNSD" else 1
    lens = (case.actual_seq_lengths if case.actual_seq_lengths is not None
            else np.full(case.B, case.key.shape[s_axis], dtype=np.int64))
    keys, values = [], []
    for b in range(case.B):
        S_b = int(min(case.key.shape[s_axis], max(1, int(lens[b]) + int(rng.integers(0, extra_hi + 1)))))
        sl = [slice(b, b + 1)] + [slice(None)] * (case.key.ndim - 1)
        sl[s_axis] = slice(0, S_b)
        keys.append(np.ascontiguousarray(case.key[tuple(sl)]))
        values.append(np.ascontiguousarray(case.value[tuple(sl)]))
    c.key, c.value = keys, values
    c.kv_format = "tensorlist"
    c.max_seq_len = max(k.shape[s_axis] for k in keys)
    return c
