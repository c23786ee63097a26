"""CPU oracle for single-query decode attention (IncreFlashAttention) and for
sparse-index MLA-absorb decode (SparseFlashAttention).

TEST INFRASTRUCTURE: only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package.  The product path (the
CUDA library and its binding) never loads it, and this package imports
nothing from the product.

The arithmetic lives in ``ifa_oracle.c`` (plain double-precision loops, see
its header for the definitions and readings).  This module compiles it with
gcc on first use and marshals numpy arrays into it.

Dtype conventions of the inputs (shared with the seeded input generators):
fp16 arrays are ``numpy.float16``; bf16 arrays are ``numpy.uint16`` holding
the bf16 bit patterns; int8 arrays are ``numpy.int8``; masks are one byte per
element (bool, int8 or uint8), nonzero meaning "excluded".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ifa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libifa_oracle.so")
_lock = threading.Lock()
_lib = None

F16, BF16, I8 = 0, 1, 2
BSH, BSND, BNSD = 0, 1, 2
CONTIG, PAGED_NBSD, PAGED_BSH = 0, 1, 2
AQ_NONE, AQ_PER_CHANNEL, AQ_PER_TENSOR = 0, 1, 2

_LAYOUT = {"BSH": BSH, "BSND": BSND, "BNSD": BNSD}


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build`` (plain C, -O2, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-Wall",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _SfaArgs(ctypes.Structure):
    """Mirror of the oracle's orc_sfa argument block (ifa_oracle.c)."""
    _fields_ = [(n, ctypes.c_int64) for n in (
        "B", "Q_S", "Q_T", "Q_N", "D", "Dr", "layout_q", "layout_kv", "kv_s", "block_size", "block_num",
        "bt_cols", "sparse_size", "sparse_block_size", "sparse_mode", "dtype")] + [("scale", ctypes.c_double)] + [
        (n, ctypes.c_void_p) for n in ("q", "q_rope", "k", "k_rope", "v", "indices", "block_table", "lens_kv",
                                       "lens_q", "out", "softmax_max", "softmax_sum")]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, ip, vp, dp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_double
            lib.ifa_oracle_run.restype = ctypes.c_int
            lib.ifa_oracle_run.argtypes = [i64, i64, i64, i64, ip, ip, ip, ip, i64, i64, i64, i64,
                                           vp, vp, vp, vp, i64, i64, i64, vp, vp, i64, vp, ip,
                                           vp, vp, dp, vp]
            lib.sfa_oracle_run.restype = ctypes.c_int
            lib.sfa_oracle_run.argtypes = [ctypes.POINTER(_SfaArgs)]
            lib.ifa_quantize_output.restype = ctypes.c_int
            lib.ifa_quantize_output.argtypes = [i64, i64, i64, vp, ip, ip, vp, vp, vp]
            lib.kv_append_oracle.restype = ctypes.c_int
            lib.kv_append_oracle.argtypes = [i64, i64, i64, ip, ip, ip, ip, i64, i64, i64, i64, vp, vp, vp, vp, ip,
                                             vp, vp, vp, vp]
            _lib = lib
    return _lib


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float16:
        return F16
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.int8:
        return I8
    raise TypeError(f"unsupported oracle input dtype {a.dtype}")


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype=None):
    if a is None:
        return None
    a = np.ascontiguousarray(a if dtype is None else np.asarray(a, dtype=dtype))
    return a


def ifa_ref(query, key, value, *, num_heads, num_kv_heads=0, scale, layout="BNSD",
            kv_format=CONTIG, block_size=0, block_table=None, atten_mask=None,
            actual_seq_lengths=None, kv_padding_size=None, antiquant=AQ_NONE,
            antiquant_scale=None, antiquant_offset=None, return_bad_tokens=False):
    """Reference output, float64 array of shape (B, numHeads, D); with return_bad_tokens,
    also the number of window tokens whose block-table entry lies outside [0, blocknum).

    query: (B,N,1,D) BNSD, (B,1,N,D) BSND or (B,1,H) BSH.
    key/value: contiguous in the same layout, or a paged cache
    (blocknum, KV_N, blockSize, D) for ``PAGED_NBSD`` / (blocknum, blockSize, H)
    for ``PAGED_BSH``.  atten_mask: (Bm, Nm, 1, S) with Bm in {1, B}, Nm in
    {1, numHeads}.  antiquant_scale/offset: (2, KV_N, D)-shaped memory
    (per channel) or (2,) (per tensor), in the query dtype.
    """
    lib = _load()
    q = _c(query)
    k = _c(key)
    v = _c(value)
    B = q.shape[0]
    N = int(num_heads)
    kvn = int(num_kv_heads) or N
    D = q.size // (B * N)
    lay = _LAYOUT[layout]
    if kv_format == CONTIG:
        if lay == BNSD:
            smax = k.shape[2]
        else:
            smax = k.shape[1]
        block_num = 0
        bt_cols = 0
    else:
        block_num = k.shape[0]
        smax = 0
        bt_cols = np.asarray(block_table).shape[1]
    bt = _c(block_table, np.int32) if block_table is not None else None
    m = None
    mB = mN = mS = 0
    if atten_mask is not None:
        m = _c(atten_mask).view(np.uint8)
        mB, mN, mS = m.shape[0], m.shape[1], m.shape[-1]
    lens = _c(actual_seq_lengths, np.int64)
    pads = _c(kv_padding_size, np.int64)
    if pads is not None:
        pads = pads.reshape(-1)
    sc = _c(antiquant_scale)
    of = _c(antiquant_offset)
    out = np.zeros((B, N, D), dtype=np.float64)
    rc = lib.ifa_oracle_run(B, N, kvn, D, _dtype_code(q), _dtype_code(k), lay, kv_format, smax,
                            int(block_size), bt_cols, block_num, _ptr(q), _ptr(k), _ptr(v),
                            _ptr(m), mB, mN, mS, _ptr(lens), _ptr(pads),
                            0 if pads is None else pads.size, _ptr(bt), int(antiquant),
                            _ptr(sc), _ptr(of), float(scale), _ptr(out))
    if rc < 0:
        raise ValueError("oracle rejected its arguments")
    return (out, rc) if return_bad_tokens else out


SFA_LAYOUT_Q = {"BSND": 0, "TND": 1}
SFA_LAYOUT_KV = {"PA_BSND": 0, "BSND": 1, "TND": 2}


def sfa_ref(query, query_rope, key, key_rope, value, sparse_indices, block_table,
            actual_seq_lengths_kv, *, scale, sparse_block_size=1, sparse_mode=0, actual_seq_lengths_query=None,
            layout_query="BSND", layout_kv="PA_BSND", return_softmax_lse=False):
    """Reference sparse MLA-absorb decode output, float64.

    layout_query BSND: query (B,Q_S,Q_N,D), query_rope (B,Q_S,Q_N,Dr), sparse_indices
    (B,Q_S,1,sparse_size), output (B,Q_S,Q_N,D), or (B,Q_N,D) when Q_S = 1;
    actual_seq_lengths_query (B,) int32 or None.  TND: query (Q_T,Q_N,D), query_rope
    (Q_T,Q_N,Dr), sparse_indices (Q_T,1,sparse_size), output (Q_T,Q_N,D);
    actual_seq_lengths_query holds prefix sums (its length is B).
    layout_kv PA_BSND: key/value (block_num, block_size, 1, D), key_rope (block_num,
    block_size, 1, Dr), block_table (B, cols), actual_seq_lengths_kv (B,).  BSND: key
    (B, KV_S, 1, D), actual_seq_lengths_kv (B,) or None; TND: key (KV_T, 1, D),
    actual_seq_lengths_kv prefix sums.  sparse_block_size > 1: each index selects that many
    consecutive tokens; sparse_mode 3: right-down causal over each batch's query tokens.
    return_softmax_lse: also return softmax_max and softmax_sum, one value per (row, head),
    shaped like the output without its last axis.
    """
    lib = _load()
    lq_code, lkv_code = SFA_LAYOUT_Q[layout_query], SFA_LAYOUT_KV[layout_kv]
    q = _c(query)
    qr = _c(query_rope)
    k = _c(key)
    kr = _c(key_rope)
    v = _c(value)
    idx = _c(sparse_indices, np.int32)
    bt = None if block_table is None else _c(block_table, np.int32)
    lens = None if actual_seq_lengths_kv is None else _c(actual_seq_lengths_kv, np.int32)
    lq = None if actual_seq_lengths_query is None else _c(actual_seq_lengths_query, np.int32)
    a = _SfaArgs()
    if lq_code == 0:
        a.B, a.Q_S, a.Q_N, a.D = q.shape[0], q.shape[1], q.shape[2], q.shape[3]
        rows = a.B * a.Q_S
        Dr = qr.shape[3]
        lead = (a.B, a.Q_S)
    else:
        a.Q_T, a.Q_N, a.D = q.shape[0], q.shape[1], q.shape[2]
        a.B = lq.shape[0]
        rows = a.Q_T
        Dr = qr.shape[2]
        lead = (a.Q_T,)
    a.Dr = Dr
    a.layout_q, a.layout_kv = lq_code, lkv_code
    if lkv_code == 0:
        a.block_num, a.block_size = k.shape[0], k.shape[1]
        a.bt_cols = bt.shape[1]
    elif lkv_code == 1:
        a.kv_s = k.shape[1]
    else:
        a.kv_s = k.shape[0]
    a.sparse_size = idx.shape[-1]
    a.sparse_block_size = int(sparse_block_size)
    a.sparse_mode = int(sparse_mode)
    a.dtype = _dtype_code(q)
    a.scale = float(scale)
    out = np.zeros(lead + (a.Q_N, a.D), dtype=np.float64)
    smax = np.zeros(lead + (a.Q_N,), dtype=np.float64)
    ssum = np.zeros(lead + (a.Q_N,), dtype=np.float64)
    a.q, a.q_rope, a.k, a.k_rope, a.v = _ptr(q), _ptr(qr), _ptr(k), _ptr(kr), _ptr(v)
    a.indices, a.block_table, a.lens_kv, a.lens_q = _ptr(idx), _ptr(bt), _ptr(lens), _ptr(lq)
    a.out, a.softmax_max, a.softmax_sum = _ptr(out), _ptr(smax), _ptr(ssum)
    assert idx.size == rows * a.sparse_size
    rc = lib.sfa_oracle_run(ctypes.byref(a))
    if rc < 0:
        raise ValueError("oracle rejected its arguments")
    if lq_code == 0 and a.Q_S == 1:
        out, smax, ssum = out[:, 0], smax[:, 0], ssum[:, 0]
    return (out, smax, ssum) if return_softmax_lse else out


def kv_append_ref(key_new, value_new, positions, key_cache, value_cache, *, layout="BNSD", kv_format=CONTIG,
                  block_size=0, block_table=None, antiquant=AQ_NONE, antiquant_scale=None, antiquant_offset=None):
    """Caches after appending one token per batch, as new arrays (the inputs are not modified),
    and the number of batches whose position lies outside the cache.

    key_new/value_new: (B, KV_N, D) in memory (any query-style layout with S = 1), fp16 or
    bf16.  key_cache/value_cache: contiguous (B,KV_N,Smax,D) BNSD, (B,Smax,KV_N,D) BSND or
    (B,Smax,H) BSH; or paged (blocknum, KV_N, blockSize, D) / (blocknum, blockSize, H); fp16,
    bf16 or int8.  positions: (B,) int64 token index of the new token.
    """
    lib = _load()
    kn = _c(key_new)
    vn = _c(value_new)
    kc = np.array(key_cache, copy=True, order="C")
    vc = np.array(value_cache, copy=True, order="C")
    pos = _c(positions, np.int64)
    bt = _c(block_table, np.int32) if block_table is not None else None
    sc = _c(antiquant_scale)
    of = _c(antiquant_offset)
    B = pos.shape[0]
    lay = _LAYOUT[layout]
    if kv_format == CONTIG:
        kvn = kc.shape[1] if lay == BNSD else (kc.shape[2] if lay == BSND else kn.size // (B * kn.shape[-1]))
        smax = kc.shape[2] if lay == BNSD else kc.shape[1]
        block_num, cols = 0, 0
    else:
        kvn = kn.size // (B * kn.shape[-1])
        smax, block_num, cols = 0, kc.shape[0], bt.shape[1]
    D = kn.size // (B * kvn)
    rc = lib.kv_append_oracle(B, kvn, D, _dtype_code(kn), _dtype_code(kc), lay, kv_format, smax, int(block_size),
                              cols, block_num, _ptr(kn), _ptr(vn), _ptr(pos), _ptr(bt), int(antiquant), _ptr(sc),
                              _ptr(of), _ptr(kc), _ptr(vc))
    if rc < 0:
        raise ValueError("oracle rejected its arguments")
    return kc, vc, rc


def quantize_output_ref(y, scale2, offset2=None):
    """int8 codes of an attention output y (B, N, D) (float64, rounded to float32 first):
    saturate(rint(y * scale2 + offset2)) with single-precision product and sum.  scale2 /
    offset2: float32 or bf16 bit patterns (uint16); one entry (per tensor) or N * D entries
    (per channel, head-major)."""
    lib = _load()
    yy = np.ascontiguousarray(y, dtype=np.float64)
    B, N, D = yy.shape
    sc = np.ascontiguousarray(scale2)
    of = None if offset2 is None else np.ascontiguousarray(offset2)
    code = 3 if sc.dtype == np.float32 else (BF16 if sc.dtype == np.uint16 else None)
    if code is None or (of is not None and of.dtype != sc.dtype):
        raise TypeError("scale2/offset2 must be float32 or bf16 bit patterns, of one dtype")
    per_channel = sc.size != 1
    if per_channel and sc.size != N * D:
        raise ValueError("per-channel scale2 needs N * D entries")
    out = np.zeros((B, N, D), dtype=np.int8)
    rc = lib.ifa_quantize_output(B, N, D, _ptr(yy), int(per_channel), code, _ptr(sc), _ptr(of), _ptr(out))
    if rc < 0:
        raise ValueError("oracle rejected its arguments")
    return out


def ifa_ref_tensorlist(query, key_list, value_list, *, num_heads, num_kv_heads=0, scale, layout="BNSD",
                       atten_mask=None, actual_seq_lengths=None, antiquant=AQ_NONE, antiquant_scale=None,
                       antiquant_offset=None):
    """Reference output (B, numHeads, D) with key/value given as one tensor per batch
    (IncreFlashAttention README, non-contiguous key/value: B tensors of batch 1 whose shapes
    differ only in S): batch b is the one-batch problem over its own tensor, tokens
    [0, actual_seq_lengths[b]) (all of its S_b when the lengths are None); a per-batch mask
    row is batch b's."""
    B = query.shape[0]
    outs = []
    for b in range(B):
        m = None
        if atten_mask is not None:
            m = atten_mask[b:b + 1] if atten_mask.shape[0] > 1 else atten_mask
        lens = None if actual_seq_lengths is None else np.asarray(actual_seq_lengths, dtype=np.int64)[b:b + 1]
        outs.append(ifa_ref(query[b:b + 1], key_list[b], value_list[b], num_heads=num_heads,
                            num_kv_heads=num_kv_heads, scale=scale, layout=layout, atten_mask=m,
                            actual_seq_lengths=lens, antiquant=antiquant, antiquant_scale=antiquant_scale,
                            antiquant_offset=antiquant_offset)[0])
    return np.stack(outs)
