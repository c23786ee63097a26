"""Python binding of ``libifa.so`` (C ABI declared in ``include/ifa.h``).

The functions below carry the C names and only marshal arguments: every step
of the computation runs in the library's CUDA kernels.  torch supplies device
memory and streams.  Loading fails loudly if the library has not been built;
there is no fallback implementation.

``IncreFlashAttention`` wraps a plan: construct it with the static problem
description, then call it with device tensors and host length arrays.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libifa.so")

IFA_OK = 0
IFA_ERR_PARAM_NULLPTR = 161001
IFA_ERR_PARAM_INVALID = 161002
IFA_ERR_RUNTIME = 361001

LAYOUTS = {"BSH": 0, "BSND": 1, "BNSD": 2}
KV_FORMATS = {"contig": 0, "paged_nbsd": 1, "paged_bsh": 2, "tensorlist": 3}
DTYPES = {"fp16": 0, "bf16": 1, "int8": 2, "uint8": 3, "bool": 4, "fp32": 5}
ANTIQUANT = {"none": 0, "per_channel": 1, "per_tensor": 2}

# Every symbol include/ifa.h declares.
EXPORTED = ("ifa_create", "ifa_run", "ifa_destroy", "ifa_get_device_errors", "ifa_last_launch_count",
            "ifa_run_noalloc", "ifa_run_tensorlist", "sfa_workspace_size", "sfa_run", "ifa_kv_append",
            "ifa_status_string")

# Fixed scratch of ifa_run_noalloc (include/ifa.h).
IFA_NOALLOC_SCRATCH_BYTES = 4 << 20
IFA_NOALLOC_MAX_BATCH = 256


class IfaParams(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int64), ("numHeads", ctypes.c_int64), ("numKeyValueHeads", ctypes.c_int64),
        ("headDim", ctypes.c_int64), ("maxSeqLen", ctypes.c_int64),
        ("q_dtype", ctypes.c_int32), ("kv_dtype", ctypes.c_int32),
        ("inputLayout", ctypes.c_int32), ("kvFormat", ctypes.c_int32),
        ("blockSize", ctypes.c_int64), ("blockNum", ctypes.c_int64), ("blockTableCols", ctypes.c_int64),
        ("has_mask", ctypes.c_int32), ("mask_dtype", ctypes.c_int32),
        ("maskB", ctypes.c_int64), ("maskN", ctypes.c_int64), ("maskS", ctypes.c_int64),
        ("antiquant", ctypes.c_int32), ("has_kv_padding", ctypes.c_int32),
        ("scaleValue", ctypes.c_double), ("splitTiles", ctypes.c_int64),
        ("out_dtype", ctypes.c_int32), ("quant2", ctypes.c_int32), ("quant2_dtype", ctypes.c_int32),
    ]


class SfaParams(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "B", "Q_S", "Q_T", "Q_N", "KV_N", "D", "Dr", "KV_S", "block_size", "block_num", "block_table_cols",
        "sparse_size", "sparse_block_size")] + [(n, ctypes.c_int32) for n in (
            "dtype", "sparse_mode", "layout_query", "layout_kv")] + [("scale_value", ctypes.c_double)]


class AppendParams(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "B", "numKeyValueHeads", "headDim", "maxSeqLen", "blockSize", "blockNum", "blockTableCols")] + [
        (n, ctypes.c_int32) for n in ("new_dtype", "kv_dtype", "inputLayout", "kvFormat", "antiquant")]


SFA_LAYOUT_QUERY = {"BSND": 0, "TND": 1}
SFA_LAYOUT_KV = {"PA_BSND": 0, "BSND": 1, "TND": 2}


_lib = None
_lock = threading.Lock()


class IfaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: status {status} ({status_string(status)})")
        self.status = status


def load_library():
    """Open libifa.so (built by ``kv_cache_incremental_split_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: run kv_cache_incremental_split_gb300.build first")
            lib = ctypes.CDLL(LIB_PATH)
            vp, sz, i64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int64
            lib.ifa_create.restype = ctypes.c_int32
            lib.ifa_create.argtypes = [ctypes.POINTER(IfaParams), ctypes.POINTER(vp), ctypes.POINTER(sz)]
            lib.ifa_run.restype = ctypes.c_int32
            lib.ifa_run.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, vp, vp, vp, vp, vp, vp, vp, sz, vp]
            lib.ifa_run_tensorlist.restype = ctypes.c_int32
            lib.ifa_run_tensorlist.argtypes = [vp, vp, ctypes.POINTER(vp), ctypes.POINTER(vp), vp, vp, vp, vp, vp,
                                               vp, vp, vp, vp, sz, vp]
            lib.ifa_destroy.restype = ctypes.c_int32
            lib.ifa_destroy.argtypes = [vp]
            lib.ifa_get_device_errors.restype = ctypes.c_int32
            lib.ifa_get_device_errors.argtypes = [vp, vp, ctypes.POINTER(i64)]
            lib.ifa_last_launch_count.restype = ctypes.c_int64
            lib.ifa_last_launch_count.argtypes = [vp]
            lib.ifa_run_noalloc.restype = ctypes.c_int32
            lib.ifa_run_noalloc.argtypes = [ctypes.POINTER(IfaParams), vp, vp, vp, vp, vp, vp, i64, vp, vp, vp,
                                            vp, vp, vp, vp, vp]
            lib.sfa_workspace_size.restype = ctypes.c_int32
            lib.sfa_workspace_size.argtypes = [ctypes.POINTER(SfaParams), ctypes.POINTER(sz)]
            lib.ifa_kv_append.restype = ctypes.c_int32
            lib.ifa_kv_append.argtypes = [ctypes.POINTER(AppendParams), vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
            lib.sfa_run.restype = ctypes.c_int32
            lib.sfa_run.argtypes = [ctypes.POINTER(SfaParams), vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                    sz, vp, vp]
            lib.ifa_status_string.restype = ctypes.c_char_p
            lib.ifa_status_string.argtypes = [ctypes.c_int32]
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load_library().ifa_status_string(int(status)).decode()


def ifa_create(params: IfaParams):
    """Returns (status, plan handle or None, workspace bytes)."""
    lib = load_library()
    plan = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    st = lib.ifa_create(ctypes.byref(params), ctypes.byref(plan), ctypes.byref(ws))
    return st, (plan.value if st == IFA_OK else None), ws.value


def ifa_run(plan, query, key, value, atten_mask, actual_seq_lengths, kv_padding_size, n_kv_padding,
            block_table, antiquant_scale, antiquant_offset, attention_out, workspace, workspace_bytes,
            stream, quant_scale2=None, quant_offset2=None) -> int:
    """All pointer arguments are integers (device addresses, or host addresses for
    ``actual_seq_lengths`` / ``kv_padding_size``) or None."""
    return load_library().ifa_run(plan, query, key, value, atten_mask, actual_seq_lengths, kv_padding_size,
                                   n_kv_padding, block_table, antiquant_scale, antiquant_offset, quant_scale2,
                                   quant_offset2, attention_out, workspace, workspace_bytes, stream)


def ifa_run_noalloc(params: IfaParams, query, key, value, atten_mask, actual_seq_lengths, kv_padding_size,
                    n_kv_padding, block_table, antiquant_scale, antiquant_offset, attention_out,
                    device_error_flags, stream, quant_scale2=None, quant_offset2=None) -> int:
    """Plan-less, allocation-free call (include/ifa.h): for callers that cannot
    allocate device memory.  Pointer arguments are integers or None."""
    return load_library().ifa_run_noalloc(ctypes.byref(params), query, key, value, atten_mask,
                                          actual_seq_lengths, kv_padding_size, n_kv_padding, block_table,
                                          antiquant_scale, antiquant_offset, quant_scale2, quant_offset2,
                                          attention_out, device_error_flags, stream)


def ifa_run_tensorlist(plan, query, key_list, value_list, kv_seq_lens, atten_mask, actual_seq_lengths,
                       antiquant_scale, antiquant_offset, quant_scale2, quant_offset2, attention_out, workspace,
                       workspace_bytes, stream) -> int:
    """key_list / value_list: sequences of B device addresses; kv_seq_lens and
    actual_seq_lengths: host addresses of int64 arrays (or None); other pointers as ifa_run."""
    n = len(key_list)
    karr = (ctypes.c_void_p * max(1, n))(*key_list)
    varr = (ctypes.c_void_p * max(1, n))(*value_list)
    return load_library().ifa_run_tensorlist(plan, query, karr, varr, kv_seq_lens, atten_mask, actual_seq_lengths,
                                             antiquant_scale, antiquant_offset, quant_scale2, quant_offset2,
                                             attention_out, workspace, workspace_bytes, stream)


def ifa_destroy(plan) -> int:
    return load_library().ifa_destroy(plan)


def ifa_get_device_errors(plan, stream) -> int:
    flags = ctypes.c_int64()
    st = load_library().ifa_get_device_errors(plan, stream, ctypes.byref(flags))
    if st != IFA_OK:
        raise IfaError(st, "ifa_get_device_errors")
    return flags.value


def _ptr(t):
    return None if t is None else int(t.data_ptr())


def _stream_handle(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


class IncreFlashAttention:
    """A plan for one decode-attention problem shape (see ``include/ifa.h``).

    Construction validates the description (``ifa_create``) and allocates the
    device workspace with torch.  Calling the object enqueues ``ifa_run`` on
    the current (or given) torch stream and returns the output tensor.

    Devices: the plan's device state is created on the CUDA device current at
    construction, so construct and call the object with the same device current
    (``device``, when given, must be that device), and pass tensors and streams
    of that device.
    """

    def __init__(self, *, batch: int, num_heads: int, num_kv_heads: int = 0, head_dim: int,
                 max_seq_len: int = 0, dtype: str = "bf16", kv_dtype: Optional[str] = None,
                 layout: str = "BSH", kv_format: str = "contig", block_size: int = 0,
                 block_num: int = 0, block_table_cols: int = 0,
                 mask_shape: Optional[Sequence[int]] = None, mask_dtype: str = "bool",
                 antiquant: str = "none", kv_padding: bool = False,
                 scale: Optional[float] = None, split_tiles: int = 0, out_dtype: Optional[str] = None,
                 quant2: str = "none", quant2_dtype: str = "fp32", device=None):
        import torch
        p = IfaParams()
        p.B, p.numHeads, p.numKeyValueHeads, p.headDim = batch, num_heads, num_kv_heads, head_dim
        p.maxSeqLen = max_seq_len
        p.q_dtype = DTYPES[dtype]
        p.kv_dtype = DTYPES[kv_dtype or dtype]
        p.inputLayout = LAYOUTS[layout]
        p.kvFormat = KV_FORMATS[kv_format]
        p.blockSize, p.blockNum, p.blockTableCols = block_size, block_num, block_table_cols
        if mask_shape is not None:
            p.has_mask = 1
            p.mask_dtype = DTYPES[mask_dtype]
            p.maskB, p.maskN, p.maskS = int(mask_shape[0]), int(mask_shape[1]), int(mask_shape[-1])
        p.antiquant = ANTIQUANT[antiquant]
        p.has_kv_padding = int(bool(kv_padding))
        p.scaleValue = (1.0 / math.sqrt(head_dim)) if scale is None else float(scale)
        p.splitTiles = split_tiles
        self.out_i8 = out_dtype == "int8"
        p.out_dtype = DTYPES["int8"] if self.out_i8 else p.q_dtype
        p.quant2 = ANTIQUANT[quant2]
        p.quant2_dtype = DTYPES[quant2_dtype] if self.out_i8 else 0
        self.params = p
        self.batch, self.num_heads, self.head_dim = batch, num_heads, head_dim
        self.dtype = dtype
        st, plan, ws = ifa_create(p)
        if st != IFA_OK:
            raise IfaError(st, "ifa_create")
        self.plan = plan
        self.workspace_bytes = ws
        dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.device = dev
        self.workspace = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)

    def __del__(self):
        plan = getattr(self, "plan", None)
        if plan is not None and _lib is not None:
            _lib.ifa_destroy(plan)
            self.plan = None

    def __call__(self, query, key, value, *, atten_mask=None, actual_seq_lengths=None,
                 kv_padding_size=None, block_table=None, antiquant_scale=None, antiquant_offset=None,
                 quant_scale2=None, quant_offset2=None, out=None, stream=None):
        import torch
        if out is None:
            out = torch.empty(query.shape, dtype=torch.int8, device=query.device) if self.out_i8 \
                else torch.empty_like(query)
        lens = None if actual_seq_lengths is None else np.ascontiguousarray(actual_seq_lengths, dtype=np.int64)
        if self.params.kvFormat == KV_FORMATS["tensorlist"]:
            # key / value: one tensor per batch; S_b is the token extent of each
            s_axis = 2 if self.params.inputLayout == LAYOUTS["BNSD"] else 1
            slen = np.ascontiguousarray([int(t.shape[s_axis]) for t in key], dtype=np.int64)
            st = ifa_run_tensorlist(self.plan, _ptr(query), [_ptr(t) for t in key], [_ptr(t) for t in value],
                                    slen.ctypes.data, _ptr(atten_mask), None if lens is None else lens.ctypes.data,
                                    _ptr(antiquant_scale), _ptr(antiquant_offset), _ptr(quant_scale2),
                                    _ptr(quant_offset2), _ptr(out), _ptr(self.workspace), self.workspace.numel(),
                                    _stream_handle(stream))
            if st != IFA_OK:
                raise IfaError(st, "ifa_run_tensorlist")
            return out
        pads = None if kv_padding_size is None else np.ascontiguousarray(kv_padding_size, dtype=np.int64).reshape(-1)
        st = ifa_run(self.plan, _ptr(query), _ptr(key), _ptr(value), _ptr(atten_mask),
                     None if lens is None else lens.ctypes.data,
                     None if pads is None else pads.ctypes.data, 0 if pads is None else pads.size,
                     _ptr(block_table), _ptr(antiquant_scale), _ptr(antiquant_offset), _ptr(out),
                     _ptr(self.workspace), self.workspace.numel(), _stream_handle(stream),
                     quant_scale2=_ptr(quant_scale2), quant_offset2=_ptr(quant_offset2))
        if st != IFA_OK:
            raise IfaError(st, "ifa_run")
        return out

    def last_launch_count(self) -> int:
        return int(load_library().ifa_last_launch_count(self.plan))

    def device_errors(self, stream=None) -> int:
        return ifa_get_device_errors(self.plan, _stream_handle(stream))


def sfa_workspace_size(params: SfaParams):
    """Returns (status, workspace bytes)."""
    ws = ctypes.c_size_t()
    st = load_library().sfa_workspace_size(ctypes.byref(params), ctypes.byref(ws))
    return st, ws.value


def sfa_run(params: SfaParams, query, query_rope, key, key_rope, value, sparse_indices, block_table,
            actual_seq_lengths_kv, actual_seq_lengths_query, attention_out, softmax_max, softmax_sum, workspace,
            workspace_bytes, device_error_flags, stream) -> int:
    """Pointer arguments are integers (device addresses) or None."""
    return load_library().sfa_run(ctypes.byref(params), query, query_rope, key, key_rope, value, sparse_indices,
                                  block_table, actual_seq_lengths_kv, actual_seq_lengths_query, attention_out,
                                  softmax_max, softmax_sum, workspace, workspace_bytes, device_error_flags, stream)


class SparseFlashAttention:
    """Sparse-index MLA-absorb decode (``sfa_run`` in ``include/ifa.h``).

    Construction validates the static description and allocates the workspace
    with torch; calling the object enqueues ``sfa_run`` on the current (or given)
    torch stream and returns the output tensor, shaped like the query.  ``q_seq_len`` is
    Q_S, the query tokens per batch with ``layout_query`` "BSND" (several for multi-token
    prediction); with "TND", ``q_total`` is Q_T and the query lengths are prefix sums.
    ``sparse_mode`` 3 masks each query token right-down causally.  ``layout_kv`` "PA_BSND"
    takes the paged caches (``block_size``, ``block_num``, ``block_table_cols``); "BSND"
    and "TND" take contiguous key rows, ``kv_rows`` per batch (BSND) or in all (TND).
    With ``return_softmax_lse`` a call also returns softmax_max and softmax_sum (float32,
    one value per query row and head).
    """

    def __init__(self, *, batch: int, num_heads: int, sparse_size: int, block_size: int = 0, block_num: int = 0,
                 block_table_cols: int = 0, dtype: str = "bf16", scale: Optional[float] = None, sparse_mode: int = 0,
                 sparse_block_size: int = 1, q_seq_len: int = 1, layout_query: str = "BSND", q_total: int = 0,
                 layout_kv: str = "PA_BSND", kv_rows: int = 0, return_softmax_lse: bool = False, device=None):
        import torch
        p = SfaParams()
        p.B, p.Q_S, p.Q_T, p.Q_N, p.KV_N, p.D, p.Dr = batch, q_seq_len, q_total, num_heads, 1, 512, 64
        p.KV_S = kv_rows
        p.block_size, p.block_num, p.block_table_cols = block_size, block_num, block_table_cols
        p.sparse_size, p.sparse_block_size = sparse_size, sparse_block_size
        p.layout_query, p.layout_kv = SFA_LAYOUT_QUERY[layout_query], SFA_LAYOUT_KV[layout_kv]
        self.return_softmax_lse = return_softmax_lse
        p.dtype = DTYPES[dtype]
        p.sparse_mode = sparse_mode
        p.scale_value = (1.0 / math.sqrt(576)) if scale is None else float(scale)
        self.params = p
        st, ws = sfa_workspace_size(p)
        if st != IFA_OK:
            raise IfaError(st, "sfa_workspace_size")
        dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.workspace = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)
        self.errors = torch.zeros(1, dtype=torch.int32, device=dev)

    def __call__(self, query, query_rope, key, key_rope, value, sparse_indices, block_table, actual_seq_lengths_kv,
                 *, actual_seq_lengths_query=None, out=None, softmax_max=None, softmax_sum=None, stream=None):
        import torch
        if out is None:
            out = torch.empty_like(query)
        if self.return_softmax_lse:
            lead = query.shape[:-1]
            if softmax_max is None:
                softmax_max = torch.empty(lead, dtype=torch.float32, device=query.device)
            if softmax_sum is None:
                softmax_sum = torch.empty(lead, dtype=torch.float32, device=query.device)
        st = sfa_run(self.params, _ptr(query), _ptr(query_rope), _ptr(key), _ptr(key_rope), _ptr(value),
                     _ptr(sparse_indices), _ptr(block_table), _ptr(actual_seq_lengths_kv),
                     _ptr(actual_seq_lengths_query), _ptr(out), _ptr(softmax_max), _ptr(softmax_sum),
                     _ptr(self.workspace), self.workspace.numel(), _ptr(self.errors), _stream_handle(stream))
        if st != IFA_OK:
            raise IfaError(st, "sfa_run")
        return (out, softmax_max, softmax_sum) if self.return_softmax_lse else out

    def device_errors(self, clear: bool = True) -> int:
        import torch
        torch.cuda.synchronize()
        v = int(self.errors.item())
        if clear:
            self.errors.zero_()
        return v


def kv_append(params: AppendParams, key_new, value_new, positions, block_table, antiquant_scale, antiquant_offset,
              key_cache, value_cache, device_error_flags, stream) -> int:
    """Pointer arguments are integers (device addresses) or None."""
    return load_library().ifa_kv_append(ctypes.byref(params), key_new, value_new, positions, block_table,
                                        antiquant_scale, antiquant_offset, key_cache, value_cache,
                                        device_error_flags, stream)


class KvCacheAppend:
    """KV-cache append (``ifa_kv_append`` in ``include/ifa.h``): writes one new token's key and
    value rows per batch into the caches in place.  ``dtype`` is the new rows' dtype,
    ``kv_dtype`` the cache's ("int8" quantises with ``antiquant`` parameters); ``layout`` and
    ``kv_format`` as for :class:`IncreFlashAttention`."""

    def __init__(self, *, batch: int, num_kv_heads: int, head_dim: int, max_seq_len: int = 0, dtype: str = "bf16",
                 kv_dtype: Optional[str] = None, layout: str = "BNSD", kv_format: str = "contig", block_size: int = 0,
                 block_num: int = 0, block_table_cols: int = 0, antiquant: str = "none", device=None):
        import torch
        p = AppendParams()
        p.B, p.numKeyValueHeads, p.headDim, p.maxSeqLen = batch, num_kv_heads, head_dim, max_seq_len
        p.blockSize, p.blockNum, p.blockTableCols = block_size, block_num, block_table_cols
        p.new_dtype = DTYPES[dtype]
        p.kv_dtype = DTYPES[kv_dtype or dtype]
        p.inputLayout = LAYOUTS[layout]
        p.kvFormat = KV_FORMATS[kv_format]
        p.antiquant = ANTIQUANT[antiquant]
        self.params = p
        dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.errors = torch.zeros(1, dtype=torch.int32, device=dev)

    def __call__(self, key_new, value_new, positions, key_cache, value_cache, *, block_table=None,
                 antiquant_scale=None, antiquant_offset=None, stream=None):
        st = kv_append(self.params, _ptr(key_new), _ptr(value_new), _ptr(positions), _ptr(block_table),
                       _ptr(antiquant_scale), _ptr(antiquant_offset), _ptr(key_cache), _ptr(value_cache),
                       _ptr(self.errors), _stream_handle(stream))
        if st != IFA_OK:
            raise IfaError(st, "ifa_kv_append")
        return key_cache, value_cache

    def device_errors(self, clear: bool = True) -> int:
        import torch
        torch.cuda.synchronize()
        v = int(self.errors.item())
        if clear:
            self.errors.zero_()
        return v
