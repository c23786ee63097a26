"""ifa_run_noalloc: the allocation-free entry point for callers that cannot
allocate device memory (code inside a memory pool or allocator it does not
own, runtimes that forbid allocation on the request path).  It must give the
results of the regular plan + workspace path, call after call, although every
call reuses one fixed scratch array that still holds the previous call's
partials.

This file is named to be collected last, so that a run stopping at the first
failure has already run every other test.
"""
import numpy as np
import pytest

from kv_cache_incremental_split_gb300 import ifa
from kv_cache_incremental_split_gb300 import inputs as gen
from harness import TOL, DeviceCase, make_op, max_abs_err, out_to_f64


def _ptr(t):
    return None if t is None else int(t.data_ptr())


def _noalloc_call(op, dc, out, err, stream):
    c = dc.case
    lens = np.ascontiguousarray(c.actual_seq_lengths, dtype=np.int64)
    pads = None if c.kv_padding_size is None else np.ascontiguousarray(c.kv_padding_size, np.int64).reshape(-1)
    return ifa.ifa_run_noalloc(op.params, _ptr(dc.q), _ptr(dc.k), _ptr(dc.v), _ptr(dc.mask), lens.ctypes.data,
                               None if pads is None else pads.ctypes.data, 0 if pads is None else pads.size,
                               _ptr(dc.bt), _ptr(dc.sc), _ptr(dc.of), _ptr(out), _ptr(err), stream)


@pytest.mark.gpu
def test_noalloc_matches_regular_path_on_consecutive_calls():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_incremental_split_gb300 import build
    build.build()
    cases = [
        (gen.gqa_padded(21, B=4, N=32, KV_N=8, D=128, Smax=2000, layout="BSH", dtype="bf16"), 3),
        (gen.int8_leftpad(22, B=5, N=16, KV_N=4, D=128, Smax=900, len_lo=1, len_hi=900), 2),
        (gen.paged_gqa(23, B=3, N=8, KV_N=2, D=64, block_size=32, len_lo=100, len_hi=700, dtype="bf16"), 0),
    ]
    stream = torch.cuda.current_stream().cuda_stream
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for rep in range(2):  # two rounds of calls in a row on the same scratch
        for case, split in cases:
            dc = DeviceCase(case)
            op = make_op(case, split)
            ref = out_to_f64(dc.run(op))
            out = torch.full_like(dc.q, float("nan"))
            st = _noalloc_call(op, dc, out, err, stream)
            assert st == ifa.IFA_OK, ifa.status_string(st)
            torch.cuda.synchronize()
            got = out_to_f64(out)
            assert np.all(np.isfinite(got))
            assert max_abs_err(got, ref) <= TOL[case.q_dtype], (case.name, rep)
    assert int(err.item()) == 0


def test_noalloc_rejects_batches_beyond_its_limit():
    ifa.load_library()
    p = ifa.IfaParams()
    p.B, p.numHeads, p.numKeyValueHeads, p.headDim, p.maxSeqLen = ifa.IFA_NOALLOC_MAX_BATCH + 1, 8, 2, 128, 64
    p.q_dtype = p.kv_dtype = ifa.DTYPES["bf16"]
    p.inputLayout = ifa.LAYOUTS["BSH"]
    p.scaleValue = 0.1
    dummy = 1 << 20  # never dereferenced: the size check comes first
    st = ifa.ifa_run_noalloc(p, dummy, dummy, dummy, None, None, None, 0, None, None, None, dummy, None, None)
    assert st == ifa.IFA_ERR_PARAM_INVALID
