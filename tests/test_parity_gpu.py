"""GPU parity: the CUDA decode kernels (through the C ABI) against the float64
CPU oracle on the same seeded inputs, element by element.

Tolerances: max abs error <= 2e-3 for fp16 outputs and <= 1.5e-2 for bf16
outputs; int8 key/value paths are compared with the oracle evaluated on the
same dequantised values (the oracle applies (x + offset) * scale itself).
"""
import math

import numpy as np
import pytest

from kv_cache_incremental_split_gb300 import inputs as gen
from harness import TOL, DeviceCase, gpu_ifa, make_op, max_abs_err, oracle_ifa, out_to_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_incremental_split_gb300 import build
    build.build()


def check(case, split_tiles=0, batches=None, tol=None):
    got = gpu_ifa(case, split_tiles)
    ref = oracle_ifa(case, batches)
    if batches is not None:
        got = got[np.asarray(batches)]
    err = max_abs_err(got, ref)
    t = tol if tol is not None else TOL[case.q_dtype]
    assert np.all(np.isfinite(got))
    assert err <= t, f"max abs err {err} > {t}"
    return got, ref


# ---------------------------------------------------------------- the five workloads, small and full

def test_worked_example_all_ones():
    """aclnnIncreFlashAttentionV2 page, Example: all-ones fp16 inputs give all-ones outputs."""
    q = np.ones((1, 2, 1, 16), dtype=np.float16)
    k = np.ones((1, 2, 16, 16), dtype=np.float16)
    case = gen.IfaCase("example", q, k, k.copy(), num_heads=2, num_kv_heads=2, scale=0.25, layout="BNSD",
                       q_dtype="fp16", kv_dtype="fp16", max_seq_len=16,
                       atten_mask=np.zeros((1, 1, 1, 16), dtype=np.int8),
                       actual_seq_lengths=np.array([16], dtype=np.int64))
    got = gpu_ifa(case)
    assert np.array_equal(got, np.ones_like(got))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tiny_mha_full_size(seed):
    check(gen.tiny_mha(seed))


@pytest.mark.parametrize("layout", ["BSH", "BSND", "BNSD"])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_gqa_padded_small(layout, dtype):
    check(gen.gqa_padded(3, B=5, N=32, KV_N=8, D=128, Smax=700, layout=layout, dtype=dtype))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_gqa_padded_full_size(seed):
    check(gen.gqa_padded(seed))


@pytest.mark.parametrize("kv_format", ["paged_nbsd", "paged_bsh"])
@pytest.mark.parametrize("block_size", [128, 16, 48])
def test_paged_small(kv_format, block_size):
    check(gen.paged_gqa(4, B=6, N=32, KV_N=8, D=128, block_size=block_size, len_lo=1, len_hi=1500,
                        kv_format=kv_format))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_paged_full_size_sampled(seed):
    case = gen.paged_gqa(seed)
    rng = np.random.default_rng(100 + seed)
    batches = np.sort(rng.choice(case.B, size=4, replace=False))
    check(case, batches=batches)


@pytest.mark.parametrize("per_tensor", [False, True])
def test_int8_leftpad_small(per_tensor):
    check(gen.int8_leftpad(5, B=6, N=64, KV_N=8, D=128, Smax=600, len_lo=1, len_hi=600, pad_extra=64,
                           per_tensor=per_tensor))


def test_int8_bf16_query():
    check(gen.int8_leftpad(6, B=3, N=16, KV_N=4, D=128, Smax=300, len_lo=1, len_hi=300, q_dtype="bf16"))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_int8_leftpad_full_size_sampled(seed):
    case = gen.int8_leftpad(seed)
    rng = np.random.default_rng(200 + seed)
    check(case, batches=np.sort(rng.choice(case.B, size=4, replace=False)))


# ---------------------------------------------------------------- split plan, determinism

@pytest.mark.parametrize("split_tiles", [1, 2, 3, 7])
def test_forced_splits_match_oracle(split_tiles):
    case = gen.gqa_padded(7, B=4, N=16, KV_N=4, D=128, Smax=1000, layout="BNSD", dtype="bf16")
    check(case, split_tiles=split_tiles)


def test_split_invariance_and_run_to_run_determinism():
    case = gen.paged_gqa(8, B=5, N=32, KV_N=8, D=128, block_size=128, len_lo=100, len_hi=3000)
    dc = DeviceCase(case)
    outs = {}
    for st in (0, 1, 5):
        op = make_op(case, st)
        a = out_to_f64(dc.run(op))
        b = out_to_f64(dc.run(op))
        assert np.array_equal(a, b), "run-to-run results differ"
        outs[st] = a
    assert max_abs_err(outs[0], outs[1]) <= TOL["bf16"]
    assert max_abs_err(outs[0], outs[5]) <= TOL["bf16"]


def test_graph_replays_of_odd_call_counts_with_eager_calls_between():
    """Pieces of a cut sequence meet on a per-sequence arrival counter that all calls of a plan
    share, so every call that completes must leave the counters at zero, whatever mix of graph
    replays and eager calls follows: a graph of three calls (an odd count), replayed three
    times with an eager call after each replay, every sequence cut into pieces."""
    kw = dict(B=4, N=16, KV_N=4, D=128, Smax=1500, layout="BSH", dtype="bf16")
    ca, cb = gen.gqa_padded(31, **kw), gen.gqa_padded(32, **kw)
    da, db = DeviceCase(ca), DeviceCase(cb)
    op = make_op(ca, split_tiles=3)
    refa, refb = oracle_ifa(ca), oracle_ifa(cb)
    outs = [torch.full_like(da.q, float("nan")) for _ in range(3)]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        da.run(op, out=outs[0], stream=s)  # eager first call: the plan's workspace exists before capture
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            da.run(op, out=outs[0], stream=s)
            db.run(op, out=outs[1], stream=s)
            da.run(op, out=outs[2], stream=s)
        for rep in range(3):
            for o in outs:
                o.fill_(float("nan"))
            g.replay()
            eager = db.run(op, stream=s)
            s.synchronize()
            for got, ref in ((outs[0], refa), (outs[1], refb), (outs[2], refa), (eager, refb)):
                got = out_to_f64(got).reshape(ref.shape)
                assert np.all(np.isfinite(got)), rep
                assert max_abs_err(got, ref) <= TOL["bf16"], rep


# ---------------------------------------------------------------- edge cases

def test_head_groupings():
    for N, KV_N in ((8, 8), (16, 1), (32, 1), (12, 4), (48, 2)):
        check(gen.gqa_padded(9, B=2, N=N, KV_N=KV_N, D=64, Smax=300, layout="BNSD", dtype="fp16"))


@pytest.mark.parametrize("D", [16, 80, 256])
def test_head_dims(D):
    check(gen.gqa_padded(10, B=2, N=8, KV_N=2, D=D, Smax=200, layout="BSND", dtype="bf16"))


def test_lengths_zero_one_and_ragged():
    case = gen.gqa_padded(11, B=6, N=8, KV_N=2, D=128, Smax=300, layout="BSH", dtype="fp16", mask=False)
    case.actual_seq_lengths = np.array([0, 1, 63, 64, 65, 300], dtype=np.int64)
    got, _ = check(case)
    assert np.all(got[0] == 0)


def test_all_lengths_zero():
    case = gen.gqa_padded(12, B=3, N=8, KV_N=2, D=64, Smax=50, layout="BNSD", dtype="bf16", mask=False)
    case.actual_seq_lengths = np.zeros(3, dtype=np.int64)
    got = gpu_ifa(case)
    assert np.all(got == 0)


def test_batch_above_inline_limit():
    case = gen.gqa_padded(13, B=300, N=4, KV_N=2, D=64, Smax=80, layout="BNSD", dtype="fp16", mask=False,
                          len_lo=0)
    check(case)


def test_batch_above_inline_limit_is_refused_under_capture():
    """Above 256 batches the per-batch windows reach the device by a pageable host copy, which a
    graph cannot hold: under capture the call is refused without touching the stream, the
    capture stays usable, and an eager call afterwards still matches the oracle."""
    from kv_cache_incremental_split_gb300.ifa import IFA_ERR_PARAM_INVALID, IfaError
    case = gen.gqa_padded(16, B=260, N=4, KV_N=2, D=64, Smax=70, layout="BSH", dtype="bf16", mask=False)
    dc = DeviceCase(case)
    op = make_op(case)
    s = torch.cuda.Stream()
    x = torch.zeros(8, device="cuda")
    with torch.cuda.stream(s):
        dc.run(op, stream=s)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            with pytest.raises(IfaError) as e:
                dc.run(op, stream=s)
            x.add_(1.0)
        g.replay()
        out = dc.run(op, stream=s)
        s.synchronize()
    assert e.value.status == IFA_ERR_PARAM_INVALID
    assert float(x.sum()) == 8.0
    ref = oracle_ifa(case)
    assert max_abs_err(out_to_f64(out).reshape(ref.shape), ref) <= TOL["bf16"]


def test_fully_masked_rows_and_per_head_mask():
    case = gen.gqa_padded(14, B=3, N=8, KV_N=2, D=128, Smax=200, layout="BNSD", dtype="bf16", mask=False)
    m = (np.random.default_rng(1).random((3, 8, 1, 200)) < 0.5)
    m[1, 3] = True  # batch 1, head 3: nothing survives
    case.atten_mask = m
    got, _ = check(case)
    assert np.all(got[1, 3] == 0)


def test_broadcast_mask_1N1S():
    case = gen.gqa_padded(15, B=3, N=8, KV_N=2, D=64, Smax=150, layout="BSH", dtype="fp16", mask=False)
    case.atten_mask = (np.random.default_rng(2).random((1, 8, 1, 150)) < 0.3).astype(np.uint8)
    check(case)


def test_padding_sizes_without_lengths_leave_the_cache_right_padded():
    """Without actualSeqLengths every batch uses its whole cache and kvPaddingSize has nothing to
    place: the call equals the one without padding sizes bit for bit, and the oracle."""
    case = gen.gqa_padded(24, B=3, N=8, KV_N=2, D=128, Smax=700, layout="BSND", dtype="bf16", mask=False)
    case.actual_seq_lengths = None
    plain = gpu_ifa(case)
    case.kv_padding_size = np.array([5, 300, 0], dtype=np.int64)
    padded = gpu_ifa(case)
    assert np.array_equal(plain, padded)
    assert max_abs_err(padded, oracle_ifa(case)) <= TOL["bf16"]


def test_left_pad_edge_windows():
    case = gen.int8_leftpad(16, B=4, N=8, KV_N=2, D=128, Smax=256, len_lo=1, len_hi=256)
    case.actual_seq_lengths = np.array([200, 10, 256, 100], dtype=np.int64)
    case.kv_padding_size = np.array([100, -7, 0, 156], dtype=np.int64)  # b0 out of range -> zeros
    got, _ = check(case)
    assert np.all(got[0] == 0)


def test_nan_beyond_the_window_does_not_leak():
    case = gen.gqa_padded(17, B=2, N=8, KV_N=2, D=128, Smax=256, layout="BNSD", dtype="fp16", mask=False)
    case.actual_seq_lengths = np.array([70, 129], dtype=np.int64)
    for b, L in enumerate(case.actual_seq_lengths):
        case.key[b, :, L:] = np.float16(np.nan)
        case.value[b, :, L:] = np.float16(np.nan)
    check(case)


def test_bad_block_table_entry_sets_error_flag():
    case = gen.paged_gqa(18, B=2, N=8, KV_N=2, D=64, block_size=64, len_lo=300, len_hi=400, dtype="bf16")
    case.block_table = case.block_table.copy()
    case.block_table[1, 2] = case.key.shape[0] + 5  # out of range: those tokens are left out
    dc = DeviceCase(case)
    op = make_op(case)
    out = out_to_f64(dc.run(op)).reshape(2, 8, 64)
    torch.cuda.synchronize()
    assert op.device_errors() & 1
    ref = oracle_ifa(case)  # the oracle leaves the same tokens out
    assert max_abs_err(out, ref) <= TOL["bf16"]
    assert op.device_errors() == 0  # cleared by the previous read


@pytest.mark.parametrize("left_pad", [False, True])
def test_mask_staged_by_the_producer(left_pad):
    """Per-batch masks whose row length is a multiple of 16 bytes are staged per tile by
    TMA; windows then start anywhere (left padding), not only on 16-byte boundaries."""
    rng = np.random.default_rng(31)
    case = gen.gqa_padded(31, B=5, N=16, KV_N=4, D=128, Smax=640, layout="BNSD", dtype="fp16", mask=False)
    case.atten_mask = rng.random((5, 1, 1, 640)) < 0.3
    if left_pad:
        case.actual_seq_lengths = np.array([100, 333, 640, 17, 500], dtype=np.int64)
        case.kv_padding_size = np.array([3, 300, 0, 611, 77], dtype=np.int64)
    check(case)
    case.atten_mask = case.atten_mask[:1]  # (1,1,1,S): one row for every batch
    check(case)


# ---- int8 key/value with two 16-token mma tiles per consumer warp (256-token tiles)


@pytest.mark.parametrize("block_size,kv_format", [(32, "paged_nbsd"), (96, "paged_nbsd"), (256, "paged_bsh")])
def test_int8_paged(block_size, kv_format):
    """Paged int8 caches: a 256-token tile spans 8, 8 or 1 cache blocks (box rows gcd(256, block))."""
    check(gen.int8_paged(41, B=5, N=16, KV_N=4, D=128, block_size=block_size, len_lo=1, len_hi=900,
                         kv_format=kv_format))


@pytest.mark.parametrize("left_pad", [False, True])
def test_int8_mask_staged_in_two_boxes(left_pad):
    """A 256-token tile's mask bytes come in two TMA boxes; windows start anywhere."""
    rng = np.random.default_rng(42)
    case = gen.int8_leftpad(42, B=5, N=16, KV_N=4, D=128, Smax=640, len_lo=1, len_hi=640)
    if not left_pad:
        case.kv_padding_size = None
    case.atten_mask = rng.random((5, 1, 1, 640)) < 0.3
    check(case)


def test_int8_per_head_mask():
    """Per-head masks are read by the consumer warps, one tile ahead, for both 16-token tiles."""
    rng = np.random.default_rng(43)
    case = gen.int8_leftpad(43, B=3, N=16, KV_N=4, D=128, Smax=600, len_lo=1, len_hi=600)
    case.atten_mask = rng.random((3, 16, 1, 600)) < 0.4
    check(case)


@pytest.mark.parametrize("split_tiles", [1, 2, 3])
def test_int8_forced_splits(split_tiles):
    check(gen.int8_leftpad(44, B=4, N=32, KV_N=4, D=128, Smax=2000, len_lo=300, len_hi=2000), split_tiles=split_tiles)
