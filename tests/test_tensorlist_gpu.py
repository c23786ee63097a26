"""GPU parity of the decode kernel with key/value given as one tensor per batch
(ifa_run_tensorlist: per-batch TMA descriptors in device memory) against the CPU oracle on
the same seeded inputs; tolerances as for the contiguous cache."""
import numpy as np
import pytest

import oracle
from kv_cache_incremental_split_gb300 import inputs as gen
from harness import TOL, make_op, max_abs_err, out_to_f64, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

AQ = {"none": oracle.AQ_NONE, "per_channel": oracle.AQ_PER_CHANNEL, "per_tensor": oracle.AQ_PER_TENSOR}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_incremental_split_gb300 import build
    build.build()


def ref_of(c):
    return oracle.ifa_ref_tensorlist(c.query, c.key, c.value, num_heads=c.num_heads, num_kv_heads=c.num_kv_heads,
                                     scale=c.scale, layout=c.layout, atten_mask=c.atten_mask,
                                     actual_seq_lengths=c.actual_seq_lengths, antiquant=AQ[c.antiquant],
                                     antiquant_scale=c.antiquant_scale, antiquant_offset=c.antiquant_offset)


def run(c, op=None, keys=None, values=None, lens="case"):
    op = op or make_op(c)
    keys = keys if keys is not None else [to_device(k) for k in c.key]
    values = values if values is not None else [to_device(v) for v in c.value]
    out = op(to_device(c.query), keys, values, atten_mask=to_device(c.atten_mask),
             actual_seq_lengths=c.actual_seq_lengths if lens == "case" else lens,
             antiquant_scale=to_device(c.antiquant_scale), antiquant_offset=to_device(c.antiquant_offset))
    torch.cuda.synchronize()
    assert op.device_errors() == 0
    return out_to_f64(out).reshape(c.B, c.num_heads, c.D), op


@pytest.mark.parametrize("layout", ["BSH", "BSND", "BNSD"])
def test_tensorlist_gqa_bf16_with_mask(layout):
    c = gen.tensorlist_from(gen.gqa_padded(100, B=6, Smax=3000, layout=layout), seed=3, extra_hi=200)
    got, _ = run(c)
    assert max_abs_err(got, ref_of(c)) <= TOL["bf16"]


def test_tensorlist_fp16_mha_whole_tensors():
    # no lengths: every batch attends over its whole tensor (S_b differ)
    base = gen.gqa_padded(101, B=5, N=8, KV_N=8, D=64, Smax=2000, layout="BNSD", dtype="fp16", mask=False)
    c = gen.tensorlist_from(base, seed=4, extra_hi=0)
    c.actual_seq_lengths = None
    got, _ = run(c, lens=None)
    assert max_abs_err(got, ref_of(c)) <= TOL["fp16"]


def test_tensorlist_int8_antiquant():
    base = gen.int8_leftpad(102, B=4, Smax=2048, len_lo=100, len_hi=2000)
    base.kv_padding_size = None  # right padding: the list has no left padding
    c = gen.tensorlist_from(base, seed=5, extra_hi=64)
    got, _ = run(c)
    assert max_abs_err(got, ref_of(c)) <= TOL["fp16"]


def test_tensorlist_max_batch_and_split_pieces():
    base = gen.gqa_padded(103, B=256, N=8, KV_N=2, D=128, Smax=700, layout="BSND", mask=False)
    c = gen.tensorlist_from(base, seed=6, extra_hi=30)
    got, _ = run(c)
    assert max_abs_err(got, ref_of(c)) <= TOL["bf16"]


def test_tensorlist_new_pointers_between_calls():
    # the second call moves one batch's tensors and changes one extent: the maps are re-encoded
    c = gen.tensorlist_from(gen.gqa_padded(104, B=3, Smax=1500), seed=7, extra_hi=100)
    got, op = run(c)
    assert max_abs_err(got, ref_of(c)) <= TOL["bf16"]
    keys = [to_device(k) for k in c.key]
    values = [to_device(v) for v in c.value]
    got2, _ = run(c, op=op, keys=keys, values=values)  # same contents, new addresses
    assert max_abs_err(got2, ref_of(c)) <= TOL["bf16"]
    got3, _ = run(c, op=op, keys=keys, values=values)  # unchanged lists: cached maps
    assert np.array_equal(got3, got2)
    c.key[1] = c.key[1][:, : int(c.actual_seq_lengths[1])].copy()  # a shorter tensor (BSH: S on axis 1)
    c.value[1] = c.value[1][:, : int(c.actual_seq_lengths[1])].copy()
    got4, _ = run(c, op=op)
    assert max_abs_err(got4, ref_of(c)) <= TOL["bf16"]


def test_tensorlist_graph_capture_needs_the_previous_lists():
    """A captured call replays with the descriptors encoded before the capture; new lists under
    capture are refused without touching the stream, so the capture stays usable."""
    from kv_cache_incremental_split_gb300.ifa import IfaError
    c = gen.tensorlist_from(gen.gqa_padded(105, B=4, Smax=1200), seed=8, extra_hi=50)
    op = make_op(c)
    keys = [to_device(k) for k in c.key]
    values = [to_device(v) for v in c.value]
    q, mask = to_device(c.query), to_device(c.atten_mask)
    out = torch.empty_like(q)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        op(q, keys, values, atten_mask=mask, actual_seq_lengths=c.actual_seq_lengths, out=out, stream=stream)
        stream.synchronize()
        moved = [k.clone() for k in keys]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            with pytest.raises(IfaError):
                op(q, moved, values, atten_mask=mask, actual_seq_lengths=c.actual_seq_lengths, out=out,
                   stream=stream)
            op(q, keys, values, atten_mask=mask, actual_seq_lengths=c.actual_seq_lengths, out=out, stream=stream)
        out.zero_()
        g.replay()
        stream.synchronize()
    assert op.device_errors() == 0
    got = out_to_f64(out).reshape(c.B, c.num_heads, c.D)
    assert max_abs_err(got, ref_of(c)) <= TOL["bf16"]
