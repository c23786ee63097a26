"""GPU parity of the int8 output quantisation fused into the decode kernel's epilogue
(quantScale2 / quantOffset2) against the CPU oracle: the oracle quantises its float64
attention output with the same single-precision steps.  The two outputs differ within
the attention tolerance, so a code may differ by one where y * scale2 + offset2 falls
within that tolerance (times the scale) of a rounding boundary; everywhere else the
codes must be equal."""
import numpy as np
import pytest

import oracle
from kv_cache_incremental_split_gb300 import inputs as gen
from harness import TOL, DeviceCase, make_op, oracle_ifa, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_incremental_split_gb300 import build
    build.build()


def params(rng, case, per_channel, pdtype, with_offset=True, scale_range=(5.0, 60.0)):
    n = case.num_heads * case.D if per_channel else 1
    s = rng.uniform(*scale_range, n).astype(np.float32)
    o = rng.uniform(-6, 6, n).astype(np.float32) if with_offset else None
    if pdtype == "bf16":
        s = gen.to_storage(s, "bf16")
        o = None if o is None else gen.to_storage(o, "bf16")
    return s, o


def as_f32(a):
    return a if a is None or a.dtype == np.float32 else (a.astype(np.uint32) << 16).view(np.float32)


def check_codes(case, per_channel, pdtype, seed=0, split_tiles=0, **kw):
    rng = np.random.default_rng(seed)
    s, o = params(rng, case, per_channel, pdtype, **kw)
    op = make_op(case, split_tiles, out_dtype="int8", quant2="per_channel" if per_channel else "per_tensor",
                 quant2_dtype="fp32" if pdtype == "fp32" else "bf16")
    out = DeviceCase(case).run(op, quant_scale2=to_device(s), quant_offset2=to_device(o))
    torch.cuda.synchronize()
    assert out.dtype == torch.int8
    got = out.cpu().numpy().reshape(case.B, case.num_heads, case.D).astype(np.int64)
    y = oracle_ifa(case)
    ref = oracle.quantize_output_ref(y, s, o).astype(np.int64)
    diff = np.abs(got - ref)
    assert diff.max() <= 1
    # exact away from rounding boundaries: |u - (k + 1/2)| > tol * |scale| for the oracle's u
    sf = as_f32(s).astype(np.float64).reshape(-1)
    of = np.zeros_like(sf) if o is None else as_f32(o).astype(np.float64).reshape(-1)
    if not per_channel:
        sf, of = np.full(case.num_heads * case.D, sf[0]), np.full(case.num_heads * case.D, of[0])
    u = y * sf.reshape(case.num_heads, case.D) + of.reshape(case.num_heads, case.D)
    margin = 2 * TOL[case.q_dtype] * np.abs(sf.reshape(case.num_heads, case.D)) + 1e-6
    near = np.abs(u - np.floor(u) - 0.5) <= margin
    inside = (u > -128.5 - margin) & (u < 127.5 + margin)
    assert np.all(diff[~near | ~inside] == 0)
    return got, ref


@pytest.mark.parametrize("per_channel,pdtype", [(True, "fp32"), (True, "bf16"), (False, "fp32"), (False, "bf16")])
def test_int8_output_gqa_padded_bf16(per_channel, pdtype):
    check_codes(gen.gqa_padded(80, B=4, Smax=1000), per_channel, pdtype)


def test_int8_output_fp16_query_per_tensor_and_no_offset():
    check_codes(gen.tiny_mha(81), False, "fp32", with_offset=False)
    check_codes(gen.gqa_padded(82, B=3, Smax=700, dtype="fp16", layout="BNSD"), True, "fp32", seed=1)


def test_int8_output_paged_and_split_pieces():
    # cut sequences: the merge of the last arriving piece writes the codes
    c = gen.paged_gqa(83, B=4, len_lo=300, len_hi=3000)
    check_codes(c, True, "fp32", seed=2)
    check_codes(c, True, "bf16", seed=3, split_tiles=3)


def test_int8_output_with_int8_cache_and_left_padding():
    c = gen.int8_leftpad(84, B=4, Smax=1024, len_lo=50, len_hi=1000)
    check_codes(c, True, "fp32", seed=4, scale_range=(20.0, 100.0))


def test_int8_output_empty_rows_quantise_zero():
    # zero-length batches give y = 0, so their codes are rint(offset2)
    c = gen.gqa_padded(85, B=3, Smax=500, mask=False)
    c.actual_seq_lengths = np.array([0, 200, 0], dtype=np.int64)
    got, ref = check_codes(c, True, "fp32", seed=5)
    assert np.array_equal(got[0], ref[0]) and np.array_equal(got[2], ref[2])
