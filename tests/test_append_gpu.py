"""GPU parity of the KV-cache append kernel (ifa_kv_append) against the CPU oracle on
the same seeded inputs: every byte of both caches after the append is compared
(bit-exact: the 16-bit path copies, the int8 path takes the same single-precision
rounding decisions as the oracle), and an attention call over the appended cache
matches the oracle within the attention tolerances."""
import numpy as np
import pytest

import oracle
from kv_cache_incremental_split_gb300 import inputs as gen
from harness import TOL, max_abs_err, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

FMT = {"contig": oracle.CONTIG, "paged_nbsd": oracle.PAGED_NBSD, "paged_bsh": oracle.PAGED_BSH}
AQ = {"none": oracle.AQ_NONE, "per_channel": oracle.AQ_PER_CHANNEL, "per_tensor": oracle.AQ_PER_TENSOR}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_incremental_split_gb300 import build
    build.build()


def storage(rng, shape, dtype):
    x = rng.standard_normal(shape).astype(np.float32) * 1.5
    return gen.to_storage(x, dtype)


def make(seed, B, KVN, D, dtype, kv_dtype, layout, kv_format, S=64, bs=16, antiquant="none"):
    rng = np.random.default_rng(seed)
    kn, vn = storage(rng, (B, KVN, D), dtype), storage(rng, (B, KVN, D), dtype)
    bt = None
    if kv_format == "contig":
        shape = {"BNSD": (B, KVN, S, D), "BSND": (B, S, KVN, D), "BSH": (B, S, KVN * D)}[layout]
    else:
        cols = S // bs
        bt = rng.permutation(B * cols).astype(np.int32).reshape(B, cols)
        shape = (B * cols, KVN, bs, D) if kv_format == "paged_nbsd" else (B * cols, bs, KVN * D)
    if kv_dtype == "int8":
        kc = rng.integers(-127, 128, shape, dtype=np.int8)
        vc = rng.integers(-127, 128, shape, dtype=np.int8)
    else:
        kc, vc = storage(rng, shape, dtype), storage(rng, shape, dtype)
    sc = of = None
    if antiquant != "none":
        pshape = (2, KVN, D) if antiquant == "per_channel" else (2,)
        sc = gen.to_storage(rng.uniform(0.005, 0.03, pshape).astype(np.float32), dtype)
        of = gen.to_storage(rng.uniform(-4, 4, pshape).astype(np.float32), dtype)
    pos = rng.integers(0, S, B).astype(np.int64)
    return kn, vn, pos, kc, vc, bt, sc, of


def run_both(B, KVN, D, dtype, kv_dtype, layout, kv_format, pos=None, S=64, bs=16, antiquant="none", seed=0):
    from kv_cache_incremental_split_gb300.ifa import KvCacheAppend
    kn, vn, p0, kc, vc, bt, sc, of = make(seed, B, KVN, D, dtype, kv_dtype, layout, kv_format, S, bs, antiquant)
    pos = p0 if pos is None else np.asarray(pos, dtype=np.int64)
    rk, rv, skipped = oracle.kv_append_ref(kn, vn, pos, kc, vc, layout=layout, kv_format=FMT[kv_format],
                                           block_size=bs, block_table=bt, antiquant=AQ[antiquant],
                                           antiquant_scale=sc, antiquant_offset=of)
    op = KvCacheAppend(batch=B, num_kv_heads=KVN, head_dim=D, max_seq_len=S, dtype=dtype, kv_dtype=kv_dtype,
                       layout=layout, kv_format=kv_format, block_size=bs,
                       block_num=kc.shape[0] if kv_format != "contig" else 0,
                       block_table_cols=bt.shape[1] if bt is not None else 0, antiquant=antiquant)
    dk, dv = to_device(kc), to_device(vc)
    op(to_device(kn), to_device(vn), to_device(pos), dk, dv, block_table=to_device(bt),
       antiquant_scale=to_device(sc), antiquant_offset=to_device(of))
    err = op.device_errors()
    gk = dk.cpu().view(torch.int16 if dk.element_size() == 2 else torch.int8).numpy()
    gv = dv.cpu().view(torch.int16 if dv.element_size() == 2 else torch.int8).numpy()
    view = np.int16 if rk.dtype.itemsize == 2 else np.int8
    return gk, gv, rk.view(view), rv.view(view), skipped, err


@pytest.mark.parametrize("layout,kv_format", [("BNSD", "contig"), ("BSND", "contig"), ("BSH", "contig"),
                                              ("BNSD", "paged_nbsd"), ("BSH", "paged_bsh")])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_append_16bit_bit_exact(layout, kv_format, dtype):
    gk, gv, rk, rv, skipped, err = run_both(5, 4, 128, dtype, dtype, layout, kv_format)
    assert skipped == 0 and err == 0
    assert np.array_equal(gk, rk) and np.array_equal(gv, rv)


@pytest.mark.parametrize("antiquant", ["per_channel", "per_tensor"])
@pytest.mark.parametrize("layout,kv_format", [("BNSD", "contig"), ("BSND", "contig"), ("BNSD", "paged_nbsd"),
                                              ("BSH", "paged_bsh")])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_append_int8_codes_bit_exact(antiquant, layout, kv_format, dtype):
    gk, gv, rk, rv, skipped, err = run_both(6, 8, 128, dtype, "int8", layout, kv_format, antiquant=antiquant, seed=1)
    assert skipped == 0 and err == 0
    assert np.array_equal(gk, rk) and np.array_equal(gv, rv)


def test_append_head_dims_and_saturating_values():
    # D = 64 and 256, values far outside the code range saturate identically on both sides
    for D in (64, 256):
        gk, gv, rk, rv, _, _ = run_both(3, 2, D, "fp16", "int8", "BNSD", "paged_nbsd", antiquant="per_channel",
                                        seed=D)
        assert np.array_equal(gk, rk) and np.array_equal(gv, rv)
    gk, gv, rk, rv, _, _ = run_both(3, 2, 16, "bf16", "bf16", "BSND", "contig", seed=9)
    assert np.array_equal(gk, rk) and np.array_equal(gv, rv)


def test_append_positions_outside_the_cache_write_nothing_and_flag():
    gk, gv, rk, rv, skipped, err = run_both(4, 2, 64, "bf16", "bf16", "BNSD", "contig", pos=[-1, 64, 10, 63])
    assert skipped == 2 and err == 1
    assert np.array_equal(gk, rk) and np.array_equal(gv, rv)
    gk, gv, rk, rv, skipped, err = run_both(3, 2, 64, "bf16", "bf16", "BNSD", "paged_nbsd", pos=[64, 3, 200])
    assert skipped == 2 and err == 1
    assert np.array_equal(gk, rk) and np.array_equal(gv, rv)


def test_append_then_attend_matches_the_oracle():
    """The incremental step: append the new token at each length, then attend over length + 1."""
    from harness import DeviceCase, make_op, oracle_ifa, out_to_f64
    from kv_cache_incremental_split_gb300.ifa import KvCacheAppend
    c = gen.paged_gqa(70, B=8, N=32, KV_N=8, D=128, block_size=128, len_lo=100, len_hi=1500)
    rng = np.random.default_rng(70)
    lens = c.actual_seq_lengths.astype(np.int64)
    cols = c.block_table.shape[1]
    # every batch needs room for one more token
    assert ((lens + 127) // 128 <= cols).all()
    kn, vn = storage(rng, (8, 8, 128), "bf16"), storage(rng, (8, 8, 128), "bf16")
    # blocks for the new token where the length is a multiple of the block size
    need = (lens // 128)
    spare = c.key.shape[0]
    extra = 0
    bt = c.block_table.copy()
    for b in range(8):
        if bt[b, need[b]] < 0:
            bt[b, need[b]] = spare + extra
            extra += 1
    if extra:
        pad = np.zeros((extra,) + c.key.shape[1:], dtype=c.key.dtype)
        c.key = np.concatenate([c.key, pad])
        c.value = np.concatenate([c.value, pad])
    c.block_table = bt
    rk, rv, skipped = oracle.kv_append_ref(kn, vn, lens, c.key, c.value, kv_format=oracle.PAGED_NBSD,
                                           block_size=128, block_table=bt)
    assert skipped == 0
    op = KvCacheAppend(batch=8, num_kv_heads=8, head_dim=128, dtype="bf16", kv_format="paged_nbsd",
                       block_size=128, block_num=c.key.shape[0], block_table_cols=cols)
    dk, dv = to_device(c.key), to_device(c.value)
    op(to_device(kn), to_device(vn), to_device(lens), dk, dv, block_table=to_device(bt))
    assert op.device_errors() == 0
    assert np.array_equal(dk.cpu().view(torch.int16).numpy(), rk.view(np.int16))
    c.key, c.value = rk, rv
    c.actual_seq_lengths = lens + 1
    dc = DeviceCase(c)
    dc.k, dc.v = dk, dv  # attend over the caches the kernel appended to
    out = dc.run(make_op(c))
    torch.cuda.synchronize()
    got = out_to_f64(out).reshape(c.B, c.num_heads, c.D)
    assert max_abs_err(got, oracle_ifa(c)) <= TOL["bf16"]
