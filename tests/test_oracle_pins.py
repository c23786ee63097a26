"""Pins of the CPU oracle to facts the pages and the mathematics fix.

Each test checks the oracle against something other than itself: the worked
example of the aclnnIncreFlashAttentionV2 page, closed forms of softmax
attention, invariants the IncreFlashAttention / SparseFlashAttention pages
state (GQA head sharing, page-attention addressing, left padding, masking,
sparse selection), and torch's float64 softmax on small shapes.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from kv_cache_incremental_split_gb300 import inputs as gen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def as_f64(a, dtype):
    if dtype == "fp16":
        return np.asarray(a, dtype=np.float16).astype(np.float64)
    if dtype == "bf16":
        return gen.bf16_bits_to_f32(a).astype(np.float64)
    return np.asarray(a).astype(np.float64)


def torch_attention(q, k, v, scale, valid=None):
    """float64 softmax(q k^T * scale) v for one head; q (D,), k/v (T, D)."""
    q = torch.as_tensor(q, dtype=torch.float64)
    k = torch.as_tensor(k, dtype=torch.float64)
    v = torch.as_tensor(v, dtype=torch.float64)
    if valid is not None:
        sel = torch.as_tensor(np.nonzero(valid)[0])
        k, v = k[sel], v[sel]
    if k.shape[0] == 0:
        return np.zeros(v.shape[1])
    p = torch.softmax((k @ q) * scale, dim=0)
    return (p @ v).numpy()


def run(case, **over):
    kw = dict(num_heads=case.num_heads, num_kv_heads=case.num_kv_heads, scale=case.scale,
              layout=case.layout, atten_mask=case.atten_mask,
              actual_seq_lengths=case.actual_seq_lengths, kv_padding_size=case.kv_padding_size)
    kw.update(over)
    return oracle.ifa_ref(case.query, case.key, case.value, **kw)


# ---------------------------------------------------------------- worked example

def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            vals[key] = rest
    return vals


def test_worked_example_of_the_v2_page():
    g = _read_golden("aclnn_ifa_v2_example.txt")
    B, N, KV_N, D, S = (int(g[k][0]) for k in ("B", "N", "KV_N", "D", "S"))
    fill = float(g["fill"][0])
    q = np.full((B, N, 1, D), fill, dtype=np.float16)
    k = np.full((B, KV_N, S, D), fill, dtype=np.float16)
    v = np.full((B, KV_N, S, D), fill, dtype=np.float16)
    mask = np.full([int(x) for x in g["mask_shape"]], int(g["mask_fill"][0]), dtype=np.int8)
    lens = np.array([int(x) for x in g["actual_seq_lengths"]], dtype=np.int64)
    out = oracle.ifa_ref(q, k, v, num_heads=N, num_kv_heads=KV_N, scale=float(g["scale"][0]),
                         layout=g["layout"][0], atten_mask=mask, actual_seq_lengths=lens)
    expected = np.array([float(x) for x in g["expected"]])
    assert out.size == expected.size == 32
    assert np.array_equal(out.reshape(-1), expected)


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_matches_torch_float64_softmax(dtype):
    """Small GQA problems against torch's float64 softmax on the same widened values."""
    for seed in range(3):
        case = gen.gqa_padded(seed, B=3, N=6, KV_N=2, D=16, Smax=37, layout="BNSD", dtype=dtype,
                              mask=False, len_lo=1)
        out = run(case)
        q = as_f64(case.query, dtype).reshape(3, 6, 16)
        k = as_f64(case.key, dtype)
        v = as_f64(case.value, dtype)
        for b in range(3):
            L = int(case.actual_seq_lengths[b])
            for n in range(6):
                h = n // 3
                ref = torch_attention(q[b, n], k[b, h, :L], v[b, h, :L], case.scale)
                np.testing.assert_allclose(out[b, n], ref, rtol=1e-12, atol=1e-13)


def test_constant_value_rows_give_that_constant():
    case = gen.gqa_padded(4, B=2, N=4, KV_N=2, D=32, Smax=50, layout="BNSD", dtype="fp16", mask=False)
    case.value = np.full_like(case.value, np.float16(0.375))
    out = run(case)
    np.testing.assert_allclose(out, 0.375, rtol=1e-14, atol=0)


def test_identical_keys_give_mean_of_values():
    case = gen.gqa_padded(5, B=2, N=4, KV_N=2, D=16, Smax=40, layout="BNSD", dtype="fp16", mask=False)
    case.key = np.broadcast_to(case.key[:, :, :1, :], case.key.shape).copy()
    out = run(case)
    v = as_f64(case.value, "fp16")
    for b in range(2):
        L = int(case.actual_seq_lengths[b])
        for n in range(4):
            np.testing.assert_allclose(out[b, n], v[b, n // 2, :L].mean(axis=0), rtol=1e-12, atol=1e-14)


def test_zero_query_gives_mean_of_values():
    case = gen.gqa_padded(6, B=2, N=2, KV_N=1, D=16, Smax=33, layout="BSND", dtype="bf16", mask=False)
    case.query = np.zeros_like(case.query)
    out = run(case)
    v = as_f64(case.value, "bf16")  # (B, S, KV_N, D)
    for b in range(2):
        L = int(case.actual_seq_lengths[b])
        for n in range(2):
            np.testing.assert_allclose(out[b, n], v[b, :L, 0].mean(axis=0), rtol=1e-12, atol=1e-14)


def test_single_valid_token_returns_its_value_row():
    case = gen.gqa_padded(7, B=3, N=4, KV_N=2, D=16, Smax=20, layout="BNSD", dtype="bf16", mask=False)
    case.actual_seq_lengths = np.array([1, 1, 1], dtype=np.int64)
    out = run(case)
    v = as_f64(case.value, "bf16")
    for b in range(3):
        for n in range(4):
            assert np.array_equal(out[b, n], v[b, n // 2, 0])
    # the same through the mask: only position 5 survives
    case.actual_seq_lengths = np.array([20, 20, 20], dtype=np.int64)
    m = np.ones((3, 1, 1, 20), dtype=bool)
    m[:, :, :, 5] = False
    out = run(case, atten_mask=m)
    for b in range(3):
        for n in range(4):
            assert np.array_equal(out[b, n], v[b, n // 2, 5])


# ---------------------------------------------------------------- invariants on the pages

def test_gqa_equals_explicitly_repeated_kv_heads():
    """numHeads a multiple of numKeyValueHeads (IncreFlashAttention README constraints)."""
    case = gen.gqa_padded(8, B=2, N=8, KV_N=2, D=16, Smax=30, layout="BNSD", dtype="fp16", mask=False)
    out_gqa = run(case)
    G = 4
    rep_k = np.repeat(case.key, G, axis=1)   # head n <- kv head n // G
    rep_v = np.repeat(case.value, G, axis=1)
    out_mha = oracle.ifa_ref(case.query, rep_k, rep_v, num_heads=8, num_kv_heads=8,
                             scale=case.scale, layout="BNSD",
                             actual_seq_lengths=case.actual_seq_lengths)
    assert np.array_equal(out_gqa, out_mha)


def test_num_kv_heads_zero_means_equal_to_num_heads():
    case = gen.gqa_padded(9, B=2, N=3, KV_N=3, D=16, Smax=12, layout="BNSD", dtype="fp16", mask=False)
    assert np.array_equal(run(case, num_kv_heads=0), run(case, num_kv_heads=3))


@pytest.mark.parametrize("layout", ["BSH", "BSND"])
def test_layouts_describe_the_same_problem(layout):
    ref = gen.gqa_padded(10, B=2, N=4, KV_N=2, D=16, Smax=21, layout="BNSD", dtype="bf16", mask=False)
    q = ref.query.reshape(2, 4, 16)
    k = np.transpose(ref.key, (0, 2, 1, 3))   # (B, S, KV_N, D)
    v = np.transpose(ref.value, (0, 2, 1, 3))
    if layout == "BSH":
        q2, k2, v2 = q.reshape(2, 1, 64), k.reshape(2, 21, 32), v.reshape(2, 21, 32)
    else:
        q2, k2, v2 = q.reshape(2, 1, 4, 16), k, v
    out = oracle.ifa_ref(q2, k2, v2, num_heads=4, num_kv_heads=2, scale=ref.scale, layout=layout,
                         actual_seq_lengths=ref.actual_seq_lengths)
    assert np.array_equal(out, run(ref))


@pytest.mark.parametrize("block_size", [16, 48, 5])
def test_paged_equals_contiguous(block_size):
    """Token t of batch b lives in block blockTable[b][t // blockSize], slot t % blockSize."""
    rng = np.random.default_rng(11)
    case = gen.gqa_padded(11, B=3, N=4, KV_N=2, D=16, Smax=100, layout="BNSD", dtype="bf16", mask=False)
    lens = case.actual_seq_lengths
    nblk = [(int(l) + block_size - 1) // block_size for l in lens]
    total = sum(nblk) + 3  # a few unused physical blocks
    perm = rng.permutation(total)
    cols = (100 + block_size - 1) // block_size
    bt = np.full((3, cols), -1, dtype=np.int32)
    cache_k = np.zeros((total, 2, block_size, 16), dtype=np.uint16)
    cache_v = np.zeros_like(cache_k)
    off = 0
    for b in range(3):
        for j in range(nblk[b]):
            blk = perm[off]; off += 1
            bt[b, j] = blk
            n_tok = min(block_size, int(lens[b]) - j * block_size)
            cache_k[blk, :, :n_tok] = case.key[b, :, j * block_size:j * block_size + n_tok]
            cache_v[blk, :, :n_tok] = case.value[b, :, j * block_size:j * block_size + n_tok]
    out_nbsd = oracle.ifa_ref(case.query, cache_k, cache_v, num_heads=4, num_kv_heads=2,
                              scale=case.scale, layout="BNSD", kv_format=oracle.PAGED_NBSD,
                              block_size=block_size, block_table=bt, actual_seq_lengths=lens)
    bsh_k = np.transpose(cache_k, (0, 2, 1, 3)).reshape(total, block_size, 32)
    bsh_v = np.transpose(cache_v, (0, 2, 1, 3)).reshape(total, block_size, 32)
    out_bsh = oracle.ifa_ref(case.query, bsh_k, bsh_v, num_heads=4, num_kv_heads=2,
                             scale=case.scale, layout="BNSD", kv_format=oracle.PAGED_BSH,
                             block_size=block_size, block_table=bt, actual_seq_lengths=lens)
    ref = run(case)
    assert np.array_equal(out_nbsd, ref)
    assert np.array_equal(out_bsh, ref)


def test_left_padded_window_equals_right_padded_cache():
    """Window [Smax - pad - len, Smax - pad) (IncreFlashAttention README, kv left padding)."""
    rng = np.random.default_rng(12)
    B, Smax = 3, 40
    right = gen.gqa_padded(12, B=B, N=4, KV_N=2, D=16, Smax=Smax, layout="BNSD", dtype="fp16", mask=False)
    lens = right.actual_seq_lengths
    pads = np.array([int(rng.integers(0, Smax - l + 1)) for l in lens], dtype=np.int64)
    k = gen.random_storage(99, 1, right.key.shape, "fp16")
    v = gen.random_storage(99, 2, right.value.shape, "fp16")
    for b in range(B):
        st = Smax - pads[b] - lens[b]
        k[b, :, st:st + lens[b]] = right.key[b, :, :lens[b]]
        v[b, :, st:st + lens[b]] = right.value[b, :, :lens[b]]
    out = oracle.ifa_ref(right.query, k, v, num_heads=4, num_kv_heads=2, scale=right.scale,
                         layout="BNSD", actual_seq_lengths=lens, kv_padding_size=pads)
    assert np.array_equal(out, run(right))


def test_left_pad_out_of_range_window_is_zero_and_negative_pad_is_zero_pad():
    case = gen.gqa_padded(13, B=3, N=2, KV_N=1, D=16, Smax=30, layout="BNSD", dtype="fp16", mask=False)
    case.actual_seq_lengths = np.array([25, 10, 30], dtype=np.int64)
    # b0: start = 30 - 8 - 25 < 0 -> zeros; b1: regular; b2: pad -5 -> treated as 0
    pads = np.array([8, 3, -5], dtype=np.int64)
    out = run(case, kv_padding_size=pads)
    assert np.all(out[0] == 0.0)
    assert not np.all(out[1] == 0.0)
    out0 = run(case, kv_padding_size=np.array([8, 3, 0], dtype=np.int64))
    assert np.array_equal(out[2], out0[2])
    # a single broadcast pad value applies to every batch
    one = run(case, kv_padding_size=np.array([0], dtype=np.int64))
    assert np.array_equal(one, run(case, kv_padding_size=np.zeros(3, dtype=np.int64)))


def test_mask_semantics():
    case = gen.gqa_padded(14, B=2, N=4, KV_N=2, D=16, Smax=24, layout="BNSD", dtype="bf16", mask=False)
    base = run(case)
    zeros = np.zeros((2, 1, 1, 24), dtype=bool)
    assert np.array_equal(run(case, atten_mask=zeros), base)
    # a mask true past each length equals the length-limited problem
    full = np.full(2, 24, dtype=np.int64)
    past = (np.arange(24)[None, :] >= case.actual_seq_lengths[:, None]).reshape(2, 1, 1, 24)
    assert np.array_equal(run(case, actual_seq_lengths=full, atten_mask=past), base)
    # per-head mask (B, N, 1, S): excluding everything for head 1 only
    m = np.zeros((2, 4, 1, 24), dtype=np.uint8)
    m[:, 1] = 1
    out = run(case, atten_mask=m)
    assert np.all(out[:, 1] == 0.0)
    assert np.array_equal(out[:, [0, 2, 3]], base[:, [0, 2, 3]])
    # a broadcast (1, N, 1, S) mask equals the same mask repeated over B
    m1 = (np.random.default_rng(3).random((1, 4, 1, 24)) < 0.3).astype(np.int8)
    assert np.array_equal(run(case, atten_mask=m1), run(case, atten_mask=np.repeat(m1, 2, axis=0)))
    # masked positions are simply dropped: compare with torch on the survivors
    q = as_f64(case.query, "bf16").reshape(2, 4, 16)
    k, v = as_f64(case.key, "bf16"), as_f64(case.value, "bf16")
    got = run(case, atten_mask=m1)
    for b in range(2):
        L = int(case.actual_seq_lengths[b])
        for n in range(4):
            valid = m1[0, n, 0, :L] == 0
            ref = torch_attention(q[b, n], k[b, n // 2, :L], v[b, n // 2, :L], case.scale, valid)
            np.testing.assert_allclose(got[b, n], ref, rtol=1e-12, atol=1e-13)


def test_zero_length_row_is_zero():
    case = gen.gqa_padded(15, B=2, N=2, KV_N=1, D=16, Smax=10, layout="BNSD", dtype="fp16", mask=False)
    case.actual_seq_lengths = np.array([0, 4], dtype=np.int64)
    out = run(case)
    assert np.all(out[0] == 0.0)
    assert not np.all(out[1] == 0.0)


def test_permuting_tokens_together_leaves_output_unchanged():
    case = gen.gqa_padded(16, B=1, N=2, KV_N=1, D=16, Smax=64, layout="BNSD", dtype="fp16", mask=False)
    case.actual_seq_lengths = np.array([64], dtype=np.int64)
    perm = np.random.default_rng(0).permutation(64)
    out = run(case)
    case.key, case.value = case.key[:, :, perm], case.value[:, :, perm]
    np.testing.assert_allclose(run(case), out, rtol=1e-13, atol=1e-15)


# ---------------------------------------------------------------- antiquant

def _int8_case(seed, per_tensor=False):
    return gen.int8_leftpad(seed, B=2, N=4, KV_N=2, D=16, Smax=48, len_lo=5, len_hi=40, pad_extra=4,
                            per_tensor=per_tensor)


def _aq(case, **over):
    kw = dict(antiquant=oracle.AQ_PER_TENSOR if case.antiquant == "per_tensor" else oracle.AQ_PER_CHANNEL,
              antiquant_scale=case.antiquant_scale, antiquant_offset=case.antiquant_offset)
    kw.update(over)
    return run(case, **kw)


def test_antiquant_value_formula_on_constant_rows():
    """With every int8 value row equal to c, out[d] = (c + offset_V[h,d]) * scale_V[h,d] exactly."""
    case = _int8_case(20)
    case.value = np.full_like(case.value, 7)
    out = _aq(case)
    s = case.antiquant_scale.astype(np.float64).reshape(2, 2, 16)
    o = case.antiquant_offset.astype(np.float64).reshape(2, 2, 16)
    for b in range(2):
        for n in range(4):
            np.testing.assert_allclose(out[b, n], (7 + o[1, n // 2]) * s[1, n // 2], rtol=1e-14)


def test_antiquant_scales_against_torch_on_dequantised_values():
    """Zero offsets: softmax over k*scale_K against v*scale_V, computed by torch in float64."""
    case = _int8_case(21)
    case.antiquant_offset = np.zeros_like(case.antiquant_offset)
    out = _aq(case)
    s = case.antiquant_scale.astype(np.float64).reshape(2, 2, 16)
    q = case.query.astype(np.float64).reshape(2, 4, 16)
    k = case.key.astype(np.float64)
    v = case.value.astype(np.float64)
    for b in range(2):
        pad = max(int(case.kv_padding_size[b]), 0)
        st = 48 - pad - int(case.actual_seq_lengths[b])
        en = 48 - pad
        for n in range(4):
            h = n // 2
            if st < 0:
                assert np.all(out[b, n] == 0)
                continue
            ref = torch_attention(q[b, n], k[b, h, st:en] * s[0, h], v[b, h, st:en] * s[1, h], case.scale)
            np.testing.assert_allclose(out[b, n], ref, rtol=1e-11, atol=1e-13)


def test_antiquant_key_offset_only_shifts_scores():
    """A per-channel key offset adds the same constant to every score of a row."""
    case = _int8_case(22)
    a = _aq(case)
    off = case.antiquant_offset.copy()
    off[0] = np.float16(0.0)
    b = _aq(case, antiquant_offset=off)
    np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-12)


def test_antiquant_per_tensor_equals_broadcast_per_channel():
    case = _int8_case(23, per_tensor=True)
    pt = _aq(case)
    sc = np.repeat(case.antiquant_scale.reshape(2, 1), 2 * 16, axis=1).reshape(2, 2, 1, 16)
    of = np.repeat(case.antiquant_offset.reshape(2, 1), 2 * 16, axis=1).reshape(2, 2, 1, 16)
    pc = _aq(case, antiquant=oracle.AQ_PER_CHANNEL, antiquant_scale=sc, antiquant_offset=of)
    assert np.array_equal(pt, pc)


def test_antiquant_identity_params_equal_plain_fp16():
    case = _int8_case(24)
    one = np.ones_like(case.antiquant_scale)
    zero = np.zeros_like(case.antiquant_offset)
    a = _aq(case, antiquant_scale=one, antiquant_offset=zero)
    kf = case.key.astype(np.float16)
    vf = case.value.astype(np.float16)
    b = oracle.ifa_ref(case.query, kf, vf, num_heads=4, num_kv_heads=2, scale=case.scale,
                       layout="BNSD", actual_seq_lengths=case.actual_seq_lengths,
                       kv_padding_size=case.kv_padding_size)
    assert np.array_equal(a, b)


# ---------------------------------------------------------------- sparse MLA decode

def _sfa(seed=0, **kw):
    base = dict(B=2, Q_N=4, D=32, Dr=8, block_size=16, kv_len=64, sparse_size=16, nvalid_lo=4,
                nvalid_hi=16)
    base.update(kw)
    return gen.sfa_mla(seed, **base)


def sref(c, **over):
    a = dict(query=c.query, query_rope=c.query_rope, key=c.key, key_rope=c.key_rope, value=c.value,
             sparse_indices=c.sparse_indices, block_table=c.block_table,
             actual_seq_lengths_kv=c.actual_seq_lengths_kv)
    a.update(over)
    return oracle.sfa_ref(a["query"], a["query_rope"], a["key"], a["key_rope"], a["value"],
                          a["sparse_indices"], a["block_table"], a["actual_seq_lengths_kv"], scale=c.scale)


def _rows(c, b, idx):
    bs = c.key.shape[1]
    return np.array([c.block_table[b, i // bs] * bs + i % bs for i in idx])


def test_sfa_dense_indices_match_torch_mla():
    c = _sfa(30)
    c.sparse_indices[:] = np.arange(16, dtype=np.int32)
    out = sref(c)
    q = as_f64(c.query, "bf16")[:, 0]
    qr = as_f64(c.query_rope, "bf16")[:, 0]
    k = as_f64(c.key, "bf16").reshape(-1, 32)
    kr = as_f64(c.key_rope, "bf16").reshape(-1, 8)
    v = as_f64(c.value, "bf16").reshape(-1, 32)
    for b in range(2):
        rows = _rows(c, b, range(16))
        for n in range(4):
            ref = torch_attention(np.concatenate([q[b, n], qr[b, n]]),
                                  np.concatenate([k[rows], kr[rows]], axis=1), v[rows], c.scale)
            np.testing.assert_allclose(out[b, n], ref, rtol=1e-12, atol=1e-13)


def test_sfa_single_index_returns_value_row_and_all_invalid_is_zero():
    c = _sfa(31)
    c.sparse_indices[:] = -1
    c.sparse_indices[0, 0, 0, 0] = 37
    out = sref(c)
    v = as_f64(c.value, "bf16").reshape(-1, 32)
    row = _rows(c, 0, [37])[0]
    for n in range(4):
        assert np.array_equal(out[0, n], v[row])
    assert np.all(out[1] == 0.0)


def test_sfa_selected_set_exact_mean():
    """Q = 0 and value row = integer code of its token: the output is the exact mean of the
    codes of exactly the valid selected tokens (invalid entries anywhere are skipped)."""
    c = _sfa(32)
    c.query[:] = 0
    c.query_rope[:] = 0
    bs = 16
    codes = np.zeros(c.value.shape, dtype=np.float32)
    # code(token) = token index of the row within its batch, recovered from the block table
    for b in range(2):
        for t in range(64):
            blk = c.block_table[b, t // bs]
            codes[blk, t % bs, 0, :] = t
    c.value = gen.to_storage(codes, "bf16")
    sel = np.array([3, 60, 17, 8, -1, 70, 5, 9], dtype=np.int32)   # 70 >= length, -1 invalid
    idx = np.full((2, 1, 1, 16), -1, dtype=np.int32)
    idx[0, 0, 0, :8] = sel
    idx[1, 0, 0, :4] = [1, 2, 3, 6]
    lens = np.array([64, 64], dtype=np.int32)
    out = sref(c, sparse_indices=idx, actual_seq_lengths_kv=lens)
    valid0 = [3, 60, 17, 8, 5, 9]
    assert np.all(out[0] == np.mean(valid0))
    assert np.all(out[1] == 3.0)
    # a shorter actual length drops index 60 as well
    out2 = sref(c, sparse_indices=idx, actual_seq_lengths_kv=np.array([40, 64], dtype=np.int32))
    assert np.all(out2[0] == np.mean([3, 17, 8, 5, 9]))


def test_sfa_index_order_is_irrelevant_and_duplicates_count_twice():
    c = _sfa(33, nvalid_lo=10, nvalid_hi=10)
    out = sref(c)
    idx = c.sparse_indices.copy()
    idx[:, :, :, :10] = idx[:, :, :, :10][..., ::-1]
    np.testing.assert_allclose(sref(c, sparse_indices=idx), out, rtol=1e-13, atol=1e-15)
    dup = c.sparse_indices.copy()
    dup[:, :, :, 10] = dup[:, :, :, 0]
    got = sref(c, sparse_indices=dup)
    q = as_f64(c.query, "bf16")[:, 0]
    qr = as_f64(c.query_rope, "bf16")[:, 0]
    k = as_f64(c.key, "bf16").reshape(-1, 32)
    kr = as_f64(c.key_rope, "bf16").reshape(-1, 8)
    v = as_f64(c.value, "bf16").reshape(-1, 32)
    for b in range(2):
        rows = _rows(c, b, dup[b, 0, 0, :11])
        for n in range(4):
            ref = torch_attention(np.concatenate([q[b, n], qr[b, n]]),
                                  np.concatenate([k[rows], kr[rows]], axis=1), v[rows], c.scale)
            np.testing.assert_allclose(got[b, n], ref, rtol=1e-12, atol=1e-13)


def sref_block(c, sbs, **over):
    a = dict(sparse_indices=c.sparse_indices, actual_seq_lengths_kv=c.actual_seq_lengths_kv)
    a.update(over)
    return oracle.sfa_ref(c.query, c.query_rope, c.key, c.key_rope, c.value, a["sparse_indices"], c.block_table,
                          a["actual_seq_lengths_kv"], scale=c.scale, sparse_block_size=sbs)


@pytest.mark.parametrize("sbs", [2, 4, 16])
def test_sfa_blockwise_selected_set_exact_mean(sbs):
    """Block-wise sparsity (SparseFlashAttention README, sparse_block_size): with Q = 0 and each
    value row holding its token index, the output is the exact mean of the indices of the valid
    tokens of the selected blocks: tokens idx*sbs .. idx*sbs+sbs-1 below the length, nothing for
    a negative entry, duplicates counted twice."""
    c = _sfa(34)
    c.query[:] = 0
    c.query_rope[:] = 0
    bs = 16
    codes = np.zeros(c.value.shape, dtype=np.float32)
    for b in range(2):
        for t in range(64):
            codes[c.block_table[b, t // bs], t % bs, 0, :] = t
    c.value = gen.to_storage(codes, "bf16")
    nblk = 64 // sbs
    idx = np.full((2, 1, 1, 16), -1, dtype=np.int32)
    sel0 = [nblk - 1, 0, -1, 2 % nblk, 0]          # last block, a duplicate, an invalid entry
    idx[0, 0, 0, :len(sel0)] = sel0
    idx[1, 0, 0, :2] = [1, nblk - 1]
    lens = np.array([64, 64 - sbs // 2 - 1], dtype=np.int32)  # batch 1: last block partly past the length
    out = sref_block(c, sbs, sparse_indices=idx, actual_seq_lengths_kv=lens)
    for b, sel in ((0, sel0), (1, [1, nblk - 1])):
        toks = [i * sbs + o for i in sel if i >= 0 for o in range(sbs) if i * sbs + o < lens[b]]
        assert np.all(out[b] == np.mean(toks)), (b, sbs)


@pytest.mark.parametrize("sbs", [2, 8])
def test_sfa_blockwise_equals_tokenwise_on_expanded_indices(sbs):
    c = _sfa(35, kv_len=64, sparse_size=8, nvalid_lo=3, nvalid_hi=8)
    rng = np.random.default_rng(35)
    nblk = 64 // sbs
    blk = np.full((2, 1, 1, 8), -1, dtype=np.int32)
    for b in range(2):
        blk[b, 0, 0, :5] = rng.choice(nblk, size=5, replace=False)
    lens = np.array([64, 50], dtype=np.int32)
    tok = np.full((2, 1, 1, 8 * sbs), -1, dtype=np.int32)
    for b in range(2):
        for j in range(8):
            if blk[b, 0, 0, j] >= 0:
                tok[b, 0, 0, j * sbs:(j + 1) * sbs] = blk[b, 0, 0, j] * sbs + np.arange(sbs)
    got = sref_block(c, sbs, sparse_indices=blk, actual_seq_lengths_kv=lens)
    want = sref_block(c, 1, sparse_indices=tok, actual_seq_lengths_kv=lens)
    assert np.array_equal(got, want)


# ------------------------------------------- multi-token queries and the right-down causal mode

def _sfa_mtp(seed, Q_S, **kw):
    base = dict(B=2, Q_N=4, D=32, Dr=8, block_size=16, kv_len=64, sparse_size=16, nvalid_lo=4,
                nvalid_hi=16, Q_S=Q_S)
    base.update(kw)
    return gen.sfa_mla(seed, **base)


def _token_codes(c, kv_len=64, bs=16):
    codes = np.zeros(c.value.shape, dtype=np.float32)
    for b in range(c.B):
        for t in range(kv_len):
            codes[c.block_table[b, t // bs], t % bs, 0, :] = t
    return gen.to_storage(codes, "bf16")


def test_sfa_multi_token_rows_match_torch_mla_per_row():
    """Q_S = 3, sparse_mode 0: query token s of batch b attends over its own index row
    (b, s) with its own query; each row is checked against the dense library attention."""
    c = _sfa_mtp(40, 3)
    out = oracle.sfa_ref(c.query, c.query_rope, c.key, c.key_rope, c.value, c.sparse_indices, c.block_table,
                         c.actual_seq_lengths_kv, scale=c.scale)
    assert out.shape == (2, 3, 4, 32)
    q = as_f64(c.query, "bf16")
    qr = as_f64(c.query_rope, "bf16")
    k = as_f64(c.key, "bf16").reshape(-1, 32)
    kr = as_f64(c.key_rope, "bf16").reshape(-1, 8)
    v = as_f64(c.value, "bf16").reshape(-1, 32)
    for b in range(2):
        for s in range(3):
            sel = [i for i in c.sparse_indices[b, s, 0] if i >= 0]
            rows = _rows(c, b, sel)
            for n in range(4):
                ref = torch_attention(np.concatenate([q[b, s, n], qr[b, s, n]]),
                                      np.concatenate([k[rows], kr[rows]], axis=1), v[rows], c.scale)
                np.testing.assert_allclose(out[b, s, n], ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("sbs", [1, 4])
def test_sfa_right_down_causal_exact_means(sbs):
    """sparse_mode 3 (rightDownCausal) with Q = 0, value row = token index and every token
    selected: with len keys and qlen valid query tokens, query token s < qlen averages tokens
    0 .. len - qlen + s exactly, i.e. (len - qlen + s) / 2; tokens s >= qlen give zero rows;
    sparse_mode 0 averages every token below len for each valid row."""
    Q_S = 4
    c = _sfa_mtp(41, Q_S)
    c.query[:] = 0
    c.query_rope[:] = 0
    c.value = _token_codes(c)
    idx = np.full((2, Q_S, 1, 64), -1, dtype=np.int32)
    idx[:, :, 0, :64 // sbs] = np.arange(64 // sbs, dtype=np.int32)
    lens = np.array([64, 50], dtype=np.int32)
    for lq in (None, np.array([4, 2], dtype=np.int32), np.array([0, 1], dtype=np.int32)):
        qlen = np.full(2, Q_S) if lq is None else lq
        for mode in (0, 3):
            out = oracle.sfa_ref(c.query, c.query_rope, c.key, c.key_rope, c.value, idx, c.block_table, lens,
                                 scale=c.scale, sparse_block_size=sbs, sparse_mode=mode,
                                 actual_seq_lengths_query=lq)
            for b in range(2):
                for s in range(Q_S):
                    if s >= qlen[b]:
                        assert np.all(out[b, s] == 0.0), (b, s, mode)
                        continue
                    last = lens[b] - qlen[b] + s if mode == 3 else lens[b] - 1
                    assert np.all(out[b, s] == last / 2.0), (b, s, mode, lq)


def test_sfa_causal_mode_equals_explicit_index_pruning():
    """Under sparse_mode 3 a selected token past a query token's causal position counts for
    nothing: the output equals sparse_mode 0 on indices with those entries set to -1."""
    Q_S = 3
    c = _sfa_mtp(42, Q_S, nvalid_lo=16, nvalid_hi=16)
    lens = np.array([60, 64], dtype=np.int32)
    lq = np.array([3, 2], dtype=np.int32)
    # make sure the last tokens are selected somewhere in every row
    c.sparse_indices[:, :, 0, :3] = np.array([lens.min() - 1, lens.min() - 2, lens.min() - 3])[None, None]
    c.sparse_indices[1, :, 0, 3:6] = np.array([63, 62, 61])
    causal = oracle.sfa_ref(c.query, c.query_rope, c.key, c.key_rope, c.value, c.sparse_indices, c.block_table,
                            lens, scale=c.scale, sparse_mode=3, actual_seq_lengths_query=lq)
    pruned = c.sparse_indices.copy()
    for b in range(2):
        for s in range(Q_S):
            row = pruned[b, s, 0]
            row[row > lens[b] - lq[b] + s] = -1
    plain = oracle.sfa_ref(c.query, c.query_rope, c.key, c.key_rope, c.value, pruned, c.block_table, lens,
                           scale=c.scale, sparse_mode=0, actual_seq_lengths_query=lq)
    assert np.array_equal(causal, plain)
    assert np.all(causal[1, 2] == 0.0)
    # something was pruned, so the modes differ on at least one valid row
    full = oracle.sfa_ref(c.query, c.query_rope, c.key, c.key_rope, c.value, c.sparse_indices, c.block_table,
                          lens, scale=c.scale, sparse_mode=0, actual_seq_lengths_query=lq)
    assert not np.array_equal(full[0, 0], causal[0, 0])


# ------------------------------------------- TND / BSND layouts and the softmax_max / softmax_sum outputs

def _contig_kv(c, kv_len=64, bs=16):
    """The paged caches of an SFA case rewritten as BSND (B, KV_S, 1, d) tensors."""
    B = c.B
    def gather(t):
        outp = np.zeros((B, kv_len) + t.shape[2:], dtype=t.dtype)
        for b in range(B):
            for tok in range(kv_len):
                outp[b, tok] = t[c.block_table[b, tok // bs], tok % bs]
        return outp
    return gather(c.key), gather(c.key_rope), gather(c.value)


@pytest.mark.parametrize("mode", [0, 3])
def test_sfa_bsnd_and_tnd_kv_equal_the_paged_cache(mode):
    """layout_kv BSND (row b * KV_S + t) and TND (row lens_kv[b-1] + t, prefix-sum lengths)
    address the same tokens as PA_BSND through the block table: identical outputs."""
    c = _sfa_mtp(50, 2, sparse_mode=mode)
    lens = np.array([64, 41], dtype=np.int32)
    paged = oracle.sfa_ref(c.query, c.query_rope, c.key, c.key_rope, c.value, c.sparse_indices, c.block_table,
                           lens, scale=c.scale, sparse_mode=mode)
    k, kr, v = _contig_kv(c)
    bsnd = oracle.sfa_ref(c.query, c.query_rope, k, kr, v, c.sparse_indices, None, lens, scale=c.scale,
                          sparse_mode=mode, layout_kv="BSND")
    assert np.array_equal(paged, bsnd)
    # TND: batch 1 packed right after batch 0's 64 rows
    kt = np.concatenate([k[0, :64], k[1, :41]])
    krt = np.concatenate([kr[0, :64], kr[1, :41]])
    vt = np.concatenate([v[0, :64], v[1, :41]])
    tnd = oracle.sfa_ref(c.query, c.query_rope, kt, krt, vt, c.sparse_indices, None,
                         np.array([64, 105], dtype=np.int32), scale=c.scale, sparse_mode=mode, layout_kv="TND")
    assert np.array_equal(paged, tnd)
    # BSND without lengths uses KV_S for every batch
    full = oracle.sfa_ref(c.query, c.query_rope, k, kr, v, c.sparse_indices, None, None, scale=c.scale,
                          sparse_mode=mode, layout_kv="BSND")
    ref = oracle.sfa_ref(c.query, c.query_rope, c.key, c.key_rope, c.value, c.sparse_indices, c.block_table,
                         np.array([64, 64], dtype=np.int32), scale=c.scale, sparse_mode=mode)
    assert np.array_equal(full, ref)


@pytest.mark.parametrize("mode", [0, 3])
def test_sfa_tnd_query_rows_match_bsnd_rows_and_torch(mode):
    """layout_query TND packs each batch's qlen valid query rows (prefix-sum
    actual_seq_lengths_query); each packed row equals the BSND row (b, s) with the same
    qlen, and matches the dense library attention over its selected tokens."""
    Q_S = 3
    c = _sfa_mtp(51, Q_S, sparse_mode=mode, nvalid_lo=16, nvalid_hi=16)
    qlen = np.array([3, 2], dtype=np.int32)
    bsnd = oracle.sfa_ref(c.query, c.query_rope, c.key, c.key_rope, c.value, c.sparse_indices, c.block_table,
                          c.actual_seq_lengths_kv, scale=c.scale, sparse_mode=mode, actual_seq_lengths_query=qlen)
    rows = [(b, s) for b in range(2) for s in range(qlen[b])]
    qt = np.stack([c.query[b, s] for b, s in rows])
    qrt = np.stack([c.query_rope[b, s] for b, s in rows])
    it = np.stack([c.sparse_indices[b, s] for b, s in rows])
    tnd = oracle.sfa_ref(qt, qrt, c.key, c.key_rope, c.value, it, c.block_table, c.actual_seq_lengths_kv,
                         scale=c.scale, sparse_mode=mode, actual_seq_lengths_query=np.cumsum(qlen).astype(np.int32),
                         layout_query="TND")
    assert tnd.shape == (5, 4, 32)
    for t, (b, s) in enumerate(rows):
        assert np.array_equal(tnd[t], bsnd[b, s])
    q = as_f64(qt, "bf16")
    qr = as_f64(qrt, "bf16")
    k = as_f64(c.key, "bf16").reshape(-1, 32)
    kr = as_f64(c.key_rope, "bf16").reshape(-1, 8)
    v = as_f64(c.value, "bf16").reshape(-1, 32)
    L = 64
    for t, (b, s) in enumerate(rows):
        lim = L - qlen[b] + s + 1 if mode == 3 else L
        sel = [i for i in it[t, 0] if 0 <= i < lim]
        r_ = _rows(c, b, sel)
        for n in range(4):
            ref = torch_attention(np.concatenate([q[t, n], qr[t, n]]), np.concatenate([k[r_], kr[r_]], axis=1),
                                  v[r_], c.scale)
            np.testing.assert_allclose(tnd[t, n], ref, rtol=1e-12, atol=1e-13)


def test_sfa_tnd_rows_past_the_last_prefix_are_zero():
    c = _sfa_mtp(52, 1)
    qt = c.query[:, 0]
    qrt = c.query_rope[:, 0]
    it = c.sparse_indices[:, 0]
    out, mx, sm = oracle.sfa_ref(qt, qrt, c.key, c.key_rope, c.value, it, c.block_table, c.actual_seq_lengths_kv,
                                 scale=c.scale, actual_seq_lengths_query=np.array([1], dtype=np.int32),
                                 layout_query="TND", return_softmax_lse=True)
    # one batch of one row: row 1 belongs to no batch
    assert np.all(out[1] == 0.0) and np.all(mx[1] == -np.inf) and np.all(sm[1] == 0.0)
    assert np.all(np.isfinite(out[0])) and np.any(out[0] != 0.0)


def test_sfa_softmax_max_and_sum_closed_forms():
    """Q = 0: every score is 0, so softmax_max = 0 and softmax_sum = the number of valid
    selected tokens (exact); rows with nothing selected give -inf and 0.  Random Q: max and
    max + log(sum) equal numpy's max and logsumexp of the scaled scores."""
    from scipy.special import logsumexp
    c = _sfa_mtp(53, 2, sparse_mode=3)
    lens = np.array([64, 30], dtype=np.int32)
    c.sparse_indices[1, 1] = -1
    zq = np.zeros_like(c.query)
    zr = np.zeros_like(c.query_rope)
    _, mx, sm = oracle.sfa_ref(zq, zr, c.key, c.key_rope, c.value, c.sparse_indices, c.block_table, lens,
                               scale=c.scale, sparse_mode=3, return_softmax_lse=True)
    for b in range(2):
        for s in range(2):
            lim = lens[b] - 2 + s + 1
            cnt = int(sum(1 for i in c.sparse_indices[b, s, 0] if 0 <= i < lim))
            if cnt == 0:
                assert np.all(mx[b, s] == -np.inf) and np.all(sm[b, s] == 0.0)
            else:
                assert np.all(mx[b, s] == 0.0) and np.all(sm[b, s] == float(cnt)), (b, s)
    out, mx, sm = oracle.sfa_ref(c.query, c.query_rope, c.key, c.key_rope, c.value, c.sparse_indices,
                                 c.block_table, lens, scale=c.scale, sparse_mode=3, return_softmax_lse=True)
    q = as_f64(c.query, "bf16")
    qr = as_f64(c.query_rope, "bf16")
    k = as_f64(c.key, "bf16").reshape(-1, 32)
    kr = as_f64(c.key_rope, "bf16").reshape(-1, 8)
    for b in range(2):
        s = 0
        lim = lens[b] - 2 + s + 1
        r_ = _rows(c, b, [i for i in c.sparse_indices[b, s, 0] if 0 <= i < lim])
        kk = np.concatenate([k[r_], kr[r_]], axis=1)
        for n in range(4):
            sc = (kk @ np.concatenate([q[b, s, n], qr[b, s, n]])) * c.scale
            assert mx[b, s, n] == pytest.approx(sc.max(), rel=1e-13, abs=1e-13)
            assert mx[b, s, n] + math.log(sm[b, s, n]) == pytest.approx(logsumexp(sc), rel=1e-12, abs=1e-12)


@pytest.mark.parametrize("Q_S,mode", [(1, 0), (2, 3)])
def test_sfa_softmax_sum_bit_probe_fingerprint(Q_S, mode):
    """The probe the GPU split-path test uses: scores -bit_j(t) at scale ln 2 make every
    probability 1 or 1/2, so softmax_sum is a count-based closed form of the selected set (the
    number of selected tokens with bit j clear, plus half of those with it set) and softmax_max
    is 0 or -ln 2.  Checked exactly, including the causal limit's last key."""
    from harness import sfa_bit_probe
    c = gen.sfa_mla(5, B=3, Q_N=16, block_size=64, kv_len=4096, sparse_size=300, nvalid_lo=100, nvalid_hi=300,
                    Q_S=Q_S, sparse_mode=mode)
    c.sparse_indices[0, :, 0, 0] = 4095  # the last key: visible to the last query token only under mode 3
    c.sparse_indices[2] = -1             # nothing selected
    c, exp_sum, exp_max = sfa_bit_probe(c)
    _, mx, sm = oracle.sfa_ref(c.query, c.query_rope, c.key, c.key_rope, c.value, c.sparse_indices,
                               c.block_table, c.actual_seq_lengths_kv, scale=c.scale, sparse_mode=mode,
                               return_softmax_lse=True)
    sm, mx = sm.reshape(exp_sum.shape), mx.reshape(exp_max.shape)
    assert np.array_equal(sm, exp_sum)
    assert np.array_equal(np.isneginf(mx), np.isneginf(exp_max))
    live = ~np.isneginf(exp_max)
    assert np.abs(mx[live] - exp_max[live]).max() <= 1e-15
    # a swapped token changes the fingerprint: move one selected index of batch 1, first query token
    c2 = c
    c2.sparse_indices = c.sparse_indices.copy()
    i0 = int(c2.sparse_indices[1, 0, 0, 1])
    c2.sparse_indices[1, 0, 0, 1] = i0 ^ 1 if (i0 ^ 1) not in set(c2.sparse_indices[1, 0, 0].tolist()) else i0 ^ 2
    _, _, sm2 = oracle.sfa_ref(c2.query, c2.query_rope, c2.key, c2.key_rope, c2.value, c2.sparse_indices,
                               c2.block_table, c2.actual_seq_lengths_kv, scale=c2.scale, sparse_mode=mode,
                               return_softmax_lse=True)
    assert not np.array_equal(sm2.reshape(exp_sum.shape)[Q_S], exp_sum[Q_S])


# ------------------------------------------- KV-cache append

def _place(cache, new, pos, layout, kv_format, block_size=0, block_table=None):
    """numpy placement of the new token rows (B, KV_N, D) at positions pos."""
    c = cache.copy()
    B, KVN, D = new.shape
    for b in range(B):
        t = int(pos[b])
        if kv_format == oracle.CONTIG:
            if layout == "BNSD":
                c[b, :, t, :] = new[b]
            elif layout == "BSND":
                c[b, t, :, :] = new[b]
            else:
                c[b, t, :] = new[b].reshape(-1)
        else:
            blk, slot = block_table[b, t // block_size], t % block_size
            if kv_format == oracle.PAGED_NBSD:
                c[blk, :, slot, :] = new[b]
            else:
                c[blk, slot, :] = new[b].reshape(-1)
    return c


@pytest.mark.parametrize("layout,kv_format", [("BNSD", oracle.CONTIG), ("BSND", oracle.CONTIG), ("BSH", oracle.CONTIG),
                                              ("BNSD", oracle.PAGED_NBSD), ("BSH", oracle.PAGED_BSH)])
def test_kv_append_16bit_places_rows_exactly(layout, kv_format):
    rng = np.random.default_rng(60)
    B, KVN, D, S, bs = 3, 2, 16, 40, 16
    kn = rng.standard_normal((B, KVN, D)).astype(np.float16)
    vn = rng.standard_normal((B, KVN, D)).astype(np.float16)
    pos = np.array([0, 17, 39])
    bt = None
    if kv_format == oracle.CONTIG:
        shape = {"BNSD": (B, KVN, S, D), "BSND": (B, S, KVN, D), "BSH": (B, S, KVN * D)}[layout]
    else:
        bt = rng.permutation(B * 3).astype(np.int32).reshape(B, 3)
        shape = (B * 3, KVN, bs, D) if kv_format == oracle.PAGED_NBSD else (B * 3, bs, KVN * D)
    kc = rng.standard_normal(shape).astype(np.float16)
    vc = rng.standard_normal(shape).astype(np.float16)
    k2, v2, bad = oracle.kv_append_ref(kn, vn, pos, kc, vc, layout=layout, kv_format=kv_format, block_size=bs,
                                       block_table=bt)
    assert bad == 0
    assert np.array_equal(k2.view(np.uint16), _place(kc, kn, pos, layout, kv_format, bs, bt).view(np.uint16))
    assert np.array_equal(v2.view(np.uint16), _place(vc, vn, pos, layout, kv_format, bs, bt).view(np.uint16))


def test_kv_append_then_attend_equals_attention_over_the_longer_cache():
    """Appending at position len and attending over len + 1 tokens equals attention over a
    cache that held the token from the start (IncreFlashAttention's incremental step)."""
    c = gen.paged_gqa(61, B=2, N=8, KV_N=2, D=32, block_size=16, len_lo=20, len_hi=40)
    rng = np.random.default_rng(61)
    lens = c.actual_seq_lengths.astype(np.int64)
    kn = gen.to_storage(rng.standard_normal((2, 2, 32)).astype(np.float32), "bf16")
    vn = gen.to_storage(rng.standard_normal((2, 2, 32)).astype(np.float32), "bf16")
    k2, v2, bad = oracle.kv_append_ref(kn, vn, lens, c.key, c.value, kv_format=oracle.PAGED_NBSD,
                                       block_size=16, block_table=c.block_table)
    assert bad == 0
    got = oracle.ifa_ref(c.query, k2, v2, num_heads=8, num_kv_heads=2, scale=c.scale, kv_format=oracle.PAGED_NBSD,
                         block_size=16, block_table=c.block_table, actual_seq_lengths=lens + 1)
    q = as_f64(c.query, "bf16").reshape(2, 8, 32)
    for b in range(2):
        L = int(lens[b])
        rows = [c.block_table[b, t // 16] for t in range(L)]
        k = np.stack([as_f64(c.key[rows[t], :, t % 16], "bf16") for t in range(L)] + [as_f64(kn[b], "bf16")])
        v = np.stack([as_f64(c.value[rows[t], :, t % 16], "bf16") for t in range(L)] + [as_f64(vn[b], "bf16")])
        for n in range(8):
            ref = torch_attention(q[b, n], k[:, n // 4], v[:, n // 4], c.scale)
            np.testing.assert_allclose(got[b, n], ref, rtol=1e-12, atol=1e-13)


def test_kv_append_int8_codes_invert_the_antiquant_reading():
    """int8 caches: the code c of x satisfies (c + offset) * scale = x exactly when x is such a
    value; otherwise |(c + offset) * scale - x| <= scale / 2 unless saturated at -128 / 127;
    an exact half rounds to the even code."""
    B, KVN, D = 2, 2, 8
    sc = np.full((2, KVN, D), 2.0 ** -6, dtype=np.float16)
    of = np.broadcast_to(np.arange(D, dtype=np.float16) - 4, (2, KVN, D)).copy()
    codes = np.arange(-60, 60, 15)[:D]
    x = ((codes[None, None, :] + of[0].astype(np.float64)) * 2.0 ** -6).astype(np.float16)
    x = np.broadcast_to(x, (B, KVN, D)).copy()
    kc = np.zeros((B, KVN, 4, D), dtype=np.int8)
    k2, v2, bad = oracle.kv_append_ref(x, x, np.array([1, 3]), kc, kc, antiquant=oracle.AQ_PER_CHANNEL,
                                       antiquant_scale=sc, antiquant_offset=of)
    assert bad == 0 and np.array_equal(k2[0, :, 1], np.broadcast_to(codes, (KVN, D)))
    rng = np.random.default_rng(62)
    xr = rng.uniform(-2.5, 2.5, (B, KVN, D)).astype(np.float16)
    sc2 = rng.uniform(0.005, 0.02, (2, KVN, D)).astype(np.float16)
    of2 = rng.uniform(-4, 4, (2, KVN, D)).astype(np.float16)
    k3, v3, _ = oracle.kv_append_ref(xr, xr, np.array([0, 0]), kc, kc, antiquant=oracle.AQ_PER_CHANNEL,
                                     antiquant_scale=sc2, antiquant_offset=of2)
    for which, cache in ((0, k3), (1, v3)):
        c = cache[:, :, 0].astype(np.float64)
        s = sc2[which].astype(np.float64)
        o = of2[which].astype(np.float64)
        back = (c + o) * s
        inside = (c > -128) & (c < 127)
        err = np.abs(back - xr.astype(np.float64))
        assert np.all(err[inside] <= s[None].repeat(B, 0)[inside] / 2 * (1 + 1e-6))
    # saturation and ties (per-tensor parameters: scale 1, offset 0 -> code = rint(x))
    one = np.array([1.0, 1.0], dtype=np.float16)
    zero = np.zeros(2, dtype=np.float16)
    xt = np.array([[[300.0, -300.0, 2.5, 3.5, -2.5, 0.5, 126.5, -128.5]]], dtype=np.float16)
    k4, _, _ = oracle.kv_append_ref(xt, xt, np.array([0]), kc[:1, :1], kc[:1, :1], antiquant=oracle.AQ_PER_TENSOR,
                                    antiquant_scale=one, antiquant_offset=zero)
    assert list(k4[0, 0, 0]) == [127, -128, 2, 4, -2, 0, 126, -128]


def test_kv_append_skips_positions_outside_the_cache():
    rng = np.random.default_rng(63)
    kn = rng.standard_normal((3, 1, 8)).astype(np.float16)
    kc = rng.standard_normal((3, 1, 5, 8)).astype(np.float16)
    k2, v2, bad = oracle.kv_append_ref(kn, kn, np.array([-1, 5, 2]), kc, kc)
    assert bad == 2
    assert np.array_equal(k2[:2], kc[:2]) and np.array_equal(k2[2, 0, 2], kn[2, 0])
    bt = np.array([[0, -1], [7, 1], [2, 3]], dtype=np.int32)  # block 7 >= blocknum 4
    pc = rng.standard_normal((4, 1, 4, 8)).astype(np.float16)
    k3, _, bad = oracle.kv_append_ref(kn, kn, np.array([5, 1, 9]), pc, pc, kv_format=oracle.PAGED_NBSD,
                                      block_size=4, block_table=bt)
    assert bad == 3 and np.array_equal(k3, pc)  # entry -1, block 7, and a position past the table


# ------------------------------------------- int8 output quantisation (quantScale2 / quantOffset2)

def test_output_quantisation_of_integer_outputs_is_exact():
    """Value rows constant per channel make the attention output that constant (to rounding far
    below a code's width), so the codes are c * scale2 + offset2 by hand: scale 1, offset 0
    gives c itself."""
    case = gen.gqa_padded(70, B=2, N=4, KV_N=2, D=16, Smax=30, layout="BNSD", dtype="fp16", mask=False)
    consts = np.arange(-8, 8, dtype=np.float64)  # channel d carries the integer d - 8
    case.value = np.broadcast_to(consts.astype(np.float16), case.value.shape).copy()
    y = run(case)
    np.testing.assert_allclose(y, np.broadcast_to(consts, y.shape), rtol=1e-13, atol=1e-13)
    codes = oracle.quantize_output_ref(y, np.array([1.0], np.float32))
    assert np.array_equal(codes, np.broadcast_to(consts.astype(np.int8), codes.shape))
    codes = oracle.quantize_output_ref(y, np.array([2.0], np.float32), np.array([3.0], np.float32))
    assert np.array_equal(codes, np.broadcast_to((consts * 2 + 3).astype(np.int8), codes.shape))
    codes = oracle.quantize_output_ref(y, np.array([40.0], np.float32), np.array([-1.0], np.float32))
    assert np.array_equal(codes, np.broadcast_to(np.clip(consts * 40 - 1, -128, 127).astype(np.int8), codes.shape))


def test_output_quantisation_per_channel_ties_saturation_and_dtypes():
    rng = np.random.default_rng(71)
    y = rng.standard_normal((3, 4, 16))
    s = rng.uniform(10, 40, 64).astype(np.float32)
    o = rng.uniform(-5, 5, 64).astype(np.float32)
    pc = oracle.quantize_output_ref(y, s, o)
    # per-channel with every entry equal is per-tensor
    same = oracle.quantize_output_ref(y, np.full(64, s[0], np.float32), np.full(64, o[0], np.float32))
    assert np.array_equal(same, oracle.quantize_output_ref(y, s[:1], o[:1]))
    # per-channel entry n * D + d scales output channel (n, d)
    y1 = np.zeros((1, 4, 16))
    y1[0, 2, 5] = 1.0
    c1 = oracle.quantize_output_ref(y1, np.arange(1, 65, dtype=np.float32))
    assert c1[0, 2, 5] == 2 * 16 + 5 + 1 and np.count_nonzero(c1) == 1
    # bf16 parameters equal float32 ones holding the same values
    sb = gen.to_storage(s, "bf16")
    ob = gen.to_storage(o, "bf16")
    sf = (sb.astype(np.uint32) << 16).view(np.float32)
    of = (ob.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(oracle.quantize_output_ref(y, sb, ob), oracle.quantize_output_ref(y, sf, of))
    # ties to even, saturation, no offset
    yt = np.array([[[0.5, 1.5, 2.5, -0.5, -1.5, 200.0, -200.0, 127.4]]])
    assert list(oracle.quantize_output_ref(yt, np.array([1.0], np.float32))[0, 0]) == [0, 2, 2, 0, -2, 127, -128, 127]
    assert pc.dtype == np.int8 and np.all(np.abs(pc.astype(np.int64)) <= 128)


# ------------------------------------------- key/value as one tensor per batch (tensor list)

@pytest.mark.parametrize("layout", ["BNSD", "BSND", "BSH"])
def test_tensorlist_equals_the_contiguous_cache(layout):
    """Per-batch tensors cut from a contiguous cache (each ending at its own S_b past the
    length) give the contiguous result, with or without a per-batch mask."""
    case = gen.gqa_padded(90, B=4, N=8, KV_N=2, D=32, Smax=80, layout=layout, dtype="fp16", mask=True)
    ref = run(case)
    tl = gen.tensorlist_from(case, seed=1, extra_hi=9)
    s_axis = 2 if layout == "BNSD" else 1
    assert len({k.shape[s_axis] for k in tl.key}) > 1  # the extents really differ
    got = oracle.ifa_ref_tensorlist(tl.query, tl.key, tl.value, num_heads=8, num_kv_heads=2, scale=case.scale,
                                    layout=layout, atten_mask=tl.atten_mask, actual_seq_lengths=tl.actual_seq_lengths)
    assert np.array_equal(got, ref)


def test_tensorlist_tokens_past_the_length_do_not_count():
    case = gen.gqa_padded(91, B=3, N=4, KV_N=4, D=16, Smax=40, layout="BNSD", dtype="fp16", mask=False)
    tl = gen.tensorlist_from(case, seed=2, extra_hi=8)
    ref = oracle.ifa_ref_tensorlist(tl.query, tl.key, tl.value, num_heads=4, scale=case.scale,
                                    actual_seq_lengths=tl.actual_seq_lengths)
    poisoned_k = [k.copy() for k in tl.key]
    for b, k in enumerate(poisoned_k):
        k[:, :, int(tl.actual_seq_lengths[b]):, :] = np.float16(np.nan)
    got = oracle.ifa_ref_tensorlist(tl.query, poisoned_k, tl.value, num_heads=4, scale=case.scale,
                                    actual_seq_lengths=tl.actual_seq_lengths)
    assert np.array_equal(got, ref)
    # without lengths each batch attends over its whole tensor
    full = oracle.ifa_ref_tensorlist(tl.query, tl.key, tl.value, num_heads=4, scale=case.scale)
    for b in range(3):
        one = oracle.ifa_ref(tl.query[b:b + 1], tl.key[b], tl.value[b], num_heads=4, scale=case.scale)
        assert np.array_equal(full[b], one[0])


# ---------------------------------------------------------------- value decoding and argument rules

def test_every_finite_16bit_pattern_decodes_exactly():
    """With one valid token the softmax weight is exactly 1, so the output is that token's
    value row: checked for every finite fp16 bit pattern (subnormals included) against numpy's
    float16, and for every finite bf16 pattern against the float32 with those upper 16 bits."""
    D = 64
    for dtype in ("fp16", "bf16"):
        bits = np.arange(65536, dtype=np.uint32)
        exp_mask, exp_shift = (0x7C00, 10) if dtype == "fp16" else (0x7F80, 7)
        finite = bits[((bits & exp_mask) >> exp_shift) != (exp_mask >> exp_shift)].astype(np.uint16)
        rows = -(-finite.size // D)
        vals = np.zeros(rows * D, dtype=np.uint16)
        vals[:finite.size] = finite
        vals = vals.reshape(rows, 1, 1, D)  # BNSD (B=rows, KV_N=1, S=1, D)
        if dtype == "fp16":
            v = vals.view(np.float16)
            expect = v.astype(np.float64)
        else:
            v = vals
            expect = (vals.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
        q = np.zeros((rows, 1, 1, D), dtype=v.dtype)
        out = oracle.ifa_ref(q, v, v, num_heads=1, scale=1.0, layout="BNSD",
                             actual_seq_lengths=np.ones(rows, dtype=np.int64))
        assert np.array_equal(out.reshape(-1), expect.reshape(-1)), dtype


def test_lengths_the_cache_cannot_hold_are_rejected():
    """Reading 10: a batch's valid tokens are tokens of its cache.  A negative length, or
    (without left padding) one above the cache's S or above blockTableCols * blockSize, is
    refused, as the library refuses it; exactly S is accepted.  Left padding of a paged cache
    is refused too (reading 9)."""
    c = gen.gqa_padded(3, B=2, N=4, KV_N=2, D=16, Smax=40, layout="BNSD", dtype="fp16", mask=False)
    run(c, actual_seq_lengths=np.array([40, 7], dtype=np.int64))
    for lens in ([41, 7], [-1, 7]):
        with pytest.raises(ValueError):
            run(c, actual_seq_lengths=np.array(lens, dtype=np.int64))
    p = gen.paged_gqa(4, B=2, N=4, KV_N=2, D=16, block_size=16, len_lo=1, len_hi=64, dtype="fp16")
    cols = p.block_table.shape[1]
    kw = dict(num_heads=4, num_kv_heads=2, scale=p.scale, layout="BNSD", kv_format=oracle.PAGED_NBSD,
              block_size=16, block_table=p.block_table)
    oracle.ifa_ref(p.query, p.key, p.value, actual_seq_lengths=np.array([cols * 16, 5], np.int64), **kw)
    with pytest.raises(ValueError):
        oracle.ifa_ref(p.query, p.key, p.value, actual_seq_lengths=np.array([cols * 16 + 1, 5], np.int64), **kw)
    with pytest.raises(ValueError):
        oracle.ifa_ref(p.query, p.key, p.value, actual_seq_lengths=p.actual_seq_lengths,
                       kv_padding_size=np.array([0], np.int64), **kw)


def test_padding_sizes_without_lengths_leave_the_window_right_padded():
    """Reading 5: without actualSeqLengths every batch uses the whole cache, and kvPaddingSize
    has nothing to place."""
    c = gen.gqa_padded(5, B=2, N=4, KV_N=2, D=16, Smax=24, layout="BSND", dtype="bf16", mask=False)
    plain = run(c, actual_seq_lengths=None)
    padded = run(c, actual_seq_lengths=None, kv_padding_size=np.array([5, 9], dtype=np.int64))
    assert np.array_equal(plain, padded)
    assert np.array_equal(plain, run(c, actual_seq_lengths=np.array([24, 24], dtype=np.int64)))


def test_out_of_range_block_entries_are_counted_once_per_token_and_left_out():
    """Reading 11: a needed block-table entry outside [0, blockNum) leaves its tokens out for
    every head (the result equals the cache with those tokens masked) and the oracle counts
    each such token of the windows once, whatever the number of heads."""
    p = gen.paged_gqa(6, B=2, N=8, KV_N=2, D=16, block_size=16, len_lo=40, len_hi=64, dtype="bf16")
    bt = p.block_table.copy()
    lens = p.actual_seq_lengths
    bt[0, 1] = p.key.shape[0] + 3     # tokens 16..31 of batch 0
    bt[1, 0] = -7                     # tokens 0..15 of batch 1
    kw = dict(num_heads=8, num_kv_heads=2, scale=p.scale, layout="BNSD", kv_format=oracle.PAGED_NBSD,
              block_size=16, actual_seq_lengths=lens)
    out, nbad = oracle.ifa_ref(p.query, p.key, p.value, block_table=bt, return_bad_tokens=True, **kw)
    assert nbad == 32
    mask = np.zeros((2, 1, 1, bt.shape[1] * 16), dtype=bool)
    mask[0, :, :, 16:32] = True
    mask[1, :, :, 0:16] = True
    ref, none_bad = oracle.ifa_ref(p.query, p.key, p.value, block_table=p.block_table, atten_mask=mask,
                                   return_bad_tokens=True, **kw)
    assert none_bad == 0
    assert np.array_equal(out, ref)


def test_sfa_bsnd_tokens_past_the_key_tensor_are_skipped():
    """layout_kv BSND with a length above KV_S: selected tokens at or past KV_S are not in
    the batch's rows of the key tensor and select nothing, exactly as if their indices were -1
    (they must not reach the next batch's rows)."""
    c = _sfa(60, B=2, sparse_size=16, nvalid_lo=16, nvalid_hi=16)
    k, kr, v = _contig_kv(c, kv_len=64)
    idx = c.sparse_indices.copy()
    idx[0, 0, 0, :4] = [64, 66, 70, 71]  # past KV_S = 64 for batch 0, inside its length of 72
    lens = np.array([72, 64], dtype=np.int32)
    got = oracle.sfa_ref(c.query, c.query_rope, k, kr, v, idx, None, lens, scale=c.scale, layout_kv="BSND")
    pruned = idx.copy()
    pruned[0, 0, 0, :4] = -1
    ref = oracle.sfa_ref(c.query, c.query_rope, k, kr, v, pruned, None, np.array([64, 64], np.int32),
                         scale=c.scale, layout_kv="BSND")
    assert np.array_equal(got, ref)


def test_kv_append_bounds_at_the_edges_of_the_cache():
    """A position of -1 in a later batch, and a paged position exactly at blockTableCols *
    blockSize (whose entry would be the next row's first), write nothing: the neighbouring
    batch's rows and blocks stay as they were."""
    rng = np.random.default_rng(64)
    kn = rng.standard_normal((2, 1, 8)).astype(np.float16)
    kc = rng.standard_normal((2, 1, 5, 8)).astype(np.float16)
    k2, _, bad = oracle.kv_append_ref(kn, kn, np.array([0, -1]), kc, kc)
    assert bad == 1
    assert np.array_equal(k2[1], kc[1]) and np.array_equal(k2[0, 0, 1:], kc[0, 0, 1:])
    assert np.array_equal(k2[0, 0, 0], kn[0, 0])
    bt = np.array([[0, 1], [2, 3]], dtype=np.int32)
    pc = rng.standard_normal((4, 1, 4, 8)).astype(np.float16)
    k3, _, bad = oracle.kv_append_ref(kn, kn, np.array([8, 3]), pc, pc, kv_format=oracle.PAGED_NBSD,
                                      block_size=4, block_table=bt)
    assert bad == 1
    # batch 1's position 3 is slot 3 of its first block (block 2); nothing else changes
    assert np.array_equal(k3[[0, 1, 3]], pc[[0, 1, 3]]) and np.array_equal(k3[2, 0, :3], pc[2, 0, :3])
    assert np.array_equal(k3[2, 0, 3], kn[1, 0])


def test_output_quantisation_of_nan_is_zero():
    """Reading 20: a NaN output quantises to code 0 (finite neighbours are unaffected)."""
    y = np.array([[[np.nan, 1.0, -2.0, np.nan]]])
    assert list(oracle.quantize_output_ref(y, np.array([3.0], np.float32))[0, 0]) == [0, 3, -6, 0]


def test_sfa_tnd_tokens_past_the_key_tensor_are_skipped():
    """layout_kv TND whose last prefix sum runs past KV_T (the key tensor's rows): the last
    batch's tokens at or past its remaining rows select nothing, as if their indices were -1."""
    c = _sfa(61, B=2, sparse_size=16, nvalid_lo=16, nvalid_hi=16)
    k, kr, v = _contig_kv(c, kv_len=64)
    kt, krt, vt = (np.concatenate([t[0, :64], t[1, :40]]) for t in (k, kr, v))  # KV_T = 104
    idx = c.sparse_indices.copy()
    idx[1, 0, 0, :4] = [40, 41, 50, 39]  # batch 1 owns rows 64..103: tokens 40+ are past KV_T
    got = oracle.sfa_ref(c.query, c.query_rope, kt, krt, vt, idx, None, np.array([64, 124], np.int32),
                         scale=c.scale, layout_kv="TND")
    pruned = idx.copy()
    pruned[1, 0, 0, :3] = -1
    ref = oracle.sfa_ref(c.query, c.query_rope, kt, krt, vt, pruned, None, np.array([64, 104], np.int32),
                         scale=c.scale, layout_kv="TND")
    assert np.array_equal(got, ref)
