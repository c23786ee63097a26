"""GPU parity of the sparse-index MLA-absorb decode kernel (tcgen05) against the
float64 CPU oracle on the same seeded inputs.  Tolerances: max abs error <=
1.5e-2 (bf16 outputs) and <= 2e-3 (fp16 outputs); the selected-set check is
bit-exact."""
import numpy as np
import pytest

import oracle
from kv_cache_incremental_split_gb300 import inputs as gen
from harness import TOL, max_abs_err, out_to_f64, sfa_bit_probe, sfa_pieces_per_row, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_incremental_split_gb300 import build
    build.build()


def sfa_op(c, sparse_mode=None, lse=False):
    from kv_cache_incremental_split_gb300.ifa import SparseFlashAttention
    tnd = c.layout_query == "TND"
    paged = c.layout_kv == "PA_BSND"
    B = len(c.actual_seq_lengths_query) if tnd else c.query.shape[0]
    kw = dict(block_size=c.key.shape[1], block_num=c.key.shape[0], block_table_cols=c.block_table.shape[1]) \
        if paged else dict(kv_rows=c.key.shape[1] if c.layout_kv == "BSND" else c.key.shape[0])
    return SparseFlashAttention(batch=B, num_heads=c.query.shape[-2], sparse_size=c.sparse_indices.shape[-1],
                                dtype=c.dtype, scale=c.scale,
                                sparse_mode=c.sparse_mode if sparse_mode is None else sparse_mode,
                                sparse_block_size=c.sparse_block_size, q_seq_len=1 if tnd else c.query.shape[1],
                                layout_query=c.layout_query, q_total=c.query.shape[0] if tnd else 0,
                                layout_kv=c.layout_kv, return_softmax_lse=lse, **kw)


def run_gpu(c, sparse_mode=None, lse=False):
    op = sfa_op(c, sparse_mode, lse)
    t = [to_device(a) for a in (c.query, c.query_rope, c.key, c.key_rope, c.value, c.sparse_indices)]
    bt = None if c.block_table is None else to_device(c.block_table)
    lk = None if c.actual_seq_lengths_kv is None else to_device(c.actual_seq_lengths_kv)
    lq = None if c.actual_seq_lengths_query is None else to_device(c.actual_seq_lengths_query)
    res = op(*t, bt, lk, actual_seq_lengths_query=lq)
    torch.cuda.synchronize()
    out = res[0] if lse else res
    if c.layout_query == "TND":
        shape = (c.query.shape[0], c.query.shape[1], 512)
    else:
        Q_S = c.query.shape[1]
        shape = (c.B, c.query.shape[2], 512) if Q_S == 1 else (c.B, Q_S, c.query.shape[2], 512)
    got = out_to_f64(out).reshape(shape)
    if lse:
        return got, res[1].double().cpu().numpy().reshape(shape[:-1]), res[2].double().cpu().numpy().reshape(shape[:-1]), op
    return got, op


def run_ref(c, batches=None, sparse_mode=None, lse=False):
    cc = c
    if batches is not None:
        import copy
        cc = copy.copy(c)
        bs = np.asarray(batches)
        cc.query, cc.query_rope = c.query[bs], c.query_rope[bs]
        cc.sparse_indices, cc.block_table = c.sparse_indices[bs], c.block_table[bs]
        cc.actual_seq_lengths_kv = c.actual_seq_lengths_kv[bs]
        if c.actual_seq_lengths_query is not None:
            cc.actual_seq_lengths_query = c.actual_seq_lengths_query[bs]
    return oracle.sfa_ref(cc.query, cc.query_rope, cc.key, cc.key_rope, cc.value, cc.sparse_indices,
                          cc.block_table, cc.actual_seq_lengths_kv, scale=cc.scale,
                          sparse_block_size=cc.sparse_block_size,
                          sparse_mode=cc.sparse_mode if sparse_mode is None else sparse_mode,
                          actual_seq_lengths_query=cc.actual_seq_lengths_query, layout_query=cc.layout_query,
                          layout_kv=cc.layout_kv, return_softmax_lse=lse)


def check(c, batches=None, sparse_mode=None):
    got, op = run_gpu(c, sparse_mode)
    ref = run_ref(c, batches, sparse_mode)
    if batches is not None:
        got = got[np.asarray(batches)]
    assert np.all(np.isfinite(got))
    err = max_abs_err(got, ref)
    assert err <= TOL[c.dtype], err
    return got, op


@pytest.mark.parametrize("B,Q_S", [(512, 2), (1025, 1)])
def test_sfa_many_rows_both_split_paths(B, Q_S):
    """Up to 1024 query rows every decode CTA derives its share from the per-row live-tile
    counts; above that the tile-count cluster computes the prefix, the shares and the piece
    records.  1024 rows (the limit) and 1025 rows, short rows (some empty), against the oracle."""
    c = gen.sfa_mla(40 + B, B=B, Q_N=16, block_size=64, kv_len=128, sparse_size=32, nvalid_lo=0, nvalid_hi=32,
                    Q_S=Q_S)
    check(c)


@pytest.mark.parametrize("seed", [0, 1])
def test_sfa_small(seed):
    check(gen.sfa_mla(seed, B=3, Q_N=128, block_size=64, kv_len=1000, sparse_size=300, nvalid_lo=1,
                      nvalid_hi=300))


@pytest.mark.parametrize("Q_N,block_size", [(16, 16), (64, 48), (1, 1024), (100, 128)])
def test_sfa_heads_and_block_sizes(Q_N, block_size):
    check(gen.sfa_mla(2, B=2, Q_N=Q_N, block_size=block_size, kv_len=3000, sparse_size=200, nvalid_lo=50,
                      nvalid_hi=200))


def test_sfa_fp16_and_sparse_mode_3():
    c = gen.sfa_mla(3, B=2, Q_N=128, block_size=64, kv_len=800, sparse_size=130, nvalid_lo=60, nvalid_hi=130,
                    dtype="fp16")
    check(c)
    check(c, sparse_mode=3)


def test_sfa_long_rows_are_split_and_merged():
    # few batches, long index rows: sequences are cut into several pieces across CTAs
    check(gen.sfa_mla(4, B=1, Q_N=128, block_size=64, kv_len=32768, sparse_size=2048, nvalid_lo=2048,
                      nvalid_hi=2048))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_sfa_full_size_sampled(seed):
    c = gen.sfa_mla(seed)
    rng = np.random.default_rng(300 + seed)
    check(c, batches=np.sort(rng.choice(c.B, size=3, replace=False)))


@pytest.mark.parametrize("Q_S,mode", [(1, 0), (2, 3)])
def test_sfa_fp16_full_size_sampled(Q_S, mode):
    """fp16 operands and output at the sparse MLA workload's full size (rows cut across CTA pairs,
    so the merge runs), sampled batches within the fp16 bound of 2e-3."""
    c = gen.sfa_mla(14 + Q_S, Q_S=Q_S, sparse_mode=mode, dtype="fp16")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    pieces, _ = sfa_pieces_per_row(c.sparse_indices.reshape(c.B * Q_S, -1), sms)
    assert (pieces >= 2).mean() >= 0.75
    got, _ = check(c, batches=np.array([0, 9, 31]))
    assert TOL["fp16"] == 2e-3


def test_sfa_mtp_full_size_sampled():
    # the multi-token workload at full size (B=32, Q_S=2, 2048 indices per row, causal), sampled batches
    c = gen.sfa_mla(0, Q_S=2, sparse_mode=3)
    c.sparse_indices[:, :, 0, 0] = 32767  # the last key: visible to query token 1 only
    check(c, batches=np.array([0, 17, 31]))


def test_sfa_edge_rows():
    c = gen.sfa_mla(5, B=4, Q_N=32, block_size=64, kv_len=512, sparse_size=100, nvalid_lo=10, nvalid_hi=100)
    c.sparse_indices[0] = -1                      # nothing selected: zeros
    c.sparse_indices[1] = -1
    c.sparse_indices[1, 0, 0, 0] = 77             # one index: that value row
    c.sparse_indices[2, 0, 0, 5] = 600            # beyond the length, in the middle: skipped
    c.sparse_indices[3, 0, 0, :4] = [9, 9, 9, 3]  # duplicates count once per occurrence
    got, _ = check(c)
    assert np.all(got[0] == 0)


def test_sfa_selected_set_bit_exact():
    """Q = 0 and value row = code of its token: the output is exactly the mean of the
    codes of the valid selected tokens (powers-of-two counts make the mean exact)."""
    c = gen.sfa_mla(6, B=2, Q_N=128, block_size=64, kv_len=4096, sparse_size=256, nvalid_lo=256, nvalid_hi=256)
    c.query[:] = 0
    c.query_rope[:] = 0
    codes = np.zeros(c.value.shape, dtype=np.float32)
    bs = 64
    for b in range(2):
        for blk_i, blk in enumerate(c.block_table[b]):
            codes[blk, :, 0, :] = (np.arange(bs) + blk_i * bs)[:, None] % 128
    c.value = gen.to_storage(codes, "bf16")
    idx = np.full((2, 1, 1, 256), -1, dtype=np.int32)
    rng = np.random.default_rng(7)
    idx[0, 0, 0, :128] = rng.choice(4096, size=128, replace=False)
    idx[1, 0, 0, :64] = rng.choice(4096, size=64, replace=False)
    c.sparse_indices = idx
    got, _ = run_gpu(c)
    ref = run_ref(c)  # exact means (power-of-two counts), representable in float32
    ref_bf16 = gen.bf16_bits_to_f32(gen.f32_to_bf16_bits(ref.astype(np.float32))).astype(np.float64)
    assert np.array_equal(got, ref_bf16)


def test_sfa_bad_block_entry_sets_error_flag():
    c = gen.sfa_mla(8, B=2, Q_N=16, block_size=64, kv_len=640, sparse_size=64, nvalid_lo=64, nvalid_hi=64)
    c.block_table[1, :] = c.key.shape[0] + 3  # every entry of batch 1 out of range: its tokens are left out
    got, op = run_gpu(c)
    assert op.device_errors() & 1
    ref = run_ref(c)
    assert max_abs_err(got, ref) <= TOL["bf16"]
    assert np.all(got[1] == 0)


def test_sfa_deterministic():
    c = gen.sfa_mla(9, B=2, Q_N=128, block_size=64, kv_len=8192, sparse_size=2048, nvalid_lo=1500,
                    nvalid_hi=2048)
    a, _ = run_gpu(c)
    b, _ = run_gpu(c)
    assert np.array_equal(a, b)


# ---- block-wise sparsity (sparse_block_size > 1)


@pytest.mark.parametrize("sbs,block_size,sparse_size,nvalid_hi", [(2, 64, 97, 60), (8, 64, 61, 50), (16, 64, 47, 40),
                                                                   (32, 64, 21, 21), (64, 64, 13, 13), (128, 128, 7, 7)])
def test_sfa_blockwise_matches_oracle(sbs, block_size, sparse_size, nvalid_hi):
    """Each index selects sbs consecutive tokens; positions span several tiles and end ragged.  From 8
    tokens on, runs move as tiled boxes of consecutive rows (8, 4, 2 or 1 per stage), else by gathers."""
    c = gen.sfa_mla(60 + sbs, B=3, Q_N=128, block_size=block_size, kv_len=4096, sparse_size=sparse_size,
                    nvalid_lo=3, nvalid_hi=nvalid_hi, sparse_block_size=sbs)
    c.actual_seq_lengths_kv[1] = 4096 - 37  # selected blocks of batch 1 may end past its length
    check(c)


def test_sfa_blockwise_invalid_entries_and_short_rows():
    c = gen.sfa_mla(70, B=4, Q_N=64, block_size=64, kv_len=2048, sparse_size=40, nvalid_lo=1, nvalid_hi=40,
                    sparse_block_size=8)
    c.sparse_indices[2, 0, 0, :] = -1  # nothing selected: zeros
    c.sparse_indices[3, 0, 0, ::3] = -1  # -1 entries scattered through the row
    got, _ = check(c)
    assert np.all(got[2] == 0)


# ------------------------------------------- multi-token queries and the right-down causal mode

@pytest.mark.parametrize("Q_S,mode", [(2, 3), (4, 0), (3, 3)])
def test_sfa_multi_token_matches_oracle(Q_S, mode):
    c = gen.sfa_mla(20 + Q_S, B=3, Q_N=64, block_size=64, kv_len=700, sparse_size=260, nvalid_lo=100,
                    nvalid_hi=260, Q_S=Q_S, sparse_mode=mode)
    # every row selects the last keys, so the causal boundary falls inside the selection
    c.sparse_indices[:, :, 0, :4] = np.array([699, 698, 697, 696], dtype=np.int32)
    check(c)


def test_sfa_multi_token_query_lengths_and_zero_rows():
    c = gen.sfa_mla(24, B=4, Q_N=128, block_size=64, kv_len=500, sparse_size=200, nvalid_lo=150,
                    nvalid_hi=200, Q_S=4, sparse_mode=3, q_lens=[4, 2, 0, 1])
    c.actual_seq_lengths_kv = np.array([500, 300, 500, 3], dtype=np.int32)
    c.sparse_indices[:, :, 0, :3] = np.array([2, 1, 0], dtype=np.int32)
    got, _ = check(c)
    assert np.all(got[1, 2:] == 0.0) and np.all(got[2] == 0.0) and np.all(got[3, 1:] == 0.0)


def test_sfa_multi_token_long_rows_split_across_ctas():
    # 2 x 2 x 2 sequences of 32 tiles: several CTAs per sequence, merged by the combine kernel
    c = gen.sfa_mla(25, B=2, Q_N=128, block_size=64, kv_len=8192, sparse_size=2048, nvalid_lo=1800,
                    nvalid_hi=2048, Q_S=2, sparse_mode=3)
    c.sparse_indices[:, :, 0, :2] = np.array([8191, 8190], dtype=np.int32)
    check(c)


@pytest.mark.parametrize("sbs", [4, 16])
def test_sfa_multi_token_blockwise_causal(sbs):
    c = gen.sfa_mla(26, B=2, Q_N=32, block_size=64, kv_len=1024, sparse_size=40, nvalid_lo=20, nvalid_hi=40,
                    Q_S=3, sparse_mode=3, sparse_block_size=sbs, q_lens=[3, 2])
    c.actual_seq_lengths_kv = np.array([1024 - sbs // 2, 1000], dtype=np.int32)
    c.sparse_indices[:, :, 0, 0] = 1024 // sbs - 1  # the last block: partly past length and causal limit
    check(c)


# ------------------------------------------- TND / BSND layouts and softmax_max / softmax_sum

LAYOUTS = [("BSND", "BSND"), ("BSND", "TND"), ("TND", "PA_BSND"), ("TND", "BSND"), ("TND", "TND")]


@pytest.mark.parametrize("lq,lk", LAYOUTS)
def test_sfa_layouts_match_oracle(lq, lk):
    c = gen.sfa_mla(30, B=4, Q_N=64, block_size=64, kv_len=900, sparse_size=260, nvalid_lo=100, nvalid_hi=260,
                    Q_S=3, sparse_mode=3, q_lens=[3, 1, 0, 2])
    c.actual_seq_lengths_kv = np.array([900, 333, 500, 64], dtype=np.int32)
    c.sparse_indices[:, :, 0, :3] = np.array([899, 332, 63], dtype=np.int32)
    check(gen.sfa_relayout(c, lq, lk))


def test_sfa_bsnd_lengths_above_the_key_rows_skip_tokens_past_them():
    """BSND keys with a batch length above KV_S (the key tensor's rows per batch): selected tokens
    at or past KV_S select nothing and must not reach the next batch's rows.  Outputs against the
    oracle; with a zero query every score is 0, so softmax_sum is the exact count of the tokens
    that count, compared exactly."""
    c = gen.sfa_mla(36, B=3, Q_N=64, block_size=64, kv_len=512, sparse_size=256, nvalid_lo=120, nvalid_hi=256)
    c.actual_seq_lengths_kv = np.array([512, 512, 512], dtype=np.int32)
    c = gen.sfa_relayout(c, "BSND", "BSND")
    kv_s = c.key.shape[1]
    assert kv_s == 512
    c.actual_seq_lengths_kv = np.array([kv_s + 40, kv_s, kv_s - 100], dtype=np.int32)
    c.sparse_indices[0, 0, 0, :6] = [kv_s, kv_s + 1, kv_s + 17, kv_s + 39, kv_s - 1, 0]
    c.sparse_indices[1, 0, 0, :2] = [kv_s - 1, 3]
    # batch 2: every entry selects a token at or past its length, so its tiles are live but empty
    nv2 = int((c.sparse_indices[2, 0, 0] >= 0).sum())
    c.sparse_indices[2, 0, 0, :nv2] = kv_s - 100 + np.arange(nv2) % 100
    got, mx, sm, op = run_gpu(c, lse=True)
    ref, rmx, rsm = run_ref(c, lse=True)
    assert max_abs_err(got, ref) <= TOL[c.dtype]
    assert np.all(got[2] == 0) and np.all(np.isneginf(mx[2])) and np.all(sm[2] == 0)
    assert op.device_errors() == 0
    c.query = np.zeros_like(c.query)
    c.query_rope = np.zeros_like(c.query_rope)
    _, _, sm0, _ = run_gpu(c, lse=True)
    _, _, rsm0 = run_ref(c, lse=True)
    assert np.array_equal(sm0, rsm0), np.argwhere(sm0 != rsm0)[:8]


@pytest.mark.parametrize("lk", ["BSND", "TND"])
def test_sfa_contiguous_keys_blockwise_runs(lk):
    # block-wise runs of 16 tokens as tiled boxes over contiguous key rows (no cache blocks)
    c = gen.sfa_mla(31, B=3, Q_N=32, block_size=64, kv_len=1024, sparse_size=40, nvalid_lo=20, nvalid_hi=40,
                    Q_S=2, sparse_mode=3, sparse_block_size=16)
    c.actual_seq_lengths_kv = np.array([1024, 1000, 250], dtype=np.int32)
    check(gen.sfa_relayout(c, "BSND", lk))


def test_sfa_tnd_long_rows_split_across_ctas():
    c = gen.sfa_mla(32, B=2, Q_N=128, block_size=64, kv_len=8192, sparse_size=2048, nvalid_lo=1800,
                    nvalid_hi=2048, Q_S=2, sparse_mode=3, q_lens=[1, 2])
    check(gen.sfa_relayout(c, "TND", "TND"))


@pytest.mark.parametrize("lq,lk,split", [("BSND", "PA_BSND", False), ("BSND", "BSND", True), ("TND", "TND", False),
                                         ("TND", "PA_BSND", True)])
def test_sfa_softmax_max_and_sum(lq, lk, split):
    """softmax_max within 2e-3 (the scores accumulate in fp32 from 16-bit operands), softmax_sum
    within 1e-3 relative (fp32 sum of exp2 approximations); -inf and 0 on empty rows."""
    kw = dict(sparse_size=2048, nvalid_lo=1800, nvalid_hi=2048, kv_len=8192) if split else \
        dict(sparse_size=200, nvalid_lo=1, nvalid_hi=200, kv_len=700)
    c = gen.sfa_mla(33, B=3, Q_N=128, block_size=64, Q_S=2, sparse_mode=3, q_lens=[2, 0, 1], **kw)
    c = gen.sfa_relayout(c, lq, lk)
    got, mx, sm, _ = run_gpu(c, lse=True)
    ref, rmx, rsm = run_ref(c, lse=True)
    assert max_abs_err(got, ref) <= TOL[c.dtype]
    empty = np.isneginf(rmx)
    assert np.array_equal(np.isneginf(mx), empty)
    assert np.all(sm[empty] == 0.0)
    live = ~empty
    assert live.any()
    assert np.abs(mx[live] - rmx[live]).max() <= 2e-3
    assert (np.abs(sm[live] - rsm[live]) / rsm[live]).max() <= 1e-3


def test_sfa_rows_without_live_tiles_and_late_indices():
    """Rows the tile count leaves out (all -1) get zero rows, max -inf and sum 0; an index that
    follows a run of -1 (or sits alone far into the row) keeps its tile live."""
    c = gen.sfa_mla(34, B=6, Q_N=128, block_size=64, sparse_size=2048, nvalid_lo=600, nvalid_hi=1500, kv_len=4096)
    c.sparse_indices[0] = -1
    c.sparse_indices[1, 0, 0, 2040] = 123        # after the -1 tail: the last tile stays live
    c.sparse_indices[2] = -1
    c.sparse_indices[2, 0, 0, 1500] = 4000       # a single index far into the row
    c.sparse_indices[4] = -1
    got, mx, sm, _ = run_gpu(c, lse=True)
    ref, rmx, rsm = run_ref(c, lse=True)
    assert max_abs_err(got, ref) <= TOL[c.dtype]
    assert np.all(got.reshape(6, -1)[[0, 4]] == 0)
    empty = np.isneginf(rmx)
    assert np.array_equal(np.isneginf(mx), empty) and np.all(sm[empty] == 0.0)
    assert empty.reshape(6, -1)[[0, 4]].all() and not empty.reshape(6, -1)[[1, 2, 3, 5]].any()
    live = ~empty
    assert np.abs(mx[live] - rmx[live]).max() <= 2e-3
    assert (np.abs(sm[live] - rsm[live]) / rsm[live]).max() <= 1e-3


# ------------------------------------------- exact selected sets on rows cut across CTA pairs

@pytest.mark.parametrize("Q_S,mode", [(1, 0), (2, 3)])
def test_sfa_selected_set_exact_on_split_rows(Q_S, mode):
    """The sparse MLA workload's shape (B=32, 2048 indices, U{1024..2048} valid per row, keys of
    32768 tokens; two query tokens with the right-down causal mode): softmax_sum of the bit probe
    is compared exactly, on every row, with the count-based closed form, and on sampled rows with
    the oracle rounded to float32.  Rows are cut across CTA pairs (asserted from the live-tile
    split); one row is re-drawn so that its live tiles end exactly on a pair boundary, and one so
    that its valid entries end exactly on a tile boundary."""
    c = gen.sfa_mla(40 + Q_S, Q_S=Q_S, sparse_mode=mode)
    B = c.query.shape[0]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rows = c.sparse_indices.reshape(B * Q_S, -1)
    rng = np.random.default_rng(400 + Q_S)

    def redraw(r, nv):
        b, s = divmod(r, Q_S)
        c.sparse_indices[b, s, 0, :] = -1
        c.sparse_indices[b, s, 0, :nv] = rng.choice(32768, size=nv, replace=False)

    redraw(3, 1280)  # ten whole tiles
    boundary_row = None
    for r in range(5, B * Q_S):
        for nv in range(1024, 2049, 128):
            keep = c.sparse_indices.copy()
            redraw(r, nv)
            pieces, on_b = sfa_pieces_per_row(rows, sms)
            if on_b[r] and pieces[r] >= 2:
                boundary_row = r
                break
            c.sparse_indices[:] = keep
        if boundary_row is not None:
            break
    assert boundary_row is not None
    pieces, _ = sfa_pieces_per_row(rows, sms)
    assert (pieces >= 2).mean() >= 0.75, pieces

    c, exp_sum, exp_max = sfa_bit_probe(c)
    got, mx, sm, _ = run_gpu(c, lse=True)
    sm = sm.reshape(B * Q_S, -1)
    assert np.array_equal(sm, exp_sum), np.argwhere(sm != exp_sum)[:8]
    # the largest score: 0 when a selected token has the probed bit clear, else -ln 2
    mx = mx.reshape(B * Q_S, -1)
    assert np.array_equal(np.isneginf(mx), np.isneginf(exp_max))
    live = ~np.isneginf(exp_max)
    assert np.abs(mx[live] - exp_max[live]).max() <= 1e-6
    # oracle on sampled batches (the boundary row's batch among them): exact sums, tolerance elsewhere
    bsel = np.unique([boundary_row // Q_S, 3 // Q_S, B - 1])
    ref, rmx, rsm = run_ref(c, batches=bsel, lse=True)
    rows_sel = np.concatenate([np.arange(b * Q_S, (b + 1) * Q_S) for b in bsel])
    assert np.array_equal(sm[rows_sel], rsm.reshape(len(rows_sel), -1).astype(np.float32).astype(np.float64))
    assert np.abs(mx[rows_sel] - rmx.reshape(len(rows_sel), -1)).max() <= 1e-6
    assert max_abs_err(got[bsel], ref) <= TOL[c.dtype]


def test_sfa_value_aliases_key():
    """`value` may be the same tensor as `key` (one cache serves both, as in MLA-absorb decode):
    the kernel reads the value half from the key rows; checked against the oracle given the same
    array for both, on a small case with split rows and on sampled rows of the full-size shape."""
    c = gen.sfa_mla(11, B=2, Q_N=128, block_size=64, kv_len=8192, sparse_size=2048, nvalid_lo=1500,
                    nvalid_hi=2048)
    c.value = c.key
    op = sfa_op(c)
    q, qr, k, kr, idx = (to_device(a) for a in (c.query, c.query_rope, c.key, c.key_rope, c.sparse_indices))
    out = op(q, qr, k, kr, k, idx, to_device(c.block_table), to_device(c.actual_seq_lengths_kv))
    torch.cuda.synchronize()
    got = out_to_f64(out).reshape(c.B, c.query.shape[2], 512)
    ref = run_ref(c)
    assert np.all(np.isfinite(got)) and max_abs_err(got, ref) <= TOL[c.dtype]
    assert op.device_errors() == 0


def test_sfa_value_aliases_key_full_size_sampled():
    c = gen.sfa_mla(12)
    c.value = c.key
    op = sfa_op(c)
    q, qr, k, kr, idx = (to_device(a) for a in (c.query, c.query_rope, c.key, c.key_rope, c.sparse_indices))
    out = op(q, qr, k, kr, k, idx, to_device(c.block_table), to_device(c.actual_seq_lengths_kv))
    torch.cuda.synchronize()
    got = out_to_f64(out).reshape(c.B, c.query.shape[2], 512)
    bsel = np.array([0, 13, 31])
    ref = run_ref(c, batches=bsel)
    assert max_abs_err(got[bsel], ref) <= TOL[c.dtype]
