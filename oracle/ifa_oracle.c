/*
 * CPU oracle for incremental (single-query decode) flash attention and for
 * sparse-index MLA-absorb decode.  TEST INFRASTRUCTURE ONLY: the tests, the
 * smoke check and the benchmark's CPU-baseline leg load this file's shared
 * library; the product path never does.
 *
 * Everything here is the plain definition, evaluated in double precision with
 * no blocking, fusion or reordering:
 *
 *   out[b, n, :] = sum_t exp(s_t - max s) * v[t, :] / sum_t exp(s_t - max s)
 *   s_t          = scaleValue * sum_d q[b, n, d] * k[t, d]
 *
 * over the valid token set T_b of batch b (IncreFlashAttention README,
 * "功能说明" formula; aclnnIncreFlashAttentionV2, "Function" formula and the
 * scaleValue parameter).  The sparse variant is the same softmax over the
 * rows that sparse_indices selects (SparseFlashAttention README, "功能说明").
 *
 * Readings of points the pages leave open (each is a deliberate choice):
 *  - GQA: query head n uses key/value head n / (numHeads / numKeyValueHeads).
 *  - attenMask: a nonzero byte EXCLUDES the position; the mask is indexed in
 *    the key/value S coordinate (absolute position under left padding).
 *  - an empty surviving set (length 0, out-of-range left-pad window, all
 *    masked, all sparse indices invalid) gives an all-zero output row.
 *  - antiquant: xhat = (x + offset) * scale, index 0 of the leading axis is
 *    for key, 1 for value; per-channel tensors are (2, KV_N, D) in memory.
 *  - sparse indices outside [0, actual_seq_lengths_kv[b]) are skipped;
 *    duplicates count once per occurrence.
 *  - lengths: negative, or (right padding, paging) above the cache's S or
 *    blockTableCols * blockSize, are refused; kvPaddingSize applies only with
 *    actualSeqLengths; a paged cache takes no left padding.
 *
 * No code, header or table is shared with the CUDA path.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* dtype codes used by this file's entry points */
#define ORC_F16 0
#define ORC_BF16 1
#define ORC_I8 2

/* layout codes (aclnnIncreFlashAttentionV2, inputLayout parameter) */
#define ORC_BSH 0
#define ORC_BSND 1
#define ORC_BNSD 2

/* key/value storage (IncreFlashAttention README, page attention constraints) */
#define ORC_CONTIG 0
#define ORC_PAGED_NBSD 1 /* (blocknum, KV_N, blockSize, D) */
#define ORC_PAGED_BSH 2  /* (blocknum, blockSize, H) */

/* antiquant modes (IncreFlashAttention README, antiquant constraints) */
#define ORC_AQ_NONE 0
#define ORC_AQ_PER_CHANNEL 1
#define ORC_AQ_PER_TENSOR 2

/* IEEE binary16 -> double, from the format's definition. */
static double half_bits_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -24);
    } else if (e == 31) {
        v = (m == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + m), e - 25);
    }
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32. */
static double bf16_bits_to_double(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double load_value(const void* base, int64_t idx, int dtype) {
    if (dtype == ORC_F16) return half_bits_to_double(((const uint16_t*)base)[idx]);
    if (dtype == ORC_BF16) return bf16_bits_to_double(((const uint16_t*)base)[idx]);
    return (double)((const int8_t*)base)[idx];
}

typedef struct {
    int64_t B, N, KV_N, D;
    int q_dtype, kv_dtype, layout, kv_format;
    int64_t Smax;
    int64_t block_size, block_table_cols, block_num;
    const void *q, *k, *v;
    const uint8_t* mask;
    int64_t maskB, maskN, maskS;
    const int64_t* lens;
    const int64_t* pads;
    int64_t n_pads;
    const int32_t* block_table;
    int antiquant;
    const void *aq_scale, *aq_offset;
    double scale;
} orc_ifa;

/* Element offset of query element (b, n, d); S_q = 1 in every layout. */
static int64_t q_offset(const orc_ifa* a, int64_t b, int64_t n, int64_t d) {
    switch (a->layout) {
    case ORC_BNSD: return ((b * a->N + n) * 1 + 0) * a->D + d;       /* (B, N, 1, D) */
    case ORC_BSND: return ((b * 1 + 0) * a->N + n) * a->D + d;       /* (B, 1, N, D) */
    default:       return (b * 1 + 0) * (a->N * a->D) + n * a->D + d; /* (B, 1, H)   */
    }
}

/*
 * Element offset of key/value element (b, h, t, d), t in the buffer's S
 * coordinate (logical token index when paged).  Returns -1 for a block-table
 * entry outside [0, blocknum).
 */
static int64_t kv_offset(const orc_ifa* a, int64_t b, int64_t h, int64_t t, int64_t d) {
    if (a->kv_format == ORC_CONTIG) {
        if (a->layout == ORC_BNSD) return ((b * a->KV_N + h) * a->Smax + t) * a->D + d;
        return ((b * a->Smax + t) * a->KV_N + h) * a->D + d; /* BSND and BSH */
    }
    int64_t blk = a->block_table[b * a->block_table_cols + t / a->block_size];
    int64_t slot = t % a->block_size;
    if (blk < 0 || blk >= a->block_num) return -1;
    if (a->kv_format == ORC_PAGED_NBSD) return ((blk * a->KV_N + h) * a->block_size + slot) * a->D + d;
    return ((blk * a->block_size + slot) * a->KV_N + h) * a->D + d; /* (blocknum, bs, H) */
}

/* Dequantised key (which = 0) or value (which = 1) element. */
static double kv_value(const orc_ifa* a, int which, int64_t off, int64_t h, int64_t d) {
    const void* base = which == 0 ? a->k : a->v;
    double x = load_value(base, off, a->kv_dtype);
    if (a->antiquant == ORC_AQ_NONE) return x;
    int64_t pidx;
    if (a->antiquant == ORC_AQ_PER_TENSOR) pidx = which;
    else pidx = (which * a->KV_N + h) * a->D + d;
    double s = load_value(a->aq_scale, pidx, a->q_dtype);
    double o = load_value(a->aq_offset, pidx, a->q_dtype);
    return (x + o) * s;
}

/*
 * Valid window [*st, *en) of batch b in the S coordinate.  Returns 0 when the
 * output row is all zeros by rule (out-of-range left-pad window), -1 for a
 * length the cache cannot hold: negative, or, without left padding, above the
 * cache's S (contiguous) or above blockTableCols * blockSize (paged) -- a batch's
 * valid tokens are tokens of its cache (aclnnIncreFlashAttentionV2,
 * actualSeqLengths; IncreFlashAttention README, page attention: the block table
 * holds every block a sequence uses).
 * Left padding: IncreFlashAttention README, "kv左padding" constraints.
 */
static int resolve_window(const orc_ifa* a, int64_t b, int64_t* st, int64_t* en) {
    int64_t len;
    if (a->lens) len = a->lens[b];
    else len = a->Smax;
    if (len < 0) return -1;
    if (a->pads && a->lens) { /* without lengths the window is right padded */
        int64_t pad = a->pads[a->n_pads == 1 ? 0 : b];
        if (pad < 0) pad = 0;
        int64_t s0 = a->Smax - pad - len;
        int64_t e0 = a->Smax - pad;
        if (s0 < 0 || e0 < 0) return 0;
        *st = s0;
        *en = e0;
        return 1;
    }
    const int64_t cap = a->kv_format == ORC_CONTIG ? a->Smax : a->block_table_cols * a->block_size;
    if (len > cap) return -1;
    *st = 0;
    *en = len;
    return 1;
}

static int masked(const orc_ifa* a, int64_t b, int64_t n, int64_t t) {
    if (!a->mask) return 0;
    int64_t mb = a->maskB > 1 ? b : 0;
    int64_t mn = a->maskN > 1 ? n : 0;
    return a->mask[((mb * a->maskN + mn) * 1 + 0) * a->maskS + t] != 0;
}

/*
 * Returns the number of tokens of the batches' windows whose block-table entry lies
 * outside [0, blocknum) (those tokens are left out of the softmax of every head),
 * or -1 on bad arguments.
 */
int ifa_oracle_run(int64_t B, int64_t N, int64_t KV_N, int64_t D, int q_dtype, int kv_dtype,
                   int layout, int kv_format, int64_t Smax, int64_t block_size,
                   int64_t block_table_cols, int64_t block_num, const void* q, const void* k,
                   const void* v, const uint8_t* mask, int64_t maskB, int64_t maskN, int64_t maskS,
                   const int64_t* lens, const int64_t* pads, int64_t n_pads,
                   const int32_t* block_table, int antiquant, const void* aq_scale,
                   const void* aq_offset, double scale, double* out) {
    orc_ifa a;
    a.B = B; a.N = N; a.KV_N = KV_N == 0 ? N : KV_N; a.D = D;
    a.q_dtype = q_dtype; a.kv_dtype = kv_dtype; a.layout = layout; a.kv_format = kv_format;
    a.Smax = Smax; a.block_size = block_size; a.block_table_cols = block_table_cols;
    a.block_num = block_num;
    a.q = q; a.k = k; a.v = v;
    a.mask = mask; a.maskB = maskB; a.maskN = maskN; a.maskS = maskS;
    a.lens = lens; a.pads = pads; a.n_pads = n_pads; a.block_table = block_table;
    a.antiquant = antiquant; a.aq_scale = aq_scale; a.aq_offset = aq_offset;
    a.scale = scale;
    if (a.KV_N <= 0 || N % a.KV_N != 0) return -1;
    if (kv_format != ORC_CONTIG && (!lens || !block_table || block_size <= 0)) return -1;
    if (kv_format != ORC_CONTIG && pads) return -1; /* left padding of a paged cache is not defined */
    int64_t G = N / a.KV_N;
    int bad = 0;

    for (int64_t b = 0; b < B; b++) {
        int64_t st = 0, en = 0;
        const int live = resolve_window(&a, b, &st, &en);
        if (live < 0) return -1;
        for (int64_t t = st; live && t < en; t++)
            if (kv_offset(&a, b, 0, t, 0) < 0) bad++;
    }
    double* s = NULL;
    int64_t cap = 0;
    for (int64_t b = 0; b < B; b++) {
        int64_t st = 0, en = 0;
        int live = resolve_window(&a, b, &st, &en);
        for (int64_t n = 0; n < N; n++) {
            double* o = out + (b * N + n) * D;
            for (int64_t d = 0; d < D; d++) o[d] = 0.0;
            if (!live || en <= st) continue;
            int64_t h = n / G;
            if (en - st > cap) {
                cap = en - st;
                free(s);
                s = (double*)malloc((size_t)cap * sizeof(double));
                if (!s) return -1;
            }
            /* pass 1: scores of the surviving tokens and their maximum */
            double smax = -INFINITY;
            int any = 0;
            for (int64_t t = st; t < en; t++) {
                double* sc = &s[t - st];
                *sc = NAN;
                if (masked(&a, b, n, t)) continue;
                int64_t off0 = kv_offset(&a, b, h, t, 0);
                if (off0 < 0) continue; /* counted above */
                double dot = 0.0;
                for (int64_t d = 0; d < D; d++)
                    dot += load_value(q, q_offset(&a, b, n, d), q_dtype) * kv_value(&a, 0, off0 + d, h, d);
                *sc = scale * dot;
                if (*sc > smax) smax = *sc;
                any = 1;
            }
            if (!any) continue;
            /* pass 2: exponentials, their sum, and the weighted sum of values */
            double denom = 0.0;
            for (int64_t t = st; t < en; t++) {
                double sc = s[t - st];
                if (isnan(sc)) continue;
                double w = exp(sc - smax);
                denom += w;
                int64_t off0 = kv_offset(&a, b, h, t, 0);
                for (int64_t d = 0; d < D; d++) o[d] += w * kv_value(&a, 1, off0 + d, h, d);
            }
            for (int64_t d = 0; d < D; d++) o[d] /= denom;
        }
    }
    free(s);
    return bad;
}

/*
 * int8 output quantisation (IncreFlashAttention README: int8 output with quantScale2 and the
 * optional quantOffset2, per-tensor or per-channel, FLOAT32 or BFLOAT16; the formula is not
 * on the pages).  Reading: code = saturate(rint(y * scale2 + offset2)) to [-128, 127], ties
 * to even, NaN -> 0, with the product and the sum each rounded to single precision (no fused
 * multiply-add), y the attention output rounded to single precision.  Per channel, element
 * (b, n, d) of the (B, N, D) output uses entry n * D + d (N query heads: the README's
 * N * D, which also equals H for BSH); per tensor, entry 0.  offset2 NULL means 0.
 * q2_dtype: 3 = FLOAT32, 1 = BFLOAT16.  Returns -1 on bad arguments.
 */
int ifa_quantize_output(int64_t B, int64_t N, int64_t D, const double* y, int per_channel, int q2_dtype,
                        const void* scale2, const void* offset2, int8_t* out) {
    if (B < 0 || N <= 0 || D <= 0 || !y || !scale2 || !out || (q2_dtype != 3 && q2_dtype != ORC_BF16)) return -1;
    for (int64_t b = 0; b < B; b++) {
        for (int64_t c = 0; c < N * D; c++) {
            const int64_t pi = per_channel ? c : 0;
            float sf, of = 0.0f;
            if (q2_dtype == 3) {
                sf = ((const float*)scale2)[pi];
                if (offset2) of = ((const float*)offset2)[pi];
            } else {
                sf = (float)bf16_bits_to_double(((const uint16_t*)scale2)[pi]);
                if (offset2) of = (float)bf16_bits_to_double(((const uint16_t*)offset2)[pi]);
            }
            const float yf = (float)y[b * N * D + c];
            const float t = yf * sf;
            const float u = t + of;
            int8_t code = 0;
            if (!isnan(u)) {
                float r = rintf(u);
                if (r > 127.0f) r = 127.0f;
                if (r < -128.0f) r = -128.0f;
                code = (int8_t)r;
            }
            out[b * N * D + c] = code;
        }
    }
    return 0;
}

/*
 * int8 code of x read back as (code + offset) * scale: the inverse of the antiquant reading,
 * taken in single precision (x, scale and offset are 16-bit values, exact in float):
 * rint(x / scale - offset), ties to even, saturated to [-128, 127]; NaN gives 0.
 */
static int8_t quantize_i8(double x, double scale, double offset) {
    const float xf = (float)x, sf = (float)scale, of = (float)offset;
    const float t = xf / sf;
    const float u = t - of;
    if (isnan(u)) return 0;
    float r = rintf(u);
    if (r > 127.0f) r = 127.0f;
    if (r < -128.0f) r = -128.0f;
    return (int8_t)r;
}

/*
 * KV-cache append: the cache grows by one token per decode step (IncreFlashAttention README,
 * incremental inference; aclnnIncreFlashAttentionV2, the key/value cache arguments).  The key
 * and value rows of the new token of every batch, (B, KV_N, D) in memory in any query-style
 * layout (S = 1), are written at token position pos[b] of the cache: contiguous BNSD, BSND or
 * BSH with Smax rows per batch, or paged through the block table (block
 * block_table[b][pos / block_size], slot pos % block_size) in the NBSD or BSH block format --
 * the addresses the attention reads.  A 16-bit cache receives the values unchanged; an int8
 * cache receives quantize_i8 of each element with the antiquant parameter it is read back
 * with (per channel: entry (0 key | 1 value, h, d); per tensor: entry 0 | 1).  A position
 * outside the cache (negative, >= Smax, past the block table, or a block id outside
 * [0, blocknum)) writes nothing for that batch.
 * Returns the number of batches skipped, -1 on bad arguments.
 */
int kv_append_oracle(int64_t B, int64_t KV_N, int64_t D, int new_dtype, int kv_dtype, int layout, int kv_format,
                     int64_t Smax, int64_t block_size, int64_t block_table_cols, int64_t block_num,
                     const void* k_new, const void* v_new, const int64_t* pos, const int32_t* block_table,
                     int antiquant, const void* aq_scale, const void* aq_offset, void* k_cache, void* v_cache) {
    if (B < 0 || KV_N <= 0 || D <= 0 || !pos) return -1;
    if (kv_format != ORC_CONTIG && (!block_table || block_size <= 0)) return -1;
    if ((kv_dtype == ORC_I8) != (antiquant != ORC_AQ_NONE)) return -1;
    if (kv_dtype != ORC_I8 && kv_dtype != new_dtype) return -1;
    orc_ifa a;
    memset(&a, 0, sizeof a);
    a.B = B; a.N = KV_N; a.KV_N = KV_N; a.D = D;
    a.q_dtype = new_dtype; a.kv_dtype = kv_dtype; a.layout = layout; a.kv_format = kv_format;
    a.Smax = Smax; a.block_size = block_size; a.block_table_cols = block_table_cols; a.block_num = block_num;
    a.block_table = block_table;
    int skipped = 0;
    for (int64_t b = 0; b < B; b++) {
        const int64_t t = pos[b];
        int ok = t >= 0;
        if (ok && kv_format == ORC_CONTIG) ok = t < Smax;
        if (ok && kv_format != ORC_CONTIG) ok = t / block_size < block_table_cols;
        if (ok && kv_offset(&a, b, 0, t, 0) < 0) ok = 0; /* block id outside [0, blocknum) */
        if (!ok) {
            skipped++;
            continue;
        }
        for (int64_t h = 0; h < KV_N; h++) {
            for (int64_t d = 0; d < D; d++) {
                const int64_t src = (b * KV_N + h) * D + d;
                const int64_t dst = kv_offset(&a, b, h, t, d);
                for (int which = 0; which < 2; which++) {
                    const void* from = which == 0 ? k_new : v_new;
                    void* to = which == 0 ? k_cache : v_cache;
                    if (kv_dtype == ORC_I8) {
                        const int64_t pidx = antiquant == ORC_AQ_PER_TENSOR ? which : (which * KV_N + h) * D + d;
                        ((int8_t*)to)[dst] = quantize_i8(load_value(from, src, new_dtype),
                                                         load_value(aq_scale, pidx, new_dtype),
                                                         load_value(aq_offset, pidx, new_dtype));
                    } else {
                        ((uint16_t*)to)[dst] = ((const uint16_t*)from)[src];
                    }
                }
            }
        }
    }
    return skipped;
}

/*
 * Sparse-index MLA-absorb decode (SparseFlashAttention README: formula in
 * "功能说明"; query/key/value/query_rope/key_rope/sparse_indices/block_table/
 * actual_seq_lengths_query/actual_seq_lengths_kv/layout_query/layout_kv in "参数说明").
 * KV_N = 1 throughout.
 *
 * Query rows.  layout_query BSND: query (B, Q_S, Q_N, D), query_rope (B, Q_S, Q_N, Dr),
 * sparse_indices (B, Q_S, 1, sparse_size), out (B, Q_S, Q_N, D): row r = b * Q_S + s, and
 * lens_q (nullable) gives each batch's valid query tokens qlen (Q_S when NULL).  layout_query
 * TND: the same arrays with Q_T rows in place of (B, Q_S); lens_q (required) holds prefix
 * sums, so batch b owns rows [lens_q[b-1], lens_q[b]) (lens_q[-1] = 0), s counts from the
 * batch's first row and qlen = lens_q[b] - lens_q[b-1]; rows past lens_q[B-1] belong to no
 * batch and are zero.
 * Key rows.  layout_kv PA_BSND: key/value (block_num, block_size, 1, D), key_rope (..., Dr);
 * token t of batch b is row block_table[b][t / block_size] * block_size + t % block_size and
 * len = lens_kv[b].  BSND: key (B, KV_S, 1, D); token t is row b * KV_S + t and len =
 * lens_kv[b] (KV_S when lens_kv is NULL).  TND: key (KV_T, 1, D); lens_kv holds prefix sums,
 * token t of batch b is row lens_kv[b-1] + t and len = lens_kv[b] - lens_kv[b-1].  Tokens
 * past the batch's rows in the key tensor (t >= KV_S; row >= KV_T) are skipped.
 * Selection.  Entry j of a row's indices selects tokens idx_j * sparse_block_size + o,
 * o = 0 .. sparse_block_size - 1 (README "sparse_block_size"; 1 = token-wise); a negative
 * entry selects nothing; a token at or past len is skipped; duplicates count once per
 * occurrence.  Rows s >= qlen select nothing.  sparse_mode 3 (README "sparse_mode",
 * rightDownCausal): row s sees only tokens below len - qlen + s + 1; sparse_mode 0 masks
 * nothing.
 * s_j = scale * (q . k[j] + q_rope . k_rope[j]);  out = softmax(s) . v (zero when nothing
 * survives).  softmax_max / softmax_sum (nullable, one value per (row, head) at r * Q_N + n,
 * i.e. the README's (B, 1, Q_S, Q_N) or (1, Q_T, Q_N)): the largest s_j, and the sum of
 * exp(s_j - softmax_max); -inf and 0 when nothing survives.
 * Returns the number of skipped out-of-range block-table entries, -1 on bad arguments.
 */
typedef struct {
    int64_t B, Q_S, Q_T, Q_N, D, Dr;
    int64_t layout_q;  /* 0 BSND, 1 TND */
    int64_t layout_kv; /* 0 PA_BSND, 1 BSND, 2 TND */
    int64_t kv_s;      /* BSND: KV_S; TND: KV_T; PA_BSND: unused */
    int64_t block_size, block_num, bt_cols;
    int64_t sparse_size, sparse_block_size, sparse_mode, dtype;
    double scale;
    const void *q, *q_rope, *k, *k_rope, *v;
    const int32_t *indices, *block_table, *lens_kv, *lens_q;
    double *out, *softmax_max, *softmax_sum;
} orc_sfa;

int sfa_oracle_run(const orc_sfa* a) {
    if (a->B < 0 || a->Q_N <= 0 || a->D <= 0 || a->Dr < 0 || a->sparse_size <= 0 || a->sparse_block_size <= 0 ||
        (a->sparse_mode != 0 && a->sparse_mode != 3) || a->layout_q < 0 || a->layout_q > 1 || a->layout_kv < 0 ||
        a->layout_kv > 2)
        return -1;
    if (a->layout_q == 0 && a->Q_S <= 0) return -1;
    if (a->layout_q == 1 && (a->Q_T < 0 || !a->lens_q)) return -1;
    if (a->layout_kv == 0 && (a->block_size <= 0 || !a->block_table || !a->lens_kv)) return -1;
    if (a->layout_kv == 2 && !a->lens_kv) return -1;
    const int64_t R = a->layout_q == 0 ? a->B * a->Q_S : a->Q_T;
    const int64_t npos = a->sparse_size * a->sparse_block_size; /* selected token positions per row */
    int bad = 0;
    double* s = (double*)malloc((size_t)(npos > 0 ? npos : 1) * sizeof(double));
    int64_t* row = (int64_t*)malloc((size_t)(npos > 0 ? npos : 1) * sizeof(int64_t));
    if (!s || !row) {
        free(s);
        free(row);
        return -1;
    }
    for (int64_t r = 0; r < R; r++) {
        /* the row's batch b, query token sq and the batch's valid query tokens qlen */
        int64_t b = -1, sq = 0, qlen = 0;
        if (a->layout_q == 0) {
            b = r / a->Q_S;
            sq = r % a->Q_S;
            qlen = a->lens_q ? a->lens_q[b] : a->Q_S;
        } else {
            for (int64_t bb = 0; bb < a->B; bb++) {
                if (r < a->lens_q[bb]) {
                    b = bb;
                    break;
                }
            }
            if (b >= 0) {
                const int64_t first = b > 0 ? a->lens_q[b - 1] : 0;
                sq = r - first;
                qlen = a->lens_q[b] - first;
            }
        }
        /* the batch's keys: length, first row (BSND, TND), and the rows the key tensor holds */
        int64_t len = 0, base = 0, avail = INT64_MAX;
        if (b >= 0) {
            if (a->layout_kv == 0) {
                len = a->lens_kv[b];
            } else if (a->layout_kv == 1) {
                len = a->lens_kv ? a->lens_kv[b] : a->kv_s;
                base = b * a->kv_s;
                avail = a->kv_s;
            } else {
                base = b > 0 ? a->lens_kv[b - 1] : 0;
                len = a->lens_kv[b] - base;
                avail = a->kv_s - base;
            }
        }
        /* keys this query row may use: [0, limit) */
        int64_t limit = len;
        if (b < 0 || sq >= qlen) limit = 0;
        else if (a->sparse_mode == 3) limit = len - qlen + sq + 1;
        if (limit > len) limit = len;
        if (limit > avail) limit = avail;
        for (int64_t j = 0; j < npos; j++) {
            const int64_t idx = a->indices[r * a->sparse_size + j / a->sparse_block_size];
            row[j] = -1;
            if (idx < 0) continue;
            const int64_t tok = idx * a->sparse_block_size + j % a->sparse_block_size;
            if (tok >= limit) continue;
            if (a->layout_kv == 0) {
                const int64_t blk = a->block_table[b * a->bt_cols + tok / a->block_size];
                if (blk < 0 || blk >= a->block_num) {
                    bad++;
                    continue;
                }
                row[j] = blk * a->block_size + tok % a->block_size;
            } else {
                row[j] = base + tok;
            }
        }
        for (int64_t n = 0; n < a->Q_N; n++) {
            double* o = a->out + (r * a->Q_N + n) * a->D;
            for (int64_t d = 0; d < a->D; d++) o[d] = 0.0;
            double smax = -INFINITY;
            int any = 0;
            for (int64_t j = 0; j < npos; j++) {
                if (row[j] < 0) continue;
                double dot = 0.0;
                for (int64_t d = 0; d < a->D; d++)
                    dot += load_value(a->q, (r * a->Q_N + n) * a->D + d, (int)a->dtype) *
                           load_value(a->k, row[j] * a->D + d, (int)a->dtype);
                for (int64_t d = 0; d < a->Dr; d++)
                    dot += load_value(a->q_rope, (r * a->Q_N + n) * a->Dr + d, (int)a->dtype) *
                           load_value(a->k_rope, row[j] * a->Dr + d, (int)a->dtype);
                s[j] = a->scale * dot;
                if (s[j] > smax) smax = s[j];
                any = 1;
            }
            double denom = 0.0;
            if (any) {
                for (int64_t j = 0; j < npos; j++) {
                    if (row[j] < 0) continue;
                    const double w = exp(s[j] - smax);
                    denom += w;
                    for (int64_t d = 0; d < a->D; d++) o[d] += w * load_value(a->v, row[j] * a->D + d, (int)a->dtype);
                }
                for (int64_t d = 0; d < a->D; d++) o[d] /= denom;
            }
            if (a->softmax_max) a->softmax_max[r * a->Q_N + n] = smax;
            if (a->softmax_sum) a->softmax_sum[r * a->Q_N + n] = denom;
        }
    }
    free(s);
    free(row);
    return bad;
}
