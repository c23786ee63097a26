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
 * output row is all zeros by rule (out-of-range left-pad window).
 * Left padding: IncreFlashAttention README, "kv左padding" constraints.
 */
static int resolve_window(const orc_ifa* a, int64_t b, int64_t* st, int64_t* en) {
    int64_t len;
    if (a->lens) len = a->lens[b];
    else len = a->Smax;
    if (a->pads) {
        int64_t pad = a->pads[a->n_pads == 1 ? 0 : b];
        if (pad < 0) pad = 0;
        int64_t s0 = a->Smax - pad - len;
        int64_t e0 = a->Smax - pad;
        if (s0 < 0 || e0 < 0) return 0;
        *st = s0;
        *en = e0;
        return 1;
    }
    if (len < 0) len = 0;
    if (a->kv_format == ORC_CONTIG && len > a->Smax) len = a->Smax;
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
 * Returns the number of block-table lookups that fell outside [0, blocknum)
 * (those tokens are left out of the softmax), or -1 on bad arguments.
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
    int64_t G = N / a.KV_N;
    int bad = 0;

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
                if (off0 < 0) {
                    if (n == 0) bad++;
                    continue;
                }
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
 * Sparse-index MLA-absorb decode (SparseFlashAttention README: formula in
 * "功能说明"; query/key/value/query_rope/key_rope/sparse_indices/block_table/
 * actual_seq_lengths_kv in "参数说明").  PA_BSND storage with KV_N = 1:
 *   key   (block_num, block_size, 1, D)   key_rope (block_num, block_size, 1, Dr)
 *   value (block_num, block_size, 1, D)   query (B, 1, Q_N, D), query_rope (B, 1, Q_N, Dr)
 *   sparse_indices (B, 1, 1, sparse_size), block_table (B, bt_cols)
 * s_j = scale * (q . k[idx_j] + q_rope . k_rope[idx_j]);  out = softmax(s) . v[idx_j].
 * sparse_block_size (README "sparse_block_size", 1 = token-wise): entry j of a row selects
 * the tokens idx_j * sparse_block_size + o, o = 0 .. sparse_block_size - 1 (block-wise:
 * the tokens of a block share the selection); a token at or past actual_seq_lengths_kv[b],
 * or any token of a negative entry, is skipped.
 * Q_S query tokens per batch (query (B, Q_S, Q_N, D), sparse_indices (B, Q_S, 1, sparse_size),
 * out (B, Q_S, Q_N, D)): each (b, s) row is its own problem over its own index row.
 * lens_q (nullable: every row valid) gives the valid query tokens of each batch; rows s at or
 * past it are all zero.  sparse_mode 3 (README "sparse_mode", rightDownCausal): query token s
 * sits at key position lens_kv[b] - lens_q[b] + s and selected tokens past it are skipped;
 * sparse_mode 0 masks nothing.
 * Returns the number of skipped out-of-range block-table entries, -1 on bad arguments.
 */
int sfa_oracle_run(int64_t B, int64_t Q_S, int64_t Q_N, int64_t D, int64_t Dr, int dtype, int64_t block_size,
                   int64_t block_num, int64_t bt_cols, int64_t sparse_size, int64_t sparse_block_size,
                   int64_t sparse_mode, const void* q, const void* q_rope, const void* k, const void* k_rope,
                   const void* v, const int32_t* sparse_indices, const int32_t* block_table,
                   const int32_t* lens_kv, const int32_t* lens_q, double scale, double* out) {
    if (B < 0 || Q_S <= 0 || Q_N <= 0 || D <= 0 || Dr < 0 || block_size <= 0 || sparse_size <= 0 ||
        sparse_block_size <= 0 || (sparse_mode != 0 && sparse_mode != 3))
        return -1;
    int bad = 0;
    const int64_t npos = sparse_size * sparse_block_size; /* selected token positions per row */
    double* s = (double*)malloc((size_t)npos * sizeof(double));
    int64_t* row = (int64_t*)malloc((size_t)npos * sizeof(int64_t));
    if (!s || !row) {
        free(s);
        free(row);
        return -1;
    }
    for (int64_t bs_row = 0; bs_row < B * Q_S; bs_row++) {
        const int64_t b = bs_row / Q_S, sq = bs_row % Q_S;
        const int64_t qlen = lens_q ? lens_q[b] : Q_S;
        /* keys this query row may use: [0, limit) */
        int64_t limit = lens_kv[b];
        if (sq >= qlen) limit = 0;
        else if (sparse_mode == 3) limit = lens_kv[b] - qlen + sq + 1;
        /* resolve the selected rows once per query row: physical row = blk * block_size + slot */
        for (int64_t j = 0; j < npos; j++) {
            int64_t idx = sparse_indices[bs_row * sparse_size + j / sparse_block_size];
            row[j] = -1;
            if (idx < 0) continue;
            int64_t tok = idx * sparse_block_size + j % sparse_block_size;
            if (tok >= lens_kv[b] || tok >= limit) continue;
            int64_t blk = block_table[b * bt_cols + tok / block_size];
            if (blk < 0 || blk >= block_num) {
                bad++;
                continue;
            }
            row[j] = blk * block_size + tok % block_size;
        }
        for (int64_t n = 0; n < Q_N; n++) {
            double* o = out + (bs_row * Q_N + n) * D;
            for (int64_t d = 0; d < D; d++) o[d] = 0.0;
            double smax = -INFINITY;
            int any = 0;
            for (int64_t j = 0; j < npos; j++) {
                if (row[j] < 0) continue;
                double dot = 0.0;
                for (int64_t d = 0; d < D; d++)
                    dot += load_value(q, (bs_row * Q_N + n) * D + d, dtype) * load_value(k, row[j] * D + d, dtype);
                for (int64_t d = 0; d < Dr; d++)
                    dot += load_value(q_rope, (bs_row * Q_N + n) * Dr + d, dtype) *
                           load_value(k_rope, row[j] * Dr + d, dtype);
                s[j] = scale * dot;
                if (s[j] > smax) smax = s[j];
                any = 1;
            }
            if (!any) continue;
            double denom = 0.0;
            for (int64_t j = 0; j < npos; j++) {
                if (row[j] < 0) continue;
                double w = exp(s[j] - smax);
                denom += w;
                for (int64_t d = 0; d < D; d++) o[d] += w * load_value(v, row[j] * D + d, dtype);
            }
            for (int64_t d = 0; d < D; d++) o[d] /= denom;
        }
    }
    free(s);
    free(row);
    return bad;
}
