/*
 * ifa.h -- C ABI of the GB300 (sm_103a) incremental flash attention library.
 *
 * Single-query decode attention
 *
 *     attentionOut[b, n, :] = softmax(scaleValue * q[b, n, :] . K_b^T) . V_b
 *
 * over the valid key/value tokens of batch b, with GQA (query head n reads
 * key/value head n / (numHeads / numKeyValueHeads)), per-batch
 * actualSeqLengths, an optional attenMask, key/value left padding
 * (kvPaddingSize), a paged cache addressed through blockTable/blockSize, and
 * int8 key/value "antiquant" with per-channel or per-tensor scale and offset.
 *
 * Sources (titles of the pages that define the operation):
 *  - "IncreFlashAttention" README: 功能说明 (function and formula), 约束说明
 *    (constraints: GQA multiple, page attention, kv左padding, antiquant shapes).
 *  - "aclnnIncreFlashAttentionV2": Function (formula), Function Prototype
 *    (two-phase workspace/run API), Parameters (query/key/value/attenMask/
 *    actualSeqLengths/numHeads/scaleValue/inputLayout/numKeyValueHeads),
 *    Return Value (error codes), Constraints (S_q = 1, determinism).
 *
 * Readings of points the pages leave open:
 *  - a nonzero attenMask byte EXCLUDES its position; the mask is indexed in
 *    the key/value S coordinate (absolute position under left padding);
 *  - an empty set of surviving tokens gives an all-zero output row;
 *  - antiquant dequantises x as (x + offset) * scale; entry 0 of the leading
 *    axis of scale/offset is for key, entry 1 for value;
 *  - kvPaddingSize is int64 with 1 (broadcast) or B entries.
 *
 * Calling model (mirrors the two-phase API of the aclnnIncreFlashAttentionV2
 * page): ifa_create validates the static problem description and returns a
 * plan plus the workspace size; ifa_run validates the per-call data and
 * enqueues the computation on the caller's stream (asynchronous); the caller
 * owns every tensor, the workspace and the stream.  Results are deterministic:
 * the same inputs give bitwise-identical outputs.
 *
 * Devices: every call works on the device current on the calling thread.  A plan's
 * device state lives on the device current at ifa_create, so run a plan with that
 * device current.  One process may use several devices (device indices below 64): the
 * kernels' launch attributes are set on each device's first call.
 *
 * Errors: no exception or abort crosses this ABI.  Return codes follow the
 * aclnnIncreFlashAttentionV2 page's Return Value table.
 */
#ifndef IFA_H
#define IFA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t ifa_status;
#define IFA_OK 0
#define IFA_ERR_PARAM_NULLPTR 161001 /* a required pointer is NULL */
#define IFA_ERR_PARAM_INVALID 161002 /* dtype/layout/shape/value outside the supported range */
#define IFA_ERR_RUNTIME 361001       /* a CUDA runtime call failed */

/* Layout of query / attentionOut (and of a contiguous key/value cache). */
typedef enum { IFA_LAYOUT_BSH = 0, IFA_LAYOUT_BSND = 1, IFA_LAYOUT_BNSD = 2 } ifa_layout;

/* Key/value storage.  CONTIG: (B,S,H) / (B,S,KV_N,D) / (B,KV_N,S,D) per
 * inputLayout.  PAGED_NBSD: (blockNum, KV_N, blockSize, D), only with a BNSD
 * query.  PAGED_BSH: (blockNum, blockSize, KV_N*D), any query layout.
 * ("IncreFlashAttention" README, page attention constraints.)  TENSORLIST: one
 * tensor per batch (the README's non-contiguous case): (1,S_b,H) / (1,S_b,KV_N,D) /
 * (1,KV_N,S_b,D), S_b the only extent that differs, B <= 256; run with
 * ifa_run_tensorlist. */
typedef enum { IFA_KV_CONTIG = 0, IFA_KV_PAGED_NBSD = 1, IFA_KV_PAGED_BSH = 2, IFA_KV_TENSORLIST = 3 } ifa_kv_format;

typedef enum { IFA_F16 = 0, IFA_BF16 = 1, IFA_I8 = 2, IFA_U8 = 3, IFA_BOOL = 4, IFA_F32 = 5 } ifa_dtype;

typedef enum {
    IFA_ANTIQUANT_NONE = 0,
    IFA_ANTIQUANT_PER_CHANNEL = 1, /* scale/offset memory (2, KV_N, D): (2,N,1,D), (2,N,D) or (2,H) */
    IFA_ANTIQUANT_PER_TENSOR = 2   /* scale/offset of shape (2) */
} ifa_antiquant;

/*
 * Static description of one decode-attention problem (sizes and options).
 * All int32 fields hold the enum values above.
 */
typedef struct ifa_params {
    int64_t B;                /* batch, 0..65536 */
    int64_t numHeads;         /* query heads N, 1..256 */
    int64_t numKeyValueHeads; /* key/value heads; 0 means numHeads; numHeads % it == 0 */
    int64_t headDim;          /* D, 1..512; a multiple of 8 (fp16/bf16 key/value) or 16 (int8) */
    int64_t maxSeqLen;        /* CONTIG: the key/value S extent (Smax); TENSORLIST: the largest S_b; ignored when paged */
    int32_t q_dtype;          /* IFA_F16 | IFA_BF16; attentionOut has this dtype */
    int32_t kv_dtype;         /* = q_dtype, or IFA_I8 (requires antiquant) */
    int32_t inputLayout;      /* ifa_layout */
    int32_t kvFormat;         /* ifa_kv_format */
    int64_t blockSize;        /* paged: tokens per block, <= 512, multiple of 16 (32 for int8) */
    int64_t blockNum;         /* paged: physical blocks in the cache */
    int64_t blockTableCols;   /* paged: second dimension of blockTable */
    int32_t has_mask;         /* 1 if attenMask is passed */
    int32_t mask_dtype;       /* IFA_BOOL | IFA_I8 | IFA_U8 (values 0 or 1; nonzero excludes) */
    int64_t maskB;            /* attenMask shape (maskB, maskN, 1, maskS): maskB in {1, B} */
    int64_t maskN;            /* maskN in {1, numHeads} (query heads) */
    int64_t maskS;            /* >= every valid window end */
    int32_t antiquant;        /* ifa_antiquant; not NONE exactly when kv_dtype is IFA_I8 */
    int32_t has_kv_padding;   /* 1 if kvPaddingSize is passed (left padding; contiguous only) */
    double scaleValue;        /* the scale applied to q . k (typically 1/sqrt(D)) */
    int64_t splitTiles;       /* 0: automatic split plan; > 0: at most this many 64-token tiles per
                                 CTA (testing split invariance); negative is invalid */
    /* Output quantisation ("IncreFlashAttention" README: int8 output with quantScale2 and the
     * optional quantOffset2; the formula is not on the pages).  With out_dtype IFA_I8 each
     * output element y becomes saturate(rint(y * scale2 + offset2)) in [-128, 127], the
     * product and the sum rounded to single precision, ties to even (NaN gives 0); an
     * all-zero row quantises y = 0.  Per channel, output element (n, d) takes entry
     * n * headDim + d of numHeads * headDim (the README's N * D, or H); per tensor, entry 0. */
    int32_t out_dtype;        /* IFA_I8: int8 attentionOut; any other value: q_dtype */
    int32_t quant2;           /* ifa_antiquant values: PER_CHANNEL or PER_TENSOR with an int8 output, else NONE */
    int32_t quant2_dtype;     /* IFA_F32, or IFA_BF16 with a bf16 query (the README's rule) */
} ifa_params;

typedef struct ifa_plan ifa_plan;

/*
 * Phase 1: validate `params` and build a plan for the current CUDA device.
 *   plan            out: owned by the library, free with ifa_destroy
 *   workspace_bytes out: device workspace every ifa_run on this plan needs
 * Returns IFA_ERR_PARAM_NULLPTR for NULL arguments, IFA_ERR_PARAM_INVALID for a
 * description outside the supported range, IFA_ERR_RUNTIME if the device
 * cannot be queried.  Allocates the plan and a small device block: the error
 * word and the per-sequence arrival counters (zero between calls).
 */
ifa_status ifa_create(const ifa_params* params, ifa_plan** plan, size_t* workspace_bytes);

/*
 * Phase 2: enqueue one decode-attention call on `stream` (a cudaStream_t,
 * NULL for the legacy default stream).  Asynchronous; host arrays are read
 * before the call returns.
 *
 * Device pointers (16-byte aligned unless noted):
 *   query            (B,N,1,D) / (B,1,N,D) / (B,1,H) of q_dtype
 *   key, value       key/value cache per kvFormat (may alias each other)
 *   attenMask        nullable unless has_mask; 1 byte per element, any alignment
 *   blockTable       int32 (B, blockTableCols), 4-byte aligned; required when paged;
 *                    entries of blocks a batch does not reach are never read
 *   antiquantScale   per-channel (2, KV_N, D) or per-tensor (2), of q_dtype, 2-byte aligned
 *   antiquantOffset  same shape and dtype
 *   quantScale2      int8 output only: quant2_dtype, 1 or numHeads * headDim entries, 4-byte
 *                    (f32) or 2-byte (bf16) aligned
 *   quantOffset2     nullable (0): same dtype and entries as quantScale2
 *   attentionOut     same shape as query; q_dtype, or int8 with out_dtype IFA_I8
 *   workspace        >= workspace_bytes from ifa_create (nullable when that is 0)
 * Host pointers:
 *   actualSeqLengths int64 (B); NULL means every batch uses maxSeqLen (contiguous only);
 *                    required when paged or left padded.  Values in [0, maxSeqLen]
 *                    (contiguous right padding) or [0, blockTableCols*blockSize] (paged).
 *   kvPaddingSize    int64, 1 or B entries (`n_kv_padding`), nullable; negative values
 *                    count as 0; window [maxSeqLen-pad-len, maxSeqLen-pad), all-zero output
 *                    when its start or end is negative.  Without actualSeqLengths the
 *                    call uses right padding.
 * Device-side data errors (a needed blockTable entry outside [0, blockNum)) leave the
 * affected tokens out and set a flag readable with ifa_get_device_errors.
 * Runs of one plan must not overlap on the GPU (they share the plan's per-sequence
 * arrival counters): use one plan per stream.  Up to B = 256 the call is one kernel launch
 * and can be captured in a CUDA graph; a captured call replays with the lengths it was
 * captured with.  Above B = 256 the per-batch windows are copied from pageable host memory
 * into the workspace on `stream` before the kernel; such a call cannot be captured: under
 * capture it returns IFA_ERR_PARAM_INVALID and leaves the stream untouched.
 * Each call that runs to the end leaves the counters at zero (the CTA that merges a split
 * sequence resets its counter once the other pieces have arrived), so captured and eager calls may be mixed and
 * replayed in any order and number.
 */
ifa_status ifa_run(ifa_plan* plan, const void* query, const void* key, const void* value,
                   const void* attenMask, const int64_t* actualSeqLengths,
                   const int64_t* kvPaddingSize, int64_t n_kv_padding, const int32_t* blockTable,
                   const void* antiquantScale, const void* antiquantOffset, const void* quantScale2,
                   const void* quantOffset2, void* attentionOut, void* workspace, size_t workspace_bytes,
                   void* stream);

/*
 * ifa_run for a plan whose kvFormat is IFA_KV_TENSORLIST: key and value are given as B
 * separate tensors ("IncreFlashAttention" README, non-contiguous key/value: the list holds
 * B tensors of batch 1 whose shapes differ only in S; B <= 256).
 *   keyList, valueList  host arrays of B device pointers (16-byte aligned), tensor b of shape
 *                       (1,S_b,H) / (1,S_b,KV_N,D) / (1,KV_N,S_b,D) per inputLayout
 *   kvSeqLens           host int64 (B): S_b, 1 <= S_b <= maxSeqLen
 * Batch b attends over tokens [0, actualSeqLengths[b]) of its tensor (all S_b when
 * actualSeqLengths is NULL; values above S_b return IFA_ERR_PARAM_INVALID); the mask, when
 * present, is indexed by token as for a contiguous cache (maskS >= the lengths).  Left
 * padding is not defined here (IFA_ERR_PARAM_INVALID at ifa_create).  The other arguments are
 * those of ifa_run.  The library keeps one TMA descriptor per tensor in device memory: a call
 * whose pointers or extents differ from the previous call's re-encodes them and copies them to
 * the device on `stream` before the kernel, so capture a CUDA graph only after a call with
 * the same lists has run: under capture, lists that differ from the previous call's return
 * IFA_ERR_PARAM_INVALID and leave the stream untouched.
 */
ifa_status ifa_run_tensorlist(ifa_plan* plan, const void* query, const void* const* keyList,
                              const void* const* valueList, const int64_t* kvSeqLens, const void* attenMask,
                              const int64_t* actualSeqLengths, const void* antiquantScale,
                              const void* antiquantOffset, const void* quantScale2, const void* quantOffset2,
                              void* attentionOut, void* workspace, size_t workspace_bytes, void* stream);

/* Release a plan (NULL is accepted). Waits for nothing; do not free while a run is in flight. */
ifa_status ifa_destroy(ifa_plan* plan);

/*
 * Synchronise `stream`, return in *flags the device error bits accumulated by this
 * plan's runs since the last call (1: blockTable entry out of range, 2: a pipeline
 * wait timed out), and clear them.  After bit 2 the arrival counters are cleared too
 * (a run that gave up may have left some set); outputs of that run are undefined.
 */
ifa_status ifa_get_device_errors(ifa_plan* plan, void* stream, int64_t* flags);

/*
 * ifa_run_noalloc -- the same computation as ifa_create + ifa_run + ifa_destroy in
 * one call that allocates nothing.  (The pages have no counterpart: their API
 * always asks the caller for a workspace.)
 *
 * For callers that cannot allocate device memory: code that runs inside a
 * memory pool or allocator it does not own, serving runtimes that forbid any
 * allocation on the request path, or processes whose device footprint must not
 * grow after start-up.  Neither this function nor anything it calls uses
 * cudaMalloc, cudaFree or any other allocating routine; host-side state lives on
 * the stack.
 *
 * Scratch: the split-KV partials and the per-sequence arrival counters live in one
 * fixed array of IFA_NOALLOC_SCRATCH_BYTES in the library's device memory.  Every GPU
 * that loads the library holds that array until the process exits, and every call on
 * a device shares it and finds the previous call's contents there.  The partial
 * slots need no clearing.  The per-sequence arrival counters start at zero when the
 * library is loaded, and each call that runs to the end leaves them at zero (the CTA
 * that merges a split sequence resets its counter), in any call order.  A call
 * whose kernel gave up on a wait (error bit 2) may leave counters set, and nothing
 * here can clear them: after that bit, results of later calls on that device are
 * undefined until the process restarts.  Calls whose kernels overlap on the GPU (for
 * example on two streams) race on the array: serialise them.  The first call on
 * each device looks the array's address up (cudaGetSymbolAddress) with that
 * device current; make that first call before any stream capture.
 *
 * Limits: params->B <= IFA_NOALLOC_MAX_BATCH (a larger B returns
 * IFA_ERR_PARAM_INVALID: the per-batch windows travel in the launch parameters),
 * and the grid is capped so that its partials fit the array.  Other arguments,
 * validation and results are those of ifa_run, except that `deviceErrorFlags`
 * (device int32, nullable) receives the device error bits (OR-ed in, never
 * cleared here) instead of a plan's error word.  Asynchronous on `stream`.
 */
#define IFA_NOALLOC_SCRATCH_BYTES (4u << 20)
#define IFA_NOALLOC_MAX_BATCH 256
ifa_status ifa_run_noalloc(const ifa_params* params, const void* query, const void* key, const void* value,
                           const void* attenMask, const int64_t* actualSeqLengths,
                           const int64_t* kvPaddingSize, int64_t n_kv_padding, const int32_t* blockTable,
                           const void* antiquantScale, const void* antiquantOffset, const void* quantScale2,
                           const void* quantOffset2, void* attentionOut, int32_t* deviceErrorFlags,
                           void* stream);

/*
 * Number of CUDA kernels the most recent ifa_run on `plan` enqueued: 1 (the split-KV
 * kernel, which also merges the sequence pieces it cut), or 0 before any run, after a
 * run with B = 0, or for a NULL plan.  Lets callers count launches, e.g. when capturing
 * CUDA graphs.
 */
int64_t ifa_last_launch_count(const ifa_plan* plan);

/*
 * Sparse-index MLA-absorb decode ("SparseFlashAttention" README: formula in 功能说明,
 * arguments in 参数说明, limits in 约束说明):
 *
 *     out[r, n, :] = softmax_j( scale_value * (q[r,n] . k[i_j] + q_rope[r,n] . k_rope[i_j]) ) . v[i_j]
 *
 * for every query row r (a (batch b, query token s) pair), over the tokens i_j its index row
 * selects with 0 <= i_j < limit(r) (tokens outside that range, e.g. from the -1 tail, are
 * skipped wherever they sit; duplicates count once per occurrence; an empty selection gives
 * an all-zero row).  Token-wise (sparse_block_size 1): i_j = sparse_indices[r, 0, j].
 * Block-wise (sparse_block_size = t > 1, README "sparse_block_size"): entry j selects the
 * t tokens sparse_indices[r, 0, j] * t + o, o = 0 .. t - 1.
 *
 * Query rows (layout_query): SFA_LAYOUT_BSND: query (B,Q_S,Q_N,D), row r = b * Q_S + s, and
 * qlen = actual_seq_lengths_query[b] (Q_S when that array is NULL; README: 0 <= qlen <= Q_S).
 * SFA_LAYOUT_TND: query (Q_T,Q_N,D); actual_seq_lengths_query (required) holds B prefix sums
 * (README: cumulative counts), batch b owns rows [cum[b-1], cum[b]) with s counted from its
 * first row and qlen = cum[b] - cum[b-1]; rows past cum[B-1] belong to no batch (zero rows).
 * Key rows (layout_kv): SFA_KV_PA_BSND: caches (block_num, block_size, 1, D); token t of batch
 * b lives in block block_table[b][t / block_size], slot t % block_size; len =
 * actual_seq_lengths_kv[b] (required).  SFA_KV_BSND: key/value (B, KV_S, 1, D), token t of
 * batch b at row b * KV_S + t, len = actual_seq_lengths_kv[b] (KV_S when NULL).  SFA_KV_TND:
 * key/value (KV_S, 1, D) (KV_S = the README's KV_T), actual_seq_lengths_kv (required) holds
 * prefix sums, token t of batch b at row cum[b-1] + t, len = cum[b] - cum[b-1].  Tokens past
 * a batch's rows in the key tensor are skipped.
 * limit(r) = 0 for s >= qlen; otherwise len under sparse_mode 0, and len - qlen + s + 1
 * under sparse_mode 3 (rightDownCausal: the last valid query token is aligned with the last
 * key).  Only what the README lists for this operator is accepted: KV_N = 1, D = 512,
 * Dr = 64, attention_mode 2 (MLA-absorb), sparse_mode 0 or 3, Q_N in 1..128.
 */
#define SFA_LAYOUT_BSND 0
#define SFA_LAYOUT_TND 1
#define SFA_KV_PA_BSND 0
#define SFA_KV_BSND 1
#define SFA_KV_TND 2
typedef struct sfa_params {
    int64_t B;               /* batch (entries of the length arrays), 1..65536 */
    int64_t Q_S;             /* BSND queries: query tokens per batch, 1..1024, B * Q_S <= 2^20 */
    int64_t Q_T;             /* TND queries: query rows, 0..2^20 */
    int64_t Q_N;             /* query heads, 1..128 */
    int64_t KV_N;            /* must be 1 */
    int64_t D;               /* 512: head dim of query, key and value */
    int64_t Dr;              /* 64: rope dim of query_rope and key_rope */
    int64_t KV_S;            /* key rows per batch (SFA_KV_BSND) or in all (SFA_KV_TND); unused when paged */
    int64_t block_size;      /* SFA_KV_PA_BSND: tokens per cache block, a multiple of 16, <= 1024 */
    int64_t block_num;       /* SFA_KV_PA_BSND: blocks in the caches */
    int64_t block_table_cols;/* SFA_KV_PA_BSND: second dimension of block_table */
    int64_t sparse_size;     /* indices per query row, >= 1 */
    int64_t sparse_block_size; /* 1 (token-wise) or a power of two <= 128 (dividing block_size when paged) */
    int32_t dtype;           /* IFA_BF16 or IFA_F16, shared by every tensor and the output */
    int32_t sparse_mode;     /* 0 or 3 */
    int32_t layout_query;    /* SFA_LAYOUT_BSND or SFA_LAYOUT_TND */
    int32_t layout_kv;       /* SFA_KV_PA_BSND, SFA_KV_BSND or SFA_KV_TND */
    double scale_value;      /* scale applied to the scores (typically 1/sqrt(D + Dr)) */
} sfa_params;

/* Workspace bytes sfa_run needs for `params` on the current device.  Returns
 * IFA_ERR_PARAM_INVALID for a description outside the supported range. */
ifa_status sfa_workspace_size(const sfa_params* params, size_t* workspace_bytes);

/*
 * Enqueue one sparse decode call on `stream` (cudaStream_t, NULL = legacy default).
 * Device pointers, 16-byte aligned unless noted (R = B * Q_S or Q_T query rows):
 *   query (R,Q_N,D), query_rope (R,Q_N,Dr), attention_out (R,Q_N,D); key and value
 *   (rows, D) and key_rope (rows, Dr) in the layout_kv shapes above, all of `dtype`;
 *   sparse_indices int32 (R,1,sparse_size); block_table int32 (B, block_table_cols), paged
 *   only (nullable otherwise); actual_seq_lengths_kv and actual_seq_lengths_query int32 (B),
 *   nullable where the layout allows (4-byte aligned); softmax_max and softmax_sum float32
 *   (R, Q_N), nullable (README softmax_max_out / softmax_sum_out, accepted with every
 *   layout): the largest scaled score and the sum of exp(score - softmax_max) of each
 *   (row, head), -inf and 0 for an empty selection; workspace of at least
 *   sfa_workspace_size bytes; deviceErrorFlags (int32, nullable) receives device error
 *   bits (1: a needed block_table entry outside [0, block_num); 2: a wait timed out).
 * `value` may alias `key`.  Calls that share a workspace must not overlap on the GPU.
 * The call enqueues three kernels: a tile-count kernel that finds each query row's live
 * tiles and writes the zero output rows of query rows with no usable index (one warp per
 * row; above 1024 query rows one cluster of 8 CTAs, which also splits the live tiles across
 * the decode kernel's CTA pairs), the decode kernel (pairs of CTAs, one per value half,
 * launched with programmatic dependent launch after the count; up to 1024 query rows each
 * CTA derives its pair's share from the counts itself) and a combine kernel that merges the
 * pieces of the (query row, value half) sequences the decode kernel split across CTA pairs.  The workspace needs no initialisation.  Returns
 * IFA_ERR_RUNTIME when no CTA pair fits on the device or a launch fails.
 */
ifa_status sfa_run(const sfa_params* params, const void* query, const void* query_rope, const void* key,
                   const void* key_rope, const void* value, const int32_t* sparse_indices,
                   const int32_t* block_table, const int32_t* actual_seq_lengths_kv,
                   const int32_t* actual_seq_lengths_query, void* attention_out, float* softmax_max,
                   float* softmax_sum, void* workspace, size_t workspace_bytes, int32_t* deviceErrorFlags,
                   void* stream);

/*
 * KV-cache append: the step before the attention in incremental decode (IncreFlashAttention
 * README: each step attends over the cache grown by the new token).  The key and value rows
 * of one new token per batch are written at token position positions[b] of the caches,
 * through the addressing ifa_run reads: contiguous (B,KV_N,Smax,D) BNSD, (B,Smax,KV_N,D) BSND
 * or (B,Smax,H) BSH (maxSeqLen = Smax), or paged (blockNum, KV_N, blockSize, D) /
 * (blockNum, blockSize, H) through blockTable (block blockTable[b][t / blockSize], slot
 * t % blockSize).  A 16-bit cache (kv_dtype = new_dtype) receives the values unchanged.  An
 * int8 cache receives, per element, rint(x / scale - offset) computed in single precision
 * (ties to even) and saturated to [-128, 127] (NaN gives 0), with the antiquant scale and
 * offset the element is read back with (per channel: (2, KV_N, D) memory, entry 0 for key and
 * 1 for value; per tensor: (2,)) -- the inverse of the reading x = (code + offset) * scale.
 */
typedef struct ifa_append_params {
    int64_t B;                /* batch, 0..2^20 */
    int64_t numKeyValueHeads; /* KV_N, 1..256 */
    int64_t headDim;          /* D: a multiple of 8 (16 for int8 caches), <= 512 */
    int64_t maxSeqLen;        /* contiguous caches: Smax */
    int64_t blockSize, blockNum, blockTableCols; /* paged caches */
    int32_t new_dtype;        /* IFA_F16 or IFA_BF16: the new rows and the antiquant parameters */
    int32_t kv_dtype;         /* = new_dtype, or IFA_I8 (requires antiquant) */
    int32_t inputLayout;      /* ifa_layout of a contiguous cache */
    int32_t kvFormat;         /* ifa_kv_format */
    int32_t antiquant;        /* ifa_antiquant; not NONE exactly when kv_dtype is IFA_I8 */
} ifa_append_params;

/*
 * Enqueue one append on `stream` (cudaStream_t, NULL = legacy default); one kernel launch.
 * Device pointers: keyNew and valueNew (B, KV_N, D) in memory (any layout with S = 1) of
 * new_dtype, 16-byte aligned; positions int64 (B), 8-byte aligned; blockTable int32
 * (B, blockTableCols), paged only; antiquantScale / antiquantOffset (int8 caches) of
 * new_dtype; keyCache and valueCache 16-byte aligned; deviceErrorFlags (int32, nullable)
 * receives bit 1 for a batch whose position lies outside the cache (negative, >= Smax, past
 * the block table, or a block id outside [0, blockNum)): that batch writes nothing.
 * Returns IFA_ERR_PARAM_NULLPTR / IFA_ERR_PARAM_INVALID / IFA_ERR_RUNTIME as ifa_run does.
 */
ifa_status ifa_kv_append(const ifa_append_params* params, const void* keyNew, const void* valueNew,
                         const int64_t* positions, const int32_t* blockTable, const void* antiquantScale,
                         const void* antiquantOffset, void* keyCache, void* valueCache, int32_t* deviceErrorFlags,
                         void* stream);

/* Static text for a status code. */
const char* ifa_status_string(ifa_status status);

#ifdef __cplusplus
}
#endif
#endif /* IFA_H */
