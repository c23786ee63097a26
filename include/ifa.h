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
 * ("IncreFlashAttention" README, page attention constraints.) */
typedef enum { IFA_KV_CONTIG = 0, IFA_KV_PAGED_NBSD = 1, IFA_KV_PAGED_BSH = 2 } ifa_kv_format;

typedef enum { IFA_F16 = 0, IFA_BF16 = 1, IFA_I8 = 2, IFA_U8 = 3, IFA_BOOL = 4 } ifa_dtype;

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
    int64_t maxSeqLen;        /* CONTIG: the key/value S extent (Smax); ignored when paged */
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
} ifa_params;

typedef struct ifa_plan ifa_plan;

/*
 * Phase 1: validate `params` and build a plan for the current CUDA device.
 *   plan            out: owned by the library, free with ifa_destroy
 *   workspace_bytes out: device workspace every ifa_run on this plan needs
 * Returns IFA_ERR_PARAM_NULLPTR for NULL arguments, IFA_ERR_PARAM_INVALID for a
 * description outside the supported range, IFA_ERR_RUNTIME if the device
 * cannot be queried.  Allocates the plan and a 4-byte device error word.
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
 *   attentionOut     same shape and dtype as query
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
 * arrival counters): use one plan per stream.  The call is one kernel launch and can be
 * captured in a CUDA graph; a captured call replays with the lengths it was captured with.
 */
ifa_status ifa_run(ifa_plan* plan, const void* query, const void* key, const void* value,
                   const void* attenMask, const int64_t* actualSeqLengths,
                   const int64_t* kvPaddingSize, int64_t n_kv_padding, const int32_t* blockTable,
                   const void* antiquantScale, const void* antiquantOffset, void* attentionOut,
                   void* workspace, size_t workspace_bytes, void* stream);

/* Release a plan (NULL is accepted). Waits for nothing; do not free while a run is in flight. */
ifa_status ifa_destroy(ifa_plan* plan);

/*
 * Synchronise `stream`, return in *flags the device error bits accumulated by this
 * plan's runs since the last call (1: blockTable entry out of range, 2: a pipeline
 * wait timed out), and clear them.
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
 * a device shares it and finds the previous call's contents there.  Nothing in it
 * needs to start at zero: the counters carry a per-call tag, so a value left by an
 * earlier (even aborted) call is ignored.  Calls whose kernels overlap on the GPU (for
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
                           const void* antiquantScale, const void* antiquantOffset, void* attentionOut,
                           int32_t* deviceErrorFlags, void* stream);

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
 *     out[b, n, :] = softmax_j( scale_value * (q[b,n] . k[i_j] + q_rope[b,n] . k_rope[i_j]) ) . v[i_j]
 *
 * for every query token s of batch b (the line holds with q[b,s,n], i_j from row (b, s) and
 * out[b,s,n]), over the selected tokens i_j with 0 <= i_j < limit(b, s) (tokens outside that
 * range, e.g. from the -1 tail, are skipped wherever they sit; duplicates count once per
 * occurrence; an empty selection gives an all-zero row).  Token-wise (sparse_block_size 1):
 * i_j = sparse_indices[b, s, 0, j].  Block-wise (sparse_block_size = t > 1, README
 * "sparse_block_size"): entry j selects the t tokens sparse_indices[b, s, 0, j] * t + o,
 * o = 0 .. t - 1.  Token i lives in block block_table[b][i / block_size], slot
 * i % block_size of the PA_BSND caches.  With len = actual_seq_lengths_kv[b] and
 * qlen = actual_seq_lengths_query[b] (Q_S when that array is NULL; README: 0 <= qlen <= Q_S):
 * limit(b, s) = 0 for s >= qlen (an all-zero row); otherwise len under sparse_mode 0, and
 * len - qlen + s + 1 under sparse_mode 3 (rightDownCausal: the last valid query token is
 * aligned with the last key).  Only the layouts and modes the README lists for this case are
 * accepted: query layout BSND, key/value layout PA_BSND, KV_N = 1, D = 512, Dr = 64,
 * attention_mode 2 (MLA-absorb), sparse_mode 0 or 3, Q_N in 1..128.
 */
typedef struct sfa_params {
    int64_t B;               /* batch, 1..65536 */
    int64_t Q_S;             /* query tokens per batch, 1..1024, B * Q_S <= 2^20 */
    int64_t Q_N;             /* query heads, 1..128 */
    int64_t KV_N;            /* must be 1 */
    int64_t D;               /* 512: head dim of query, key and value */
    int64_t Dr;              /* 64: rope dim of query_rope and key_rope */
    int64_t block_size;      /* tokens per cache block: a multiple of 16, <= 1024 */
    int64_t block_num;       /* blocks in the caches */
    int64_t block_table_cols;/* second dimension of block_table */
    int64_t sparse_size;     /* indices per query row, >= 1 */
    int64_t sparse_block_size; /* 1 (token-wise) or a power of two <= 128 dividing block_size */
    int32_t dtype;           /* IFA_BF16 or IFA_F16, shared by every tensor and the output */
    int32_t sparse_mode;     /* 0 or 3 */
    double scale_value;      /* scale applied to the scores (typically 1/sqrt(D + Dr)) */
} sfa_params;

/* Workspace bytes sfa_run needs for `params` on the current device.  Returns
 * IFA_ERR_PARAM_INVALID for a description outside the supported range. */
ifa_status sfa_workspace_size(const sfa_params* params, size_t* workspace_bytes);

/*
 * Enqueue one sparse decode call on `stream` (cudaStream_t, NULL = legacy default).
 * Device pointers, 16-byte aligned unless noted:
 *   query (B,Q_S,Q_N,D), query_rope (B,Q_S,Q_N,Dr), key and value (block_num, block_size, 1, D),
 *   key_rope (block_num, block_size, 1, Dr), attention_out (B,Q_S,Q_N,D), all of `dtype`;
 *   sparse_indices int32 (B,Q_S,1,sparse_size), block_table int32 (B, block_table_cols),
 *   actual_seq_lengths_kv int32 (B) and actual_seq_lengths_query int32 (B, nullable)
 *   (4-byte aligned); workspace of at least
 *   sfa_workspace_size bytes; deviceErrorFlags (int32, nullable) receives device error
 *   bits (1: a needed block_table entry outside [0, block_num); 2: a wait timed out).
 * `value` may alias `key`.  Calls that share a workspace must not overlap on the GPU.
 * The call enqueues two kernels: the decode kernel, and a combine kernel that merges
 * the pieces of the (batch, value-half) sequences the decode kernel split across CTAs.
 */
ifa_status sfa_run(const sfa_params* params, const void* query, const void* query_rope, const void* key,
                   const void* key_rope, const void* value, const int32_t* sparse_indices,
                   const int32_t* block_table, const int32_t* actual_seq_lengths_kv,
                   const int32_t* actual_seq_lengths_query, void* attention_out, void* workspace,
                   size_t workspace_bytes, int32_t* deviceErrorFlags, void* stream);

/* Static text for a status code. */
const char* ifa_status_string(ifa_status status);

#ifdef __cplusplus
}
#endif
#endif /* IFA_H */
