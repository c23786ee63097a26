// Launch parameters and compile-time configuration of the split-KV decode
// kernels (partial kernel + log-sum-exp combine), shared by the kernels and by
// the host planner that fills them in.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ifa {

constexpr int kTileTokens = 64;      // key/value tokens per pipeline stage
constexpr int kWarpTokens = 16;      // tokens of a stage owned by one consumer warp
constexpr int kConsumerWarps = kTileTokens / kWarpTokens;
constexpr int kThreads = (kConsumerWarps + 1) * 32;  // + one producer warp
constexpr int kInlineB = 256;        // per-batch windows travel in the launch parameters up to this B
constexpr int kMaxCtas = 256;        // upper bound on the partial kernel's grid
constexpr int kMaxJobs = kMaxCtas;   // combine jobs (split sequences) per call
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // bounded spin-waits: 2 s

// Device error word bits (OR-ed into the plan's error word).
constexpr int kErrBadBlock = 1;      // a needed blockTable entry outside [0, blockNum)
constexpr int kErrTimeout = 2;       // a pipeline wait ran out of time

enum KvKind : int { KV_BF16 = 0, KV_F16 = 1, KV_I8 = 2 };

// Per-batch windows, laid out as int32 st[B], len[B], pre[B+1]:
//   st  : first valid position in the key/value S coordinate
//   len : valid tokens (0 = all-zero output row)
//   pre : exclusive prefix of tiles over batches (tiles of b times the
//         number of (kv head, query-head slice) sequences of b)
struct alignas(128) DecodeParams {
    CUtensorMap tmK;  // 4-D map (x=d, y=token, z=kv head, w=batch or block)
    CUtensorMap tmV;
    const void* q;
    void* out;
    const uint8_t* mask;
    const int32_t* block_table;
    const void* aq_scale;
    const void* aq_offset;
    float* partials;
    int* err;
    const int32_t* ext_bdata;  // per-batch windows in global memory when B > kInlineB
    long long W;               // total tiles
    int P;                     // CTAs of this launch
    int B, N, KV_N, D, G, GT, NGS;
    int q_bf16;
    int paged;
    int block_size, bt_cols, block_num, box_rows;
    long long mask_bstride, mask_nstride;
    int has_mask;
    int aq_per_channel;
    float scale_log2;          // scaleValue * log2(e)
    int slot_floats;
    int bdata_inline[3 * kInlineB + 1];
};

struct CombineJob {
    int seq;          // (b * KV_N + h) * NGS + gs
    int c_first;      // first CTA holding a piece
    int c_last;       // last CTA holding a piece
    int first_odd;    // the first piece sits in slot 2*c_first + 1 (else 2*c_first)
};

struct CombineParams {
    void* out;
    const float* partials;
    const void* aq_scale;
    const void* aq_offset;
    int N, D, G, GT, NGS, KV_N;
    int q_bf16, kv_i8, aq_per_channel;
    int slot_floats, d_pad, gt_pad;
    int njobs;
    CombineJob jobs[kMaxJobs];
};

__host__ __device__ constexpr int round_up_c(int x, int m) { return (x + m - 1) / m * m; }

template <int KV, int DPAD, int NT>
struct DecodeCfg {
    static constexpr int ES = KV == KV_I8 ? 1 : 2;            // key/value element bytes
    static constexpr int CG_ELEMS = 128 / ES;                  // elements per 128-byte column group
    static constexpr int NCG = DPAD * ES / 128;                // column groups per row
    static constexpr int T = kTileTokens;
    static constexpr int KT_BYTES = NCG * T * 128;             // one K (or V) tile
    static constexpr int GT_PAD = 8 * NT;                      // query heads per CTA, padded
    static constexpr int QROW = DPAD * 2 + 16;                 // padded query row in shared memory
    static constexpr int Q_BYTES = GT_PAD * QROW;
    static constexpr int STAGE_BYTES = round_up_c(2 * KT_BYTES + Q_BYTES, 1024);
    static constexpr int MERGE_BYTES = kConsumerWarps * GT_PAD * (DPAD + 2) * 4;
    static constexpr int BUDGET = 220 * 1024;
    static constexpr int STAGES_FIT = (BUDGET - MERGE_BYTES - 2048) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT < 2 ? 2 : (STAGES_FIT > 8 ? 8 : STAGES_FIT);
    static constexpr int BAR_BYTES = 256;
    static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + MERGE_BYTES + BAR_BYTES;
    static constexpr int SLOT_FLOATS = GT_PAD * DPAD + 2 * GT_PAD;
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

// Host-side launchers (defined per key/value kind in their own translation units).
typedef cudaError_t (*DecodeLaunchFn)(const DecodeParams&, int grid, cudaStream_t);
DecodeLaunchFn decode_launcher(int kv_kind, int dpad, int nt);
cudaError_t launch_combine(const CombineParams& p, int max_pieces, cudaStream_t stream);

}  // namespace ifa
