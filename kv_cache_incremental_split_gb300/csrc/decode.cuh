// Launch parameters and compile-time configuration of the split-KV decode
// kernel, and the host planning helpers that fill them in.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ifa.h"

namespace ifa {

constexpr int kMaskBox = 128;        // bytes per mask TMA box; a tile's boxes land back to back on 128-byte
                                     // boundaries (a tensor copy's shared-memory destination must be)
constexpr int kInlineB = 256;        // per-batch windows travel in the launch parameters up to this B
constexpr int kMaxCtas = 256;        // upper bound on the grid
constexpr int kMinPieceTiles = 4;    // do not cut sequences into pieces shorter than this (tiles)
// Fixed work of a sequence piece, in key/value bytes of tile time, weighing the CTA split: a
// whole sequence pays its epilogue (kPieceCostBytes); each piece of a sequence that CTA
// boundaries cut pays the partial write, the arrival and its share of the merge, which sit
// on the latency path at the end of a CTA's range (kCutCostBytes).
constexpr int kPieceCostBytes = 64 * 1024;
constexpr int kCutCostBytes = 160 * 1024;
constexpr int kPieceCostBytesI8 = 192 * 1024;
constexpr int kCutCostBytesI8 = 320 * 1024;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // bounded spin-waits: 2 s
constexpr int kMaxDevices = 64;      // devices whose one-time kernel set-up is tracked

// The current device as an index for per-device one-time set-up (kernel attributes such as the
// dynamic shared-memory limit are set per device), or -1 when it cannot be read or is kMaxDevices
// or beyond.
inline int current_device_slot() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    return (dev >= 0 && dev < kMaxDevices) ? dev : -1;
}

// Device error word bits (OR-ed into the error word).
constexpr int kErrBadBlock = 1;      // a needed blockTable entry outside [0, blockNum)
constexpr int kErrTimeout = 2;       // a pipeline wait ran out of time

enum KvKind : int { KV_BF16 = 0, KV_F16 = 1, KV_I8 = 2 };

// Per-batch windows, laid out as int32 st[B], len[B], pre[B+1]:
//   st  : first valid position in the key/value S coordinate
//   len : valid tokens (0 = all-zero output row)
//   pre : exclusive prefix over batches of (tiles of b) x (sequences of b)
struct alignas(128) DecodeParams {
    CUtensorMap tmK;   // 4-D map (x=d, y=token, z=kv head, w=batch or block), box_rows-row boxes
    CUtensorMap tmV;
    CUtensorMap tmKt;  // the same tensors with tail_rows-row boxes, for the last tile of a window
    CUtensorMap tmVt;
    CUtensorMap tmM;   // 2-D (mask position, mask row) over a per-batch mask, used when mask_tma
    const void* q;
    void* out;
    const uint8_t* mask;
    const int32_t* block_table;
    const void* aq_scale;
    const void* aq_offset;
    float* partials;           // 2 slots per CTA
    unsigned int* counters;    // arrival counters [kMaxCtas], zero between calls (the merging CTA resets)
    int* err;
    const int32_t* ext_bdata;  // per-batch windows in global memory when B > kInlineB
    long long W;               // total tiles
    int P;                     // CTAs of this launch
    int B, N, KV_N, D, G, GT, NGS;
    int q_bf16;
    int paged;
    int block_size, bt_cols, block_num, box_rows, tail_rows;
    long long mask_bstride, mask_nstride;
    int has_mask;
    int mask_tma;              // the producer stages each tile's mask bytes (per-batch masks)
    int aq_per_channel;
    int aq_stage;              // per-channel key scales reach shared memory with each piece's query
    const CUtensorMap* kv_maps;  // one tensor per batch: 4 maps per batch (K, K tail, V, V tail), else null
    int out_i8;                // int8 output: code = saturate(rint(y * scale2 + offset2))
    int q2_per_channel;        // scale2/offset2 entry n * D + d (else entry 0)
    int q2_bf16;               // scale2/offset2 are bf16 (else fp32)
    const void* q2_scale;
    const void* q2_offset;     // nullable: 0
    float scale_log2;          // scaleValue * log2(e)
    int slot_floats;
    int bdata_inline[3 * kInlineB + 1];
    int bounds[kMaxCtas + 1];  // CTA c takes the tiles [bounds[c], bounds[c+1]), strictly increasing
};

__host__ __device__ constexpr int round_up_c(int x, int m) { return (x + m - 1) / m * m; }
__host__ __device__ constexpr int clamp_c(int x, int lo, int hi) { return x < lo ? lo : (x > hi ? hi : x); }

template <int KV, int DPAD, int NT>
struct DecodeCfg {
    static constexpr int ES = KV == KV_I8 ? 1 : 2;            // key/value element bytes
    static constexpr int CG_ELEMS = 128 / ES;                  // elements per 128-byte column group
    static constexpr int NCG = DPAD * ES / 128;                // column groups per row
    static constexpr int NWC = DPAD <= 128 ? 8 : 4;            // consumer warps
    // Eight consumer warps plus a producer would leave 168 registers a thread (three warps
    // on one SM sub-partition); with twelve warps the producer's warpgroup gives registers
    // back (setmaxnreg) so the two consumer warpgroups get CONSUMER_REGS each.
    static constexpr bool SPLIT_REGS = NWC == 8;
    static constexpr int THREADS = SPLIT_REGS ? 12 * 32 : (NWC + 1) * 32;  // consumers + producer (+ 3 idle)
    static constexpr int CONSUMER_REGS = 200, PRODUCER_REGS = 56;
    static constexpr int REG_POOL_NEEDED = NWC * 32 * CONSUMER_REGS + 4 * 32 * PRODUCER_REGS;
    // int8 tiles are half the bytes of 16-bit ones: each consumer warp takes two 16-token
    // mma M tiles, so a stage holds as many bytes and the per-tile work is shared by 32 tokens.
    static constexpr int KWT = (KV == KV_I8 && DPAD <= 128) ? 32 : 16;  // tokens of a stage per consumer warp
    static constexpr int MTW = KWT / 16;                        // 16-token mma M tiles per consumer warp
    static constexpr int T = KWT * NWC;                         // tokens per stage (one tile)
    static constexpr int KT_BYTES = NCG * T * 128;             // one K (or V) tile
    static constexpr int GT_PAD = 8 * NT;                      // query heads per CTA, padded
    static constexpr int QROW = DPAD * 2 + 16;                 // padded query row in shared memory
    static constexpr int Q_BYTES = GT_PAD * QROW;
    static constexpr int MASK_LOADS = (T + 16 + kMaskBox - 1) / kMaskBox;  // mask boxes per tile
    static constexpr int MASK_BYTES = MASK_LOADS * kMaskBox;  // one tile's mask bytes, contiguous
    static constexpr int MASK_OFF = 2 * KT_BYTES + Q_BYTES;    // within a stage
    static constexpr int AQ_OFF = MASK_OFF + MASK_BYTES;       // int8: the key scale row of a piece's kv head
    static constexpr int AQ_BYTES = KV == KV_I8 ? DPAD * 2 : 0;
    static constexpr int STAGE_BYTES = round_up_c(2 * KT_BYTES + Q_BYTES + MASK_BYTES + AQ_BYTES, 1024);
    static constexpr int MW = NWC < 4 ? NWC : 4;               // warps the merge buffer holds at once
    static constexpr int FRAG4 = (DPAD / 16) * NT;             // float4 accumulator groups per lane
    // merge buffer: MW warps' accumulator fragments, lane-contiguous float4; also holds the
    // (M, L) of up to kMaxCtas pieces when a cut sequence's first CTA merges it
    static constexpr int MERGE_BYTES = MW * FRAG4 * 32 * 16 > 2 * kMaxCtas * GT_PAD * 4 ? MW * FRAG4 * 32 * 16
                                                                                          : 2 * kMaxCtas * GT_PAD * 4;
    static constexpr int ML_BYTES = 2 * NWC * GT_PAD * 4;      // per-warp running max and sum of each head
    static constexpr int BD_BYTES = round_up_c((3 * kInlineB + 1 + kMaxCtas + 1) * 4, 128);  // windows, bounds
    static constexpr int INFO_BYTES = 8 * 32;                  // TileInfo of each stage
    static constexpr int BAR_BYTES = 256;
    static constexpr int AUX_BYTES = MERGE_BYTES + ML_BYTES + BD_BYTES + INFO_BYTES + BAR_BYTES;
    static constexpr int BUDGET = 225 * 1024;
    static constexpr int STAGES = clamp_c((BUDGET - AUX_BYTES - 1024) / STAGE_BYTES, 2, 8);
    static constexpr int PREFETCH_TILES = STAGES;  // tiles pulled into L2 before the previous kernel ends
    static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + AUX_BYTES;
    static constexpr int SLOT_FLOATS = GT_PAD * DPAD + 2 * GT_PAD;
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
    static_assert(T % 32 == 0, "tiles are whole 32-row sub-boxes");
    static_assert(MASK_OFF % 128 == 0 && kMaskBox % 128 == 0 && T + 16 <= MASK_BYTES, "mask staging area");
    static_assert(T <= 256, "TMA boxes hold at most 256 rows");
};

typedef cudaError_t (*DecodeLaunchFn)(const DecodeParams&, int grid, cudaStream_t);

// ---------------------------------------------------------------- host planning (plan.cu)

// Kernel variant and sizes chosen for one problem description.
struct KernelChoice {
    int KV_N, G, GT, NT, NGS;
    int kv_kind, es, dpad;
    int T;          // tokens per tile
    int box_rows;   // rows per TMA box of a full tile (a whole tile, or one cache block)
    int tail_rows;  // rows per TMA box of a window's last, partial tile
    int piece_cost; // fixed work of a whole sequence, in 1/16 tiles (weights the CTA split)
    int cut_cost;   // fixed work of each piece of a cut sequence, in 1/16 tiles
    int slot_floats, smem, threads;
    DecodeLaunchFn launch;
};

// Paged key/value caches (a block table maps tokens to blocks).
inline bool kv_paged(const ifa_params& p) {
    return p.kvFormat == IFA_KV_PAGED_NBSD || p.kvFormat == IFA_KV_PAGED_BSH;
}
bool params_are_valid(const ifa_params& p);
ifa_status choose_kernel(const ifa_params& p, KernelChoice* kc);
// Fills st/len/pre of every batch into bd (3B+1 ints); returns W and the longest sequence in tiles.
ifa_status build_windows(const ifa_params& p, const KernelChoice& kc, const int64_t* lens, const int64_t* pads,
                         int64_t n_pads, int32_t* bd, int64_t* W, int* max_seq_tiles);
int choose_grid(const ifa_params& p, int64_t W, int max_seq_tiles, int P_max);
// Tile ranges of the P CTAs (bounds[0..P]), from the windows build_windows wrote.
void build_bounds(const ifa_params& p, const KernelChoice& kc, const int32_t* bd, int64_t W, int P, int32_t* bounds);
// Checks of the per-call pointers shared by both run entry points.
ifa_status check_run_pointers(const ifa_params& p, const void* query, const void* key, const void* value,
                              const void* attenMask, const int64_t* actualSeqLengths, const int64_t* kvPaddingSize,
                              int64_t n_kv_padding, const int32_t* blockTable, const void* antiquantScale,
                              const void* antiquantOffset, const void* quantScale2, const void* quantOffset2,
                              const void* attentionOut);
bool encode_kv_map(const ifa_params& p, const KernelChoice& kc, const void* base, int box_rows, CUtensorMap* map);
// The four maps a call needs (key/value x full/tail boxes).
bool encode_kv_maps(const ifa_params& p, const KernelChoice& kc, const void* key, const void* value, DecodeParams& dp);
// Stages per-tile mask bytes by TMA when the mask is per batch and 16-byte aligned: sets
// dp.mask_tma and dp.tmM.  Returns false only when encoding fails.
bool encode_mask_map(const ifa_params& p, const KernelChoice& kc, const void* mask, DecodeParams& dp);
// Everything but the tensor maps, the scratch pointers and the window table.
void fill_decode_params(DecodeParams& dp, const ifa_params& p, const KernelChoice& kc, const void* query,
                        const void* attenMask, const int32_t* blockTable, const void* antiquantScale,
                        const void* antiquantOffset, const void* quantScale2, const void* quantOffset2,
                        void* attentionOut, int64_t W, int P);

DecodeLaunchFn decode_launcher(int kv_kind, int dpad, int nt, bool tensorlist);
bool decode_cfg(int kv_kind, int dpad, int nt, int* slot_floats, int* smem, int* tile_tokens, int* threads);

}  // namespace ifa
