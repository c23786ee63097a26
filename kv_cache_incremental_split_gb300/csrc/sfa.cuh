// Sparse-index MLA-absorb decode ("SparseFlashAttention" README): launch
// parameters and fixed sizes of the tcgen05 kernel, its tile-count and combine kernels
// (sfa_kernel.cu).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ifa.h"

namespace ifa {

constexpr int kSfaTile = 128;       // sparse positions per tile (the N of S = Q K^T)
constexpr int kSfaD = 512;          // head dim of query, key and value
constexpr int kSfaDr = 64;          // rope dim
constexpr int kSfaHalf = 256;       // value channels per CTA sequence (one half of D)
constexpr int kSfaQBlocks = 9;      // 64-column blocks of [q | q_rope]
constexpr int kSfaVBlocks = 4;      // 64-column blocks of one value half
constexpr int kSfaStages = 4;       // 16 KB ring stages (kSfaTile rows x 128 B)
constexpr int kSfaStageBytes = kSfaTile * 128;
constexpr int kSfaQBytes = kSfaQBlocks * 128 * 128;
constexpr int kSfaRSlots = 8;       // resolved tiles the resolver warp may run ahead
constexpr int kSfaRSlotBytes = 544; // rows[kSfaTile], valid mask, flag (16-byte aligned)
constexpr int kSfaIssuers = 4;     // warps that issue the ring's gathers (a stage's kSfaTile / 4 row groups split evenly)
constexpr int kSfaThreads = 10 * 32;  // producer, MMA issuer, four softmax warps, resolver, three more gatherers
// partial slot: the normalised O of one piece as [64 channel quads][128 head rows][4 floats],
// then M, L and the largest score of each head row
constexpr int kSfaSlotFloats = 128 * kSfaHalf + 3 * 128;
constexpr int kSfaBarBytes = 512;
constexpr int kSfaSmem = 1024 + kSfaQBytes + kSfaStages * kSfaStageBytes + kSfaRSlots * kSfaRSlotBytes + kSfaBarBytes;
// workspace: [0, 256) error word; [kSfaStartOffset, + 32 * kMaxCtas) each pair's start (SfaStart);
// partial slots from kSfaPartialOffset; then live tiles per query row (R ints), their prefix
// over rows (R + 1 ints) and, 16-byte aligned, the pieces of each row (R SfaPieces)
constexpr size_t kSfaStartOffset = 1024;
constexpr size_t kSfaPartialOffset = 16384;
constexpr int kSfaCountCtas = 8;        // the cluster tile-count kernel (above kSfaLocalRows query rows)
constexpr int kSfaCountThreads = 512;
constexpr int kSfaCountSmemRows = 4096;  // rows whose counts the count kernel scans in shared memory
constexpr int kSfaLocalRows = 1024;  // up to this many query rows each decode CTA derives the split itself
// The smallest share of live tiles a CTA pair takes.  A pair's first tile costs about as much
// as two more (the query and the first key stages land together), so small problems run
// fastest spread over every pair, one tile each.
constexpr int kSfaMinShareTiles = 1;
constexpr int kSfaRowCountWarps = 2;  // rows (one per warp) of a CTA of the per-row count kernel
constexpr int kSfaCombineThreads = 256;  // threads of a combine block: 8 head rows x 32 groups of 8 channels
constexpr float kSfaRescaleSlack = 8.0f;    // log2 units the running max may trail before O is rescaled
constexpr float kLn2 = 0.6931471805599453f;  // scores in log2 units -> natural units

// Where a CTA of the decode kernel starts: tiles [lo, hi) of the live-tile order, the first
// one tile t of sequence (query row r, value half h), a sequence of n tiles whose first tile
// has index `first`.
struct SfaStart {
    int lo, hi, r, h, t, n, first, pad;
};
static_assert(sizeof(SfaStart) == 32, "start table entry");

// Where the pieces of query row r's two sequences sit: pairs c_first .. c_first + np - 1 (np = 0
// for a row with no live tile, 1 for a row one pair holds whole); the first piece's partial
// slot within its CTA (0 when the row starts that pair's share, else 1).
struct alignas(16) SfaPieces {
    int c_first, np, slot0, pad;
};

struct alignas(128) SfaParams {
    CUtensorMap tmQ;    // 3-D (d, head, query row) over query, 64 x 128 x 1 boxes
    CUtensorMap tmQr;   // same over query_rope
    CUtensorMap tmK;    // 2-D (d, cache row) over key, 64 x 1 boxes (row gathers)
    CUtensorMap tmKr;   // over key_rope
    CUtensorMap tmV;    // over value
    CUtensorMap tmKb;   // block-wise runs (sparse_block_size >= 8): the same tensors with
    CUtensorMap tmKrb;  //   64 x min(sparse_block_size, 64) boxes of consecutive rows
    CUtensorMap tmVb;
    const int32_t* indices;
    const int32_t* block_table;
    const int32_t* lens;    // key lengths per batch; prefix sums when the key layout is TND
    const int32_t* lens_q;  // valid query tokens per batch (nullable: all Q_S); prefix sums for TND queries
    void* out;
    float* lse_max;         // nullable: largest scaled score of each (query row, head)
    float* lse_sum;         // nullable: sum of exp(score - lse_max) of each (query row, head)
    float* partials;
    int* err;
    SfaStart* starts;   // per pair, written by the cluster tile-count kernel (above kSfaLocalRows rows)
    int* eff;           // live tiles of each query row (a sequence's tiles), 0 when no index is usable
    int* pre;           // prefix over rows of eff (R + 1 entries), written by the cluster tile-count kernel
    SfaPieces* pieces;  // per query row, for the combine kernel: written by the tile-count kernel (rows with
                        // no live tile, and every row above kSfaLocalRows rows) or by the decode kernel's pairs
    long long W;        // tiles before the count: R * tiles_per_seq (an upper bound)
    int P;              // CTAs: an even count; CTAs 2c and 2c + 1 (the two value halves) form pair c
    int R, QS, QN, S_sp, tiles_per_seq;  // R query rows: B * QS (row r: batch r / QS, query token r % QS), or
                                         // the TND rows; S_sp: indices per row; tiles cover S_sp << sbs_log2
    int B;                           // batches (entries of the length arrays)
    int q_tnd;                       // query rows packed per batch (prefix-sum lens_q)
    int kv_layout;                   // 0 PA_BSND (block table), 1 BSND (row b * kv_s + t), 2 TND (prefix-sum lens)
    int kv_s;                        // BSND: tokens per batch in the key tensor; TND: key rows
    int causal;                      // sparse_mode 3: query token s of a batch sees keys up to len - qlen + s
    int sbs_log2;                    // log2(sparse_block_size): position p reads index p >> sbs_log2
    int block_size, bt_cols, block_num, total_rows;
    int is_bf16;
    float scale_log2;
};

// CTA pairs of the decode kernel that can be resident at once (0 when the query fails).
int sfa_max_pairs();

// Enqueues the tile-count kernel, the decode kernel and the combine kernel (three launches).
cudaError_t launch_sfa(const SfaParams& p, cudaStream_t stream);

}  // namespace ifa
