// Sparse-index MLA-absorb decode on the 5th-generation tensor cores.
//
//   out[b, n, :] = softmax_j(scale * (q[b,n] . k[i_j] + q_rope[b,n] . k_rope[i_j])) . v[i_j]
//   ("SparseFlashAttention" README, 功能说明 formula; i_j = sparse_indices[b,0,0,j]).
//
// Work: a sequence is (batch b, value half h): 128 query heads x 256 of the 512
// value channels (a full 128 x 512 fp32 accumulator would fill all of TMEM, so
// the two halves are separate sequences; the two CTAs of a pair hold the halves
// of the same positions, walk them at the same time and each gather the key rows
// themselves: the second read of a key row mostly hits L2).
// A sequence is cut into 128-position tiles of its sparse index row.  A first
// kernel finds each row's live tiles (up to the last tile holding a usable index:
// the invalid tail after it costs nothing); persistent CTA pairs take equal
// contiguous shares of the live tiles.  Up to kSfaLocalRows query rows every
// decode CTA derives its pair's share from the counts itself; above that the
// count kernel (one cluster) computes the prefix over rows and every share.  A
// piece of a sequence that a CTA boundary cuts goes to a partial slot (normalised
// O, running max M and sum L per head) and the combine kernel merges the pieces
// of every cut sequence.  The count kernel writes the zero rows of query rows
// with no live tile.
//
// Per CTA:
//  * resolver (warp 6): for each tile, the cache row of every position (index ->
//    block table, software-pipelined over three tiles) and the valid mask, into a
//    ring of kSfaRSlots resolved tiles.  A tile with no valid position is skipped
//    by every role below.
//  * producer (warp 0) and gatherers (warps 7-9): warp 0 loads Q of query row b
//    (9 column blocks of [q | q_rope], 128 rows, 147 KB, resident while b does not
//    change) by 3-D TMA tiles, the first row's before any tile is resolved and each
//    next one once the MMA issuer has released the buffer after the previous row's
//    last score MMAs; per tile, the 128 key rows (9 column blocks incl.
//    rope) and, one tile later, the 128 value rows of half h (4 blocks) go by TMA
//    tile::gather4 into a ring of 16 KB stages.  The four warps take eight of each
//    stage's 32 groups of 4 rows each (one warp alone cannot issue gathers fast
//    enough).  Invalid positions gather an out-of-range row (zero fill, no memory
//    traffic).  Every copy lands in this CTA's own shared memory.
//  * MMA issuer (warp 1): S_n[128 x 128] = Q K_n^T into one of two TMEM score
//    buffers (36 MMAs, M=128 N=128 K=16: the issuer's instruction stream is what
//    paces the kernel, and N=128 runs at the full tensor rate), then
//    O += P_{n-1} V_{n-1} with P from TMEM and V (MN-major) from shared memory, so
//    the scores of tile n are computed while the softmax warps work on tile n-1.
//  * softmax warps (2-5): thread = head row.  Masked scores in two passes of
//    32-column TMEM loads (maximum, then probabilities), running max; O is rescaled
//    (tcgen05.ld/st) only when the max grows by more than 8 in log2 units, so P
//    stays below 2^8; P goes as 16-bit pairs over the first half of its own score
//    buffer, into columns already read.
// Every wait is bounded; on a timeout the kernel records error bit 2, drains its
// copies and MMAs, frees TMEM and returns.
#include <atomic>

#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "decode.cuh"
#include "ptx.cuh"
#include "sfa.cuh"

namespace ifa {

namespace cg = cooperative_groups;

namespace {

__device__ __forceinline__ float ex2f_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// CTA whose tile range [floor(c W / P), floor((c+1) W / P)) holds global tile t.
__device__ __forceinline__ int cta_of_tile(long long t, long long W, int P) {
    return (int)(((t + 1) * (long long)P - 1) / W);
}

// CTA pairs that share W live tiles: at most the launch's P, and shares of at least
// min(tiles per sequence, kSfaMinShareTiles) tiles, so every one of them holds a tile.
__device__ __forceinline__ int active_ctas(long long W, int P, int tps) {
    const long long share = max(1, min(tps, kSfaMinShareTiles));
    const long long want = (W + share - 1) / share;
    return (int)max(1LL, min((long long)P, want));
}

__device__ __forceinline__ uint32_t pack2(float a, float b, bool bf) {
    if (bf) {
        __nv_bfloat162 v2 = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&v2);
    }
    __half2 v2 = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v2);
}

// Resolved tile in the resolver ring.
struct RSlot {
    int rows[kSfaTile];              // cache row of each position (total_rows = invalid)
    uint32_t vmask[kSfaTile / 32];   // valid positions, 32 per word
    int any;             // some position is valid
};
static_assert(sizeof(RSlot) <= kSfaRSlotBytes, "resolver slot");
constexpr int kPosPerLane = kSfaTile / 32;  // positions of a tile per resolver lane
struct LaneInts {
    int v[kPosPerLane];
};

// Next ring stage: position stg of round rnd (no division on the hot path).
__device__ __forceinline__ void ring_next(int& stg, uint32_t& rnd) {
    if (++stg == kSfaStages) {
        stg = 0;
        ++rnd;
    }
}

// Position in a pair's tile order: tile t of the n live tiles of query row r, whose first tile
// has index `first`.  Rows with no live tile are stepped over.
struct SeqCursor {
    int r, t, n;
    long long first;
    __device__ __forceinline__ void init(const SfaStart& s) {
        r = s.r;
        t = s.t;
        n = s.n;
        first = s.first;
    }
    __device__ __forceinline__ void next(const int* eff, int R) {
        if (++t < n) return;
        t = 0;
        first += n;
        n = 0;
        while (++r < R && (n = __ldcg(eff + r)) == 0) {
        }
    }
};

// Last entry of query row r's index row whose index selects a token, or -1 (one warp; lanes
// stride the row, whole 16-byte groups when the rows allow it).
__device__ __forceinline__ int row_last_usable(const SfaParams& p, int r, int lane) {
    const int idx_max = INT32_MAX >> p.sbs_log2;
    const int32_t* row = p.indices + (long long)r * p.S_sp;
    const bool vec = (p.S_sp & 3) == 0 && (reinterpret_cast<uintptr_t>(p.indices) & 15) == 0;
    int last = -1;
    if (vec) {
        const int4* row4 = reinterpret_cast<const int4*>(row);
        const int n4 = p.S_sp >> 2;
#pragma unroll 16
        for (int j = lane; j < n4; j += 32) {
            const int4 v = __ldg(row4 + j);
            if (v.x >= 0 && v.x <= idx_max) last = 4 * j;
            if (v.y >= 0 && v.y <= idx_max) last = 4 * j + 1;
            if (v.z >= 0 && v.z <= idx_max) last = 4 * j + 2;
            if (v.w >= 0 && v.w <= idx_max) last = 4 * j + 3;
        }
    } else {
#pragma unroll 8
        for (int i = lane; i < p.S_sp; i += 32) {
            const int idx = __ldg(row + i);
            if (idx >= 0 && idx <= idx_max) last = i;
        }
    }
    return __reduce_max_sync(0xffffffffu, last);
}

// Live tiles of a row whose last usable entry is `last`.
__device__ __forceinline__ int live_tiles(const SfaParams& p, int last) {
    return last < 0 ? 0 : (int)((((long long)last + 1) << p.sbs_log2) + kSfaTile - 1) / kSfaTile;
}

// A query row with no live tile: the decode kernel never visits it, so its output is all zero
// (largest score -inf, sum 0), written here by one warp.
__device__ __forceinline__ void write_empty_row(const SfaParams& p, int r, int lane) {
    uint4* o = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.out) + (long long)r * p.QN * kSfaD);
    for (int i = lane; i < p.QN * kSfaD / 8; i += 32) o[i] = make_uint4(0u, 0u, 0u, 0u);
    if (p.lse_max) {
        for (int i = lane; i < p.QN; i += 32) {
            p.lse_max[(long long)r * p.QN + i] = -INFINITY;
            p.lse_sum[(long long)r * p.QN + i] = 0.f;
        }
    }
}

// The share of pair c when every decode CTA derives the split itself (up to kSfaLocalRows query
// rows): the prefix of the live-tile counts over rows, the same equal contiguous shares as the
// tile-count kernel computes for more rows, and this pair's start.  The pair's first CTA also
// writes the piece record of every row whose first tile its share holds.  All threads; s_pre
// holds R + 1 ints, s_wsum one entry per warp and the total.
__device__ void local_split(const SfaParams& p, int* s_pre, long long* s_wsum, SfaStart* sst, int c,
                            bool write_pieces) {
    constexpr int NT = kSfaThreads, NW = kSfaThreads / 32;
    constexpr int kMaxChunk = (kSfaLocalRows + NT - 1) / NT;
    const int R = p.R;
    const int tid = (int)threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int chunk = (R + NT - 1) / NT;
    const int r0 = min(R, tid * chunk), r1 = min(R, r0 + chunk);
    int e[kMaxChunk];
    long long mine = 0;
#pragma unroll
    for (int k = 0; k < kMaxChunk; ++k) {
        e[k] = r0 + k < r1 ? __ldcg(p.eff + r0 + k) : 0;
        mine += e[k];
    }
    long long incl = mine;  // inclusive scan within the warp
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const long long v = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += v;
    }
    if (lane == 31) s_wsum[warp] = incl;
    __syncthreads();
    if (tid == 0) {
        long long run = 0;
        for (int w = 0; w < NW; ++w) {
            const long long v = s_wsum[w];
            s_wsum[w] = run;
            run += v;
        }
        s_wsum[NW] = run;
    }
    __syncthreads();
    long long run = s_wsum[warp] + incl - mine;  // exclusive prefix of this thread's rows
#pragma unroll
    for (int k = 0; k < kMaxChunk; ++k)
        if (r0 + k < r1) {
            s_pre[r0 + k] = (int)run;
            run += e[k];
        }
    const long long Wl = s_wsum[NW];
    if (tid == 0) s_pre[R] = (int)Wl;
    __syncthreads();
    const int Pa = active_ctas(Wl, p.P >> 1, p.tiles_per_seq);  // pairs from Pa on stay idle
    const int lo = c < Pa ? (int)(c * Wl / Pa) : 0;
    const int hi = c < Pa ? (int)((c + 1) * Wl / Pa) : 0;
    if (tid == 0) {
        SfaStart st;
        st.lo = lo;
        st.hi = hi;
        st.r = st.h = st.t = st.n = st.first = st.pad = 0;
        if (lo < hi) {
            // the last row with pre <= lo: a row with live tiles, since lo < the total
            int a = 0, z = R - 1;
            while (a < z) {
                const int mid = (a + z + 1) >> 1;
                if (s_pre[mid] <= lo) a = mid;
                else z = mid - 1;
            }
            st.r = a;
            st.n = s_pre[a + 1] - s_pre[a];
            st.t = lo - s_pre[a];
            st.first = s_pre[a];
        }
        *sst = st;
    }
    if (write_pieces && lo < hi) {
        for (int r = tid; r < R; r += NT) {
            const int g0 = s_pre[r], n = s_pre[r + 1] - g0;
            if (n > 0 && g0 >= lo && g0 < hi) {
                SfaPieces pc;
                pc.c_first = c;
                pc.np = cta_of_tile((long long)g0 + n - 1, Wl, Pa) - c + 1;
                pc.slot0 = g0 == lo ? 0 : 1;
                pc.pad = 0;
                p.pieces[r] = pc;
            }
        }
    }
}

}  // namespace

__global__ void __launch_bounds__(kSfaThreads, 1) sfa_kernel(const __grid_constant__ SfaParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sq = smem;                                   // [9][128 rows][128 B]
    uint8_t* ring = smem + kSfaQBytes;                    // [kSfaStages][kSfaTile rows][128 B]
    uint8_t* rbase = ring + kSfaStages * kSfaStageBytes;  // [kSfaRSlots] RSlot
    uint64_t* full = reinterpret_cast<uint64_t*>(rbase + kSfaRSlots * kSfaRSlotBytes);
    uint64_t* empty = full + kSfaStages;
    uint64_t* r_full = empty + kSfaStages;
    uint64_t* r_empty = r_full + kSfaRSlots;
    uint64_t* q_full = r_empty + kSfaRSlots;
    uint64_t* q_empty = q_full + 1;
    uint64_t* s_full = q_empty + 1;  // [2] scores of processed tile n in buffer n & 1
    uint64_t* p_full = s_full + 2;   // [2]
    uint64_t* o_full = p_full + 2;   // [2] P . V of processed tile n has completed
    uint64_t* done_bar = o_full + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    // this CTA's start, 16-byte aligned past the barriers, the TMEM address and the abort flag
    SfaStart* sst = reinterpret_cast<SfaStart*>(reinterpret_cast<uint8_t*>(full) + 384);
    static_assert(2 * kSfaStages * 8 + 2 * kSfaRSlots * 8 + 10 * 8 + 8 <= 384, "barrier area");
    static_assert(384 + sizeof(SfaStart) <= kSfaBarBytes, "barrier area");
    static_assert((kSfaQBytes + kSfaStages * kSfaStageBytes + kSfaRSlots * kSfaRSlotBytes) % 16 == 0, "alignment");

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // CTAs 2c and 2c + 1 form pair c: CTA 2c + h takes value half h of the pair's tiles
    const int h = (int)(blockIdx.x & 1);
    auto slot_of = [&](long long k) { return reinterpret_cast<RSlot*>(rbase + (int)(k % kSfaRSlots) * kSfaRSlotBytes); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kSfaStages; ++s) {
            mbar_init(&full[s], kSfaIssuers);
            mbar_init(&empty[s], 1);  // a stage is free once this CTA's MMAs have read it
        }
        for (int s = 0; s < kSfaRSlots; ++s) {
            mbar_init(&r_full[s], 1);
            mbar_init(&r_empty[s], kSfaIssuers + 5);  // gatherers, MMA issuer, four softmax warps
        }
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 4);
            mbar_init(&o_full[i], 1);
        }
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    // The start table and the live-tile counts come from the tile-count kernel (programmatic
    // dependent launch: everything above overlaps it).
    pdl_wait_primary();
    if (p.R <= kSfaLocalRows) {
        // the resolver slots serve as scratch until the roles start
        static_assert((kSfaLocalRows + 1) * sizeof(int) + (kSfaThreads / 32 + 1) * sizeof(long long) <=
                          kSfaRSlots * kSfaRSlotBytes, "split scratch");
        int* s_pre = reinterpret_cast<int*>(rbase);
        long long* s_wsum = reinterpret_cast<long long*>(rbase + ((kSfaLocalRows + 1) * sizeof(int) + 7) / 8 * 8);
        local_split(p, s_pre, s_wsum, sst, (int)(blockIdx.x >> 1), h == 0);
    } else if (threadIdx.x == 0) {
        const int4* src = reinterpret_cast<const int4*>(p.starts + (blockIdx.x >> 1));
        reinterpret_cast<int4*>(sst)[0] = __ldcg(src);
        reinterpret_cast<int4*>(sst)[1] = __ldcg(src + 1);
    }
    // barriers, the TMEM address and the start are in place before any role uses them
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const long long lo = sst->lo;
    const long long hi = sst->hi;
    const uint32_t tbase = *tmem_slot;
    const uint32_t O_T = tbase + 256;  // columns [256, 512): output accumulator
    // TMEM: two score buffers of kSfaTile columns at [0, 256); the softmax writes a tile's
    // probabilities (16-bit pairs, kSfaTile / 2 columns) over its own score buffer, into columns
    // it has already read; the output accumulator at [256, 512).
    auto S_T = [&](int buf) { return tbase + (uint32_t)kSfaTile * (uint32_t)buf; };
    auto P_T = [&](int buf) { return S_T(buf); };
    static_assert(2 * kSfaTile + kSfaHalf <= 512, "TMEM columns");

    if (warp == 6 && lo < hi) {
        // ================================================================ resolver
        // Three tiles in flight: the indices of tile g+2, the block-table entries and
        // length of tile g+1, and the rows of tile g.
        // token of position pos (-1 when its index is negative): index pos >> sbs_log2 selects
        // the tokens index << sbs_log2 .. + (1 << sbs_log2) - 1 (token-wise when sbs_log2 = 0)
        const int npos = p.S_sp << p.sbs_log2;
        const int smask = (1 << p.sbs_log2) - 1;
        // tokens of positions lane + 32 u of tile g (u < kPosPerLane), -1 where none
        auto load_idx = [&](long long g, const SeqCursor& c) {
            LaneInts tok;
#pragma unroll
            for (int u = 0; u < kPosPerLane; ++u) tok.v[u] = -1;
            if (g >= hi) return tok;
            const int32_t* row = p.indices + (long long)c.r * p.S_sp;
#pragma unroll
            for (int u = 0; u < kPosPerLane; ++u) {
                const int pos = c.t * kSfaTile + lane + 32 * u;
                if (pos < npos) {
                    const int idx = __ldg(row + (pos >> p.sbs_log2));
                    if (idx >= 0 && idx <= (INT32_MAX >> p.sbs_log2)) tok.v[u] = (idx << p.sbs_log2) + (pos & smask);
                }
            }
            return tok;
        };
        // block-table entry of token idx of batch b (read only when it lies inside the table), -1 otherwise
        auto load_blk = [&](int b, int idx) -> int {
            if (idx < 0 || idx / p.block_size >= p.bt_cols) return -1;
            return __ldg(p.block_table + (long long)b * p.bt_cols + idx / p.block_size);
        };
        // TND query rows: the batch of a row is the first whose prefix sum exceeds it.  Rows only
        // rise within a CTA's range, so a binary search places the first and the rest step on.
        const bool paged = p.kv_layout == 0;
        int tnd_b = 0;
        SeqCursor c0, c1, c2;  // tiles g, g + 1, g + 2
        c0.init(*sst);
        c1 = c0;
        c1.next(p.eff, p.R);
        c2 = c1;
        c2.next(p.eff, p.R);
        if (p.q_tnd) {
            const int r_first = c0.r;
            int a = 0, z = p.B;  // first b in [a, z] with lens_q[b] > r_first (z = B: none)
            while (a < z) {
                const int mid = (a + z) >> 1;
                if (__ldg(p.lens_q + mid) > r_first) z = mid;
                else a = mid + 1;
            }
            tnd_b = a;
        }
        // Batch of query row r (-1: none), the keys it may use ([0, limit): rows past the
        // batch's valid query tokens use none; under the right-down causal mode token s sits at
        // key len - qlen + s), and the batch's first key row (BSND and TND key layouts).
        auto row_info = [&](int r, int& b, int& limit, int& base) {
            int s, qlen;
            b = -1;
            limit = 0;
            base = 0;
            if (p.q_tnd) {
                while (tnd_b < p.B && __ldg(p.lens_q + tnd_b) <= r) ++tnd_b;
                if (tnd_b >= p.B) return;
                const int first = tnd_b > 0 ? __ldg(p.lens_q + tnd_b - 1) : 0;
                b = tnd_b;
                s = r - first;
                qlen = __ldg(p.lens_q + tnd_b) - first;
            } else {
                b = r / p.QS;
                s = r - b * p.QS;
                qlen = p.lens_q ? __ldg(p.lens_q + b) : p.QS;
            }
            long long len, avail = INT32_MAX;
            if (paged) {
                len = __ldg(p.lens + b);
            } else if (p.kv_layout == 1) {
                len = p.lens ? __ldg(p.lens + b) : p.kv_s;
                base = b * p.kv_s;  // < 2^31: the host checks B * KV_S
                avail = p.kv_s;
            } else {
                base = b > 0 ? __ldg(p.lens + b - 1) : 0;
                len = (long long)__ldg(p.lens + b) - base;
                avail = (long long)p.kv_s - base;
                if (base < 0) avail = 0;  // a malformed prefix: nothing to read
            }
            long long lim = len;
            if (s >= qlen) lim = 0;
            else if (p.causal) lim = len - qlen + s + 1;  // <= len since s < qlen
            if (lim > avail) lim = avail;
            limit = lim < 0 ? 0 : (int)lim;
        };
        LaneInts i0 = load_idx(lo, c0), i1 = load_idx(lo + 1, c1), bt0, bt1;
        int b0, len0, base0;
        row_info(c0.r, b0, len0, base0);
#pragma unroll
        for (int u = 0; u < kPosPerLane; ++u) bt0.v[u] = paged && b0 >= 0 ? load_blk(b0, i0.v[u]) : -1;
        long long k = 0;
        for (long long g = lo; g < hi; ++g, ++k) {
            const LaneInts i2 = load_idx(g + 2, c2);
            int b1 = -1, len1 = 0, base1 = 0;
#pragma unroll
            for (int u = 0; u < kPosPerLane; ++u) bt1.v[u] = -1;
            if (g + 1 < hi) {
                row_info(c1.r, b1, len1, base1);
                if (paged && b1 >= 0) {
#pragma unroll
                    for (int u = 0; u < kPosPerLane; ++u) bt1.v[u] = load_blk(b1, i1.v[u]);
                }
            }
            // rows of tile g: invalid (total_rows) outside [0, limit); bad block-table entries are flagged
            int rows2[kPosPerLane];
            bool bad = false;
#pragma unroll
            for (int u = 0; u < kPosPerLane; ++u) {
                const int idx = i0.v[u];
                const int blk = bt0.v[u];
                int r = p.total_rows;
                if (idx >= 0 && idx < len0) {
                    if (!paged) r = base0 + idx;  // < total_rows: the limit stops at the tensor's end
                    else if (blk < 0 || blk >= p.block_num) bad = true;  // includes a length beyond the block table
                    else r = blk * p.block_size + idx % p.block_size;
                }
                rows2[u] = r;
            }
            if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(p.err, kErrBadBlock);
            uint32_t vm[kPosPerLane];
#pragma unroll
            for (int u = 0; u < kPosPerLane; ++u) vm[u] = __ballot_sync(0xffffffffu, rows2[u] != p.total_rows);
            const int slot = (int)(k % kSfaRSlots);
            const uint32_t round = (uint32_t)(k / kSfaRSlots);
            if (round > 0 && !mbar_wait_bounded(&r_empty[slot], (round - 1) & 1, kWaitLimitNs)) {
                if (lane == 0) atomicOr(p.err, kErrTimeout);
                *abort_flag = 1;
                break;
            }
            RSlot* rs = slot_of(k);
            uint32_t any = 0;
#pragma unroll
            for (int u = 0; u < kPosPerLane; ++u) {
                rs->rows[lane + 32 * u] = rows2[u];
                any |= vm[u];
            }
            if (lane == 0) {
#pragma unroll
                for (int u = 0; u < kPosPerLane; ++u) rs->vmask[u] = vm[u];
                rs->any = any != 0;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&r_full[slot]);
            i0 = i1;
            i1 = i2;
            bt0 = bt1;
            b0 = b1;
            len0 = len1;
            base0 = base1;
            c0 = c1;
            c1 = c2;
            c2.next(p.eff, p.R);
            if (*abort_flag) break;
        }
    } else if ((warp == 0 || warp >= 7) && lo < hi) {
        // ================================================================ producer and gatherers
        const int gi = warp == 0 ? 0 : warp - 6;  // this warp's quarter of each stage's row groups
        if (lane == 0 && gi == 0) {
            prefetch_tensormap(&p.tmQ);
            prefetch_tensormap(&p.tmQr);
            prefetch_tensormap(&p.tmK);
            prefetch_tensormap(&p.tmKr);
            prefetch_tensormap(&p.tmV);
            if (p.sbs_log2 >= 3) {
                prefetch_tensormap(&p.tmKb);
                prefetch_tensormap(&p.tmKrb);
                prefetch_tensormap(&p.tmVb);
            }
        }
        // value rows are read once; key rows twice, by both CTAs of the pair, so they keep the
        // default L2 priority for the second read
        const uint64_t pol_v = policy_evict_first();
        const uint64_t pol_k = policy_evict_normal();
        long long it = 0;
        int stg = 0;  // ring position of stage `it`: stg = it mod kSfaStages, rnd = it / kSfaStages
        uint32_t rnd = 0;
        int epoch = 0;
        int prev_b = -1;
        bool ok = true;
        if (gi == 0) {
            // the first row's query: its row is in the start record, so it need not wait for the
            // first resolved tile (index and block-table loads)
            prev_b = sst->r;
            if (lane == 0) {
                mbar_arrive_expect_tx(q_full, kSfaQBytes);
                for (int kb = 0; kb < 8; ++kb) tma_load_3d(sq + kb * 16384, &p.tmQ, q_full, kb * 64, 0, prev_b);
                tma_load_3d(sq + 8 * 16384, &p.tmQr, q_full, 0, 0, prev_b);
            }
            epoch = 1;
        }
        // Gathers column blocks [blk0, blk0 + nblk) of the rows of resolved tile `rs` (blocks
        // 0..7: key, 8: key rope, 9..12: value half h) into this CTA's ring.
        constexpr int kGroups = kSfaTile / 4 / kSfaIssuers;  // gather4 row groups per warp and stage
        // Block-wise selections of 8 or more tokens are runs of consecutive cache rows: one tiled
        // box of run_rows rows per run (or per 64-row half of a 128-token run) instead of gathers.
        const bool runs = p.sbs_log2 >= 3;
        const int run_rows = runs ? min(1 << p.sbs_log2, kSfaTile) : 0;
        const int nruns = runs ? kSfaTile / run_rows : 0;  // boxes per stage: 16, 8, 4, 2 or 1
        int my_runs = 0;                                    // this warp takes runs gi, gi + 4, ...
        for (int k = gi; k < nruns; k += kSfaIssuers) ++my_runs;
        auto gather = [&](const RSlot* rs, int blk0, int nblk) {
            const int grp = gi * kGroups + lane;
            const int4 r4 = lane < kGroups ? reinterpret_cast<const int4*>(rs->rows)[grp] : make_int4(0, 0, 0, 0);
            for (int blk = blk0; blk < blk0 + nblk; ++blk, ++it, ring_next(stg, rnd)) {
                const int stage = stg;
                const uint32_t round = rnd;
                if (round > 0 && !mbar_wait_bounded(&empty[stage], (round - 1) & 1, kWaitLimitNs)) {
                    if (lane == 0) atomicOr(p.err, kErrTimeout);
                    *abort_flag = 1;
                    ok = false;
                    return;
                }
                if (runs) {
                    if (lane == 0) mbar_arrive_expect_tx(&full[stage], (uint32_t)(my_runs * run_rows * 128));
                    __syncwarp();
                    const int k = gi + kSfaIssuers * lane;  // run this lane loads
                    if (lane < my_runs) {
                        const CUtensorMap* map;
                        int x;
                        if (blk < 8) {
                            map = &p.tmKb;
                            x = blk * 64;
                        } else if (blk == 8) {
                            map = &p.tmKrb;
                            x = 0;
                        } else {
                            map = &p.tmVb;
                            x = h * kSfaHalf + (blk - kSfaQBlocks) * 64;
                        }
                        // the run's first row; an invalid run starts past the last row (zero fill)
                        uint8_t* dst = ring + stage * kSfaStageBytes + k * run_rows * 128;
                        tma_load_2d(dst, map, &full[stage], x, rs->rows[k * run_rows]);
                    }
                    __syncwarp();
                    continue;
                }
                if (lane == 0) mbar_arrive_expect_tx(&full[stage], kSfaStageBytes / kSfaIssuers);
                __syncwarp();
                if (lane < kGroups) {
                    const CUtensorMap* map;
                    int x;
                    if (blk < 8) {
                        map = &p.tmK;
                        x = blk * 64;
                    } else if (blk == 8) {
                        map = &p.tmKr;
                        x = 0;
                    } else {
                        map = &p.tmV;
                        x = h * kSfaHalf + (blk - kSfaQBlocks) * 64;
                    }
                    uint8_t* dst = ring + stage * kSfaStageBytes + grp * 512;
                    tma_gather4(dst, map, &full[stage], x, r4.x, r4.y, r4.z, r4.w, blk < kSfaQBlocks ? pol_k : pol_v);
                }
                __syncwarp();
            }
        };
        long long pend = -1;  // resolved tile whose value rows are still to be gathered
        auto flush = [&]() {
            if (pend < 0) return;
            gather(slot_of(pend), kSfaQBlocks, kSfaVBlocks);
            __syncwarp();
            if (lane == 0) mbar_arrive(&r_empty[(int)(pend % kSfaRSlots)]);
            pend = -1;
        };
        long long k = 0;
        SeqCursor cur;
        cur.init(*sst);
        for (long long g = lo; g < hi && ok && !*abort_flag; ++g, ++k, cur.next(p.eff, p.R)) {
            const int slot = (int)(k % kSfaRSlots);
            if (!mbar_wait_bounded(&r_full[slot], (uint32_t)(k / kSfaRSlots) & 1, kWaitLimitNs)) {
                if (lane == 0) atomicOr(p.err, kErrTimeout);
                *abort_flag = 1;
                break;
            }
            const RSlot* rs = slot_of(k);
            const int b = cur.r;  // query row
            if (!rs->any) {
                flush();
                __syncwarp();
                if (lane == 0) mbar_arrive(&r_empty[slot]);
                continue;
            }
            if (b != prev_b && gi == 0) {  // new query row: wait until the MMAs using the old query are done
                if (epoch > 0 && !mbar_wait_bounded(q_empty, (epoch - 1) & 1, kWaitLimitNs)) {
                    if (lane == 0) atomicOr(p.err, kErrTimeout);
                    *abort_flag = 1;
                    break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(q_full, kSfaQBytes);
                    for (int kb = 0; kb < 8; ++kb) tma_load_3d(sq + kb * 16384, &p.tmQ, q_full, kb * 64, 0, b);
                    tma_load_3d(sq + 8 * 16384, &p.tmQr, q_full, 0, 0, b);
                }
                ++epoch;
            }
            prev_b = b;
            gather(rs, 0, kSfaQBlocks);
            if (!ok) break;
            flush();
            pend = k;
        }
        if (ok && !*abort_flag) flush();
        // Let every issued copy land before shared memory can be released.
        if (lane == 0) {
            for (long long j = (it > kSfaStages ? it - kSfaStages : 0); j < it; ++j)
                mbar_wait_bounded(&full[j % kSfaStages], (uint32_t)(j / kSfaStages) & 1, kWaitLimitNs);
            if (epoch > 0) mbar_wait_bounded(q_full, (epoch - 1) & 1, kWaitLimitNs);
        }
    } else if (warp == 1 && lo < hi) {
        // ================================================================ MMA issuer
        if (lane == 0) {
            const bool bf = p.is_bf16 != 0;
            const uint32_t idesc_qk = umma_idesc(bf, false, 128, kSfaTile);
            const uint32_t idesc_pv = umma_idesc(bf, true, 128, 64);
            const uint32_t sq_addr = smem_u32(sq);
            const uint32_t ring_addr = smem_u32(ring);
            long long it = 0;
            int epoch = 0;             // query loads waited for
            int prev_b = sst->r;       // row of the query in place (the producer loads the first at once)
            bool q_waited = false;     // that query has been waited for
            int n = 0;             // processed (non-empty) tiles so far
            int pending = -1;      // processed tile whose P . V is still to be issued
            uint32_t pend_acc = 0;
            bool fresh = true;     // no processed tile yet in the current piece
            bool q_freed = false;  // the query blocks were released after the current row's last scores
            bool ok = true;
            int stg = 0;        // ring position of stage `it`: stg = it mod kSfaStages, rnd = it / kSfaStages
            uint32_t rnd = 0;
            auto wait_stage = [&]() -> int {
                const int stage = stg;
                if (!mbar_wait_bounded(&full[stage], rnd & 1, kWaitLimitNs)) {
                    ok = false;
                    return -1;
                }
                tc_fence_after();
                return stage;
            };
            auto do_pv = [&](int m, uint32_t acc) {
                if (!mbar_wait_bounded(&p_full[m & 1], (uint32_t)(m >> 1) & 1, kWaitLimitNs)) {
                    ok = false;
                    return;
                }
                tc_fence_after();
                for (int vb = 0; vb < kSfaVBlocks; ++vb, ++it, ring_next(stg, rnd)) {
                    const int stage = wait_stage();
                    if (stage < 0) return;
#pragma unroll
                    for (int k = 0; k < kSfaTile / 16; ++k) {
                        const uint64_t bd = umma_sdesc(ring_addr + stage * kSfaStageBytes + k * 2048, 8192, 1024);
                        umma_ts(O_T + vb * 64, P_T(m & 1) + k * 8, bd, idesc_pv, (acc != 0 || k > 0) ? 1u : 0u);
                    }
                    umma_commit(&empty[stage]);
                }
                umma_commit(&o_full[m & 1]);
            };
            long long kk = 0;
            SeqCursor cur;
            cur.init(*sst);
            for (long long g = lo; g < hi && ok; ++g, ++kk, cur.next(p.eff, p.R)) {
                const int b = cur.r;  // query row
                if (cur.t == 0 || g == lo) fresh = true;
                const int slot = (int)(kk % kSfaRSlots);
                if (!mbar_wait_bounded(&r_full[slot], (uint32_t)(kk / kSfaRSlots) & 1, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                const int any = slot_of(kk)->any;
                mbar_arrive(&r_empty[slot]);
                if (!any) {
                    if (pending >= 0) do_pv(pending, pend_acc);
                    pending = -1;
                    continue;
                }
                if (b != prev_b) {
                    // the query in place may never have been used (its row's tiles here were all
                    // empty): it must have landed before the producer overwrites it
                    if (!q_waited) {
                        if (!mbar_wait_bounded(q_full, epoch & 1, kWaitLimitNs)) {
                            ok = false;
                            break;
                        }
                        ++epoch;
                    }
                    if (!q_freed) umma_commit(q_empty);
                    q_freed = false;
                    q_waited = false;
                    prev_b = b;
                }
                if (!q_waited) {
                    if (!mbar_wait_bounded(q_full, epoch & 1, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    ++epoch;
                    q_waited = true;
                }
                tc_fence_after();
                // ---- S_n = [q | q_rope] . [k | k_rope]^T
                for (int kb = 0; kb < kSfaQBlocks; ++kb, ++it, ring_next(stg, rnd)) {
                    const int stage = wait_stage();
                    if (stage < 0) break;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint64_t ad = umma_sdesc(sq_addr + kb * 16384 + k * 32, 16, 1024);
                        const uint64_t bd = umma_sdesc(ring_addr + stage * kSfaStageBytes + k * 32, 16, 1024);
                        umma_ss(S_T(n & 1), ad, bd, idesc_qk, (kb | k) != 0);
                    }
                    umma_commit(&empty[stage]);
                }
                if (!ok) break;
                umma_commit(&s_full[n & 1]);
                // The row's last tile: once these score MMAs finish, the query blocks may take the
                // next row's query, which then lands while this row's last P . V waits for its
                // probabilities.
                if (cur.t + 1 >= cur.n && g + 1 < hi) {
                    umma_commit(q_empty);
                    q_freed = true;
                }
                // ---- O += P_{n-1} . V_{n-1} while the softmax warps work on S_n
                if (pending >= 0) do_pv(pending, pend_acc);
                pending = n;
                pend_acc = fresh ? 0u : 1u;
                fresh = false;
                ++n;
            }
            if (ok && pending >= 0) do_pv(pending, pend_acc);
            if (!ok) {
                atomicOr(p.err, kErrTimeout);
                *abort_flag = 1;
            }
            // every MMA issued so far has completed once done_bar flips
            umma_commit(done_bar);
            mbar_wait_bounded(done_bar, 0, kWaitLimitNs);
        }
        __syncwarp();
    } else if (warp >= 2 && warp < 6 && lo < hi) {
        // ================================================================ softmax warps
        const int quad = warp & 3;                 // TMEM lane quadrant this warp may access
        const int row = quad * 32 + lane;          // query head of this thread
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const bool bf = p.is_bf16 != 0;
        float m_used = -INFINITY, l_sum = 0.f;
        float m_top = -INFINITY;  // largest scaled score of the piece (m_used may trail it by the slack)
        int n = 0;        // processed tiles so far
        int n_last = -1;  // last processed tile of the current piece
        auto fail = [&]() {
            if (lane == 0) atomicOr(p.err, kErrTimeout);
            *abort_flag = 1;
        };
        long long kk = 0;
        SeqCursor cur;
        cur.init(*sst);
        for (long long g = lo; g < hi; ++g, ++kk, cur.next(p.eff, p.R)) {
            const int b = cur.r;  // query row
            if (cur.t == 0 || g == lo) {
                m_used = -INFINITY;
                m_top = -INFINITY;
                l_sum = 0.f;
                n_last = -1;
            }
            const int slot = (int)(kk % kSfaRSlots);
            if (!mbar_wait_bounded(&r_full[slot], (uint32_t)(kk / kSfaRSlots) & 1, kWaitLimitNs)) {
                fail();
                break;
            }
            const RSlot* rs = slot_of(kk);
            const int any = rs->any;
            if (!any) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&r_empty[slot]);
            }
            if (any) {
                if (!mbar_wait_bounded(&s_full[n & 1], (uint32_t)(n >> 1) & 1, kWaitLimitNs)) {
                    fail();
                    break;
                }
                tc_fence_after();
                const uint32_t S0 = S_T(n & 1) + lane_off;
                // pass 1: the tile's largest scaled score over its valid positions (the valid mask
                // stays in the resolver slot until pass 2 has read it)
                float tmax = -INFINITY;
#pragma unroll 1
                for (int c = 0; c < kSfaTile / 32; ++c) {
                    uint32_t sa[32];
                    tmem_ld32(S0 + 32 * c, sa);
                    const uint32_t vmc = rs->vmask[c];
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if ((vmc >> j) & 1) tmax = fmaxf(tmax, __uint_as_float(sa[j]) * p.scale_log2);
                }
                m_top = fmaxf(m_top, tmax);
                const float m_new = fmaxf(m_used, tmax);
                const bool need = m_new > m_used + kSfaRescaleSlack;  // also true when m_used = -inf < m_new
                if (__any_sync(0xffffffffu, need)) {
                    const float alpha = need ? (m_used == -INFINITY ? 0.f : ex2f_approx(m_used - m_new)) : 1.f;
                    if (n_last >= 0) {
                        // O holds this piece's earlier tiles: rescale it once P_{n-1} . V_{n-1} is in
                        if (!mbar_wait_bounded(&o_full[(n - 1) & 1], (uint32_t)((n - 1) >> 1) & 1, kWaitLimitNs)) {
                            fail();
                            break;
                        }
                        tc_fence_after();
                        for (int c = 0; c < kSfaHalf / 32; ++c) {
                            uint32_t o[32];
                            tmem_ld32(O_T + lane_off + c * 32, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                            tmem_st32(O_T + lane_off + c * 32, o);
                        }
                        tmem_wait_st();
                    }
                    if (need) {
                        l_sum *= alpha;
                        m_used = m_new;
                    }
                }
                // P buffer n & 1 is free once P_{n-2} . V_{n-2} has completed
                if (n >= 2) {
                    if (!mbar_wait_bounded(&o_full[n & 1], (uint32_t)((n - 2) >> 1) & 1, kWaitLimitNs)) {
                        fail();
                        break;
                    }
                    tc_fence_after();
                }
                const float m_use = m_used == -INFINITY ? 0.f : m_used;
                // pass 2: probabilities as 16-bit pairs (column m: positions 2m, 2m + 1), written
                // over the score buffer 32 columns at a time after the 64 scores they replace
                // have been read
#pragma unroll 1
                for (int c2 = 0; c2 < kSfaTile / 64; ++c2) {
                    uint32_t pk[32];
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const int c = 2 * c2 + h2;
                        uint32_t sa[32];
                        tmem_ld32(S0 + 32 * c, sa);
                        const uint32_t vmc = rs->vmask[c];
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const float x0 = ((vmc >> (2 * j)) & 1) ? __uint_as_float(sa[2 * j]) * p.scale_log2 : -INFINITY;
                            const float x1 =
                                ((vmc >> (2 * j + 1)) & 1) ? __uint_as_float(sa[2 * j + 1]) * p.scale_log2 : -INFINITY;
                            const float p0 = ex2f_approx(x0 - m_use);
                            const float p1 = ex2f_approx(x1 - m_use);
                            l_sum += p0 + p1;
                            pk[16 * h2 + j] = pack2(p0, p1, bf);
                        }
                    }
                    tmem_st32(P_T(n & 1) + lane_off + 32 * c2, pk);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&r_empty[slot]);  // the slot's last read was above
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[n & 1]);
                n_last = n;
                ++n;
            }
            const bool last = (cur.t == cur.n - 1) || (g == hi - 1);
            if (!last) continue;
            // ============================================================ piece epilogue
            const long long seq_first = cur.first;
            const bool complete = seq_first >= lo && seq_first + cur.n <= hi;
            const long long orow = ((long long)b * p.QN + row) * kSfaD + h * kSfaHalf;
            const int slot_p = 2 * (int)blockIdx.x + (seq_first <= lo ? 0 : 1);
            float* sp = p.partials + (long long)slot_p * kSfaSlotFloats;
            const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
            if (n_last >= 0) {
                if (!mbar_wait_bounded(&o_full[n_last & 1], (uint32_t)(n_last >> 1) & 1, kWaitLimitNs)) {
                    fail();
                    break;
                }
                tc_fence_after();
            }
            for (int c = 0; c < kSfaHalf / 32; ++c) {
                uint32_t o[32];
                if (n_last >= 0) {
                    tmem_ld32(O_T + lane_off + c * 32, o);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] = 0u;  // empty selection: all-zero row
                }
                if (complete) {
                    if (row < p.QN) {
                        uint32_t w[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            w[j] = pack2(__uint_as_float(o[2 * j]) * inv, __uint_as_float(o[2 * j + 1]) * inv, bf);
                        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.out) + orow + c * 32);
#pragma unroll
                        for (int j = 0; j < 4; ++j) dst[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
                    }
                } else {
                    // slot layout [channel quad][head row]: the warp's 32 rows store 512
                    // contiguous bytes per instruction
                    float4* dst = reinterpret_cast<float4*>(sp) + c * 8 * 128 + row;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        dst[j * 128] = make_float4(__uint_as_float(o[4 * j]) * inv, __uint_as_float(o[4 * j + 1]) * inv,
                                             __uint_as_float(o[4 * j + 2]) * inv, __uint_as_float(o[4 * j + 3]) * inv);
                }
            }
            tc_fence_before();
            if (!complete) {
                sp[128 * kSfaHalf + row] = m_used;
                sp[128 * kSfaHalf + 128 + row] = l_sum;
                sp[128 * kSfaHalf + 256 + row] = m_top;
            } else if (p.lse_max && h == 0 && row < p.QN) {
                // the largest score and the sum of exp(score - it), in natural units: the scores
                // here are log2(e) * scale * q.k
                const long long li = (long long)b * p.QN + row;
                p.lse_max[li] = m_top == -INFINITY ? -INFINITY : m_top * kLn2;
                p.lse_sum[li] = m_top == -INFINITY ? 0.f : l_sum * ex2f_approx(m_used - m_top);
            }
        }
    }
    // ==================================================================== teardown
    // Every role is done with TMEM (the MMA issuer has waited for all its MMAs and so for
    // their commits) before it is freed.
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tbase, 512);
}

// Per query row: its live tiles, up to the last tile that holds a usable index (tiles past it
// hold only invalid positions), and, by the cluster's first CTA after a cluster barrier, the
// prefix over rows and the start of each CTA pair of the decode kernel: equal contiguous
// shares of the live tiles (each pair runs its tiles once per value half).  One cluster of kSfaCountCtas CTAs; warp = row.  Up to
// kSfaCountSmemRows rows, each warp also stores its row's count into the first CTA's shared
// memory, which then scans and searches there; beyond that the first CTA reads global memory.
__global__ void __launch_bounds__(kSfaCountThreads) sfa_count(const __grid_constant__ SfaParams p) {
    __shared__ int s_eff[kSfaCountSmemRows];
    __shared__ int s_pre[kSfaCountSmemRows + 1];
    __shared__ long long wsum[kSfaCountThreads / 32];
    __shared__ long long total;
    pdl_launch_dependents();  // the decode kernel's prologue may start; it waits for this grid's end
    cg::cluster_group cluster = cg::this_cluster();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int NW = kSfaCountThreads / 32;
    const int R = p.R;
    const bool in_smem = R <= kSfaCountSmemRows;
    int* eff0 = cluster.map_shared_rank(s_eff, 0);  // the first CTA's copy
    for (int r = blockIdx.x * NW + warp; r < R; r += gridDim.x * NW) {
        const int last = row_last_usable(p, r, lane);
        if (lane == 0) {
            const int e = live_tiles(p, last);
            p.eff[r] = e;
            if (in_smem) eff0[r] = e;
        }
        if (last < 0) write_empty_row(p, r, lane);
    }

    __threadfence();
    cluster.sync();
    if (blockIdx.x != 0) return;
    auto eff_of = [&](int r) { return in_smem ? s_eff[r] : __ldcg(p.eff + r); };
    // prefix over rows: thread k sums its contiguous chunk, a block scan places the chunks
    const int chunk = (R + kSfaCountThreads - 1) / kSfaCountThreads;
    const int r0 = min(R, (int)threadIdx.x * chunk), r1 = min(R, r0 + chunk);
    long long mine = 0;
    for (int r = r0; r < r1; ++r) mine += eff_of(r);
    long long incl = mine;  // inclusive scan within the warp
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const long long v = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += v;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (threadIdx.x == 0) {
        long long run = 0;
        for (int w = 0; w < NW; ++w) {
            const long long v = wsum[w];
            wsum[w] = run;
            run += v;
        }
        total = run;
    }
    __syncthreads();
    long long run = wsum[warp] + incl - mine;  // exclusive prefix of this thread's chunk
    for (int r = r0; r < r1; ++r) {
        if (in_smem) s_pre[r] = (int)run;
        p.pre[r] = (int)run;
        run += eff_of(r);
    }
    if (threadIdx.x == 0) {
        p.pre[R] = (int)total;
        if (in_smem) s_pre[R] = (int)total;
    }
    __syncthreads();
    auto pre_of = [&](int r) { return in_smem ? s_pre[r] : p.pre[r]; };
    // each pair's share [lo, hi) and where it begins: the last row r < R with pre[r] <= lo (a row
    // with live tiles, since lo < total)
    const long long Wl = total;
    const int pairs = p.P >> 1;
    const int Pa = active_ctas(Wl, pairs, p.tiles_per_seq);  // pairs from Pa on stay idle
    for (int c = threadIdx.x; c < pairs; c += kSfaCountThreads) {
        SfaStart st;
        st.lo = c < Pa ? (int)(c * Wl / Pa) : 0;
        st.hi = c < Pa ? (int)((c + 1) * Wl / Pa) : 0;
        st.r = st.h = st.t = st.n = st.first = st.pad = 0;
        if (st.lo < st.hi) {
            int a = 0, z = R - 1;
            while (a < z) {
                const int mid = (a + z + 1) >> 1;
                if (pre_of(mid) <= st.lo) a = mid;
                else z = mid - 1;
            }
            st.r = a;
            st.n = eff_of(a);
            st.t = st.lo - pre_of(a);
            st.first = pre_of(a);
        }
        p.starts[c] = st;
    }
    // for the combine kernel: where each row's pieces sit (one record instead of a search)
    for (int r = threadIdx.x; r < R; r += kSfaCountThreads) {
        const long long g0 = pre_of(r);
        const int n = eff_of(r);
        SfaPieces pc;
        pc.c_first = pc.np = pc.slot0 = pc.pad = 0;
        if (n > 0) {
            pc.c_first = cta_of_tile(g0, Wl, Pa);
            pc.np = cta_of_tile(g0 + n - 1, Wl, Pa) - pc.c_first + 1;
            pc.slot0 = g0 <= (long long)pc.c_first * Wl / Pa ? 0 : 1;
        }
        p.pieces[r] = pc;
    }
}

// Per query row, up to kSfaLocalRows rows: its live tiles (the decode CTAs derive the split from
// them), and for a row without one the all-zero output and an empty piece record.  One warp per
// row and few rows per CTA, so that the index rows spread over many SMs.
__global__ void __launch_bounds__(kSfaRowCountWarps * 32) sfa_count_rows(const __grid_constant__ SfaParams p) {
    pdl_launch_dependents();  // the decode kernel's prologue may start; it waits for this grid's end
    const int lane = (int)threadIdx.x & 31;
    const int r = (int)blockIdx.x * kSfaRowCountWarps + ((int)threadIdx.x >> 5);
    if (r >= p.R) return;
    const int last = row_last_usable(p, r, lane);
    if (lane == 0) {
        p.eff[r] = live_tiles(p, last);
        if (last < 0) {
            SfaPieces pc;
            pc.c_first = pc.np = pc.slot0 = pc.pad = 0;
            p.pieces[r] = pc;
        }
    }
    if (last < 0) write_empty_row(p, r, lane);
}

// Merges the pieces of every sequence that CTA boundaries cut, for problems whose shares average
// four tiles or more (rows of a few pieces): grid (2R sequences, 16 blocks of 8 head rows), 128
// threads; thread = (head row, 16 channels).  Piece k weighs
// L_k 2^(M_k - M) / sum_j L_j 2^(M_j - M) with M the largest M_k.  One record from the count
// kernel says where the pieces sit; then every piece's M, L and channels are loaded at once.
__global__ void __launch_bounds__(128) sfa_combine_few(const __grid_constant__ SfaParams p) {
    constexpr int kCh = 16;                          // channels per thread
    constexpr int kTpr = kSfaHalf / kCh;             // threads per head row
    constexpr int kMaxFast = 4;                      // pieces loaded together
    const int s = blockIdx.x;
    const int b = s >> 1, h = s & 1;
    const SfaPieces pc = p.pieces[b];
    if (pc.np < 2) return;  // the count kernel or the decode kernel wrote this sequence
    // rows vary fastest across the threads: a slot holds channel quads of consecutive head rows
    const int row = blockIdx.y * (128 / kTpr) + (int)threadIdx.x % (128 / kTpr);
    const int col0 = ((int)threadIdx.x / (128 / kTpr)) * kCh;
    if (row >= p.QN) return;
    const int np = pc.np;
    // pairs c_first .. c_first + np - 1 hold the row's tiles; CTA 2c + h of pair c value half h
    auto slot_ptr = [&](int k) {
        const int sl = k == 0 ? 2 * (2 * pc.c_first + h) + pc.slot0 : 2 * (2 * (pc.c_first + k) + h);
        return p.partials + (long long)sl * kSfaSlotFloats;
    };
    float acc[kCh];
#pragma unroll
    for (int j = 0; j < kCh; ++j) acc[j] = 0.f;
    float S = 0.f;
    if (np <= kMaxFast) {
        float m[kMaxFast], l[kMaxFast];
        float4 v[kMaxFast][kCh / 4];
#pragma unroll
        for (int k = 0; k < kMaxFast; ++k) {
            m[k] = -INFINITY;
            l[k] = 0.f;
            if (k < np) {
                const float* pp = slot_ptr(k);
                m[k] = __ldcg(pp + 128 * kSfaHalf + row);
                l[k] = __ldcg(pp + 128 * kSfaHalf + 128 + row);
#pragma unroll
                for (int j = 0; j < kCh / 4; ++j)
                    v[k][j] = __ldcg(reinterpret_cast<const float4*>(pp) + (col0 / 4 + j) * 128 + row);
            } else {
#pragma unroll
                for (int j = 0; j < kCh / 4; ++j) v[k][j] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        float M = m[0];
#pragma unroll
        for (int k = 1; k < kMaxFast; ++k) M = fmaxf(M, m[k]);
#pragma unroll
        for (int k = 0; k < kMaxFast; ++k) {
            const float w = m[k] == -INFINITY ? 0.f : l[k] * ex2f_approx(m[k] - M);
            S += w;
#pragma unroll
            for (int j = 0; j < kCh / 4; ++j) {
                acc[4 * j] += w * v[k][j].x;
                acc[4 * j + 1] += w * v[k][j].y;
                acc[4 * j + 2] += w * v[k][j].z;
                acc[4 * j + 3] += w * v[k][j].w;
            }
        }
    } else {
        float M = -INFINITY;
        for (int k = 0; k < np; ++k) M = fmaxf(M, __ldcg(slot_ptr(k) + 128 * kSfaHalf + row));
        for (int k = 0; k < np; ++k) {
            const float* pp = slot_ptr(k);
            const float mk = __ldcg(pp + 128 * kSfaHalf + row);
            const float w = mk == -INFINITY ? 0.f : __ldcg(pp + 128 * kSfaHalf + 128 + row) * ex2f_approx(mk - M);
            S += w;
#pragma unroll
            for (int j = 0; j < kCh / 4; ++j) {
                const float4 x = __ldcg(reinterpret_cast<const float4*>(pp) + (col0 / 4 + j) * 128 + row);
                acc[4 * j] += w * x.x;
                acc[4 * j + 1] += w * x.y;
                acc[4 * j + 2] += w * x.z;
                acc[4 * j + 3] += w * x.w;
            }
        }
    }
    const float inv = S > 0.f ? 1.f / S : 0.f;
    const bool bf = p.is_bf16 != 0;
    if (p.lse_max && h == 0 && col0 == 0) {
        float Mt = -INFINITY;
        for (int k = 0; k < np; ++k) Mt = fmaxf(Mt, __ldcg(slot_ptr(k) + 128 * kSfaHalf + 256 + row));
        float St = 0.f;
        for (int k = 0; k < np; ++k) {
            const float* pp = slot_ptr(k);
            const float mk = __ldcg(pp + 128 * kSfaHalf + row);
            if (mk != -INFINITY) St += __ldcg(pp + 128 * kSfaHalf + 128 + row) * ex2f_approx(mk - Mt);
        }
        const long long li = (long long)b * p.QN + row;
        p.lse_max[li] = Mt == -INFINITY ? -INFINITY : Mt * kLn2;
        p.lse_sum[li] = Mt == -INFINITY ? 0.f : St;
    }
    uint32_t wv[kCh / 2];
#pragma unroll
    for (int j = 0; j < kCh / 2; ++j) wv[j] = pack2(acc[2 * j] * inv, acc[2 * j + 1] * inv, bf);
    uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.out) + ((long long)b * p.QN + row) * kSfaD +
                                          h * kSfaHalf + col0);
#pragma unroll
    for (int j = 0; j < kCh / 8; ++j) dst[j] = make_uint4(wv[4 * j], wv[4 * j + 1], wv[4 * j + 2], wv[4 * j + 3]);
}

// Merges the pieces of every sequence that CTA boundaries cut, for problems with smaller shares
// (rows of many pieces): grid (2R sequences, 16 blocks of 8 head rows), 256 threads; thread =
// (head row, 8 channels).  Piece k weighs
// L_k 2^(M_k - M) / sum_j L_j 2^(M_j - M) with M the largest M_k.  One record says where the
// pieces sit; then the pieces are merged four at a time (their M, L and channels loaded
// together, one round trip per group) against the running largest M, the running sums rescaled
// when a group raises it: up to four pieces, one group with M the largest M_k.
__global__ void __launch_bounds__(kSfaCombineThreads) sfa_combine_many(const __grid_constant__ SfaParams p) {
    constexpr int kCh = 8;                                   // channels per thread
    constexpr int kRows = kSfaCombineThreads * kCh / kSfaHalf;  // head rows per block
    constexpr int kGroup = 4;                                // pieces loaded together
    const int s = blockIdx.x;
    const int b = s >> 1, h = s & 1;
    const SfaPieces pc = p.pieces[b];
    if (pc.np < 2) return;  // the count kernel or the decode kernel wrote this sequence
    // rows vary fastest across the threads: a slot holds channel quads of consecutive head rows
    const int row = blockIdx.y * kRows + (int)threadIdx.x % kRows;
    const int col0 = ((int)threadIdx.x / kRows) * kCh;
    if (row >= p.QN) return;
    const int np = pc.np;
    // pairs c_first .. c_first + np - 1 hold the row's tiles; CTA 2c + h of pair c value half h
    auto slot_ptr = [&](int k) {
        const int sl = k == 0 ? 2 * (2 * pc.c_first + h) + pc.slot0 : 2 * (2 * (pc.c_first + k) + h);
        return p.partials + (long long)sl * kSfaSlotFloats;
    };
    float acc[kCh];
#pragma unroll
    for (int j = 0; j < kCh; ++j) acc[j] = 0.f;
    float S = 0.f, M = -INFINITY;
    for (int k0 = 0; k0 < np; k0 += kGroup) {
        float m[kGroup], l[kGroup];
        float4 v[kGroup][kCh / 4];
#pragma unroll
        for (int k = 0; k < kGroup; ++k) {
            m[k] = -INFINITY;
            l[k] = 0.f;
            if (k0 + k < np) {
                const float* pp = slot_ptr(k0 + k);
                m[k] = __ldcg(pp + 128 * kSfaHalf + row);
                l[k] = __ldcg(pp + 128 * kSfaHalf + 128 + row);
#pragma unroll
                for (int j = 0; j < kCh / 4; ++j)
                    v[k][j] = __ldcg(reinterpret_cast<const float4*>(pp) + (col0 / 4 + j) * 128 + row);
            } else {
#pragma unroll
                for (int j = 0; j < kCh / 4; ++j) v[k][j] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        float Mn = M;
#pragma unroll
        for (int k = 0; k < kGroup; ++k) Mn = fmaxf(Mn, m[k]);
        if (Mn != M && M != -INFINITY) {
            const float r = ex2f_approx(M - Mn);
            S *= r;
#pragma unroll
            for (int j = 0; j < kCh; ++j) acc[j] *= r;
        }
        M = Mn;
#pragma unroll
        for (int k = 0; k < kGroup; ++k) {
            const float w = m[k] == -INFINITY ? 0.f : l[k] * ex2f_approx(m[k] - M);
            S += w;
#pragma unroll
            for (int j = 0; j < kCh / 4; ++j) {
                acc[4 * j] += w * v[k][j].x;
                acc[4 * j + 1] += w * v[k][j].y;
                acc[4 * j + 2] += w * v[k][j].z;
                acc[4 * j + 3] += w * v[k][j].w;
            }
        }
    }
    const float inv = S > 0.f ? 1.f / S : 0.f;
    const bool bf = p.is_bf16 != 0;
    if (p.lse_max && h == 0 && col0 == 0) {
        // the largest score over the pieces and the sum of exp(score - it), grouped the same way
        float Mt = -INFINITY, St = 0.f;
        for (int k0 = 0; k0 < np; k0 += kGroup) {
            float mt[kGroup], m[kGroup], l[kGroup];
#pragma unroll
            for (int k = 0; k < kGroup; ++k) {
                mt[k] = m[k] = -INFINITY;
                l[k] = 0.f;
                if (k0 + k < np) {
                    const float* pp = slot_ptr(k0 + k);
                    mt[k] = __ldcg(pp + 128 * kSfaHalf + 256 + row);
                    m[k] = __ldcg(pp + 128 * kSfaHalf + row);
                    l[k] = __ldcg(pp + 128 * kSfaHalf + 128 + row);
                }
            }
            float Mn = Mt;
#pragma unroll
            for (int k = 0; k < kGroup; ++k) Mn = fmaxf(Mn, mt[k]);
            if (Mn != Mt && Mt != -INFINITY) St *= ex2f_approx(Mt - Mn);
            Mt = Mn;
#pragma unroll
            for (int k = 0; k < kGroup; ++k)
                if (m[k] != -INFINITY) St += l[k] * ex2f_approx(m[k] - Mt);
        }
        const long long li = (long long)b * p.QN + row;
        p.lse_max[li] = Mt == -INFINITY ? -INFINITY : Mt * kLn2;
        p.lse_sum[li] = Mt == -INFINITY ? 0.f : St;
    }
    uint32_t wv[kCh / 2];
#pragma unroll
    for (int j = 0; j < kCh / 2; ++j) wv[j] = pack2(acc[2 * j] * inv, acc[2 * j + 1] * inv, bf);
    uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.out) + ((long long)b * p.QN + row) * kSfaD +
                                          h * kSfaHalf + col0);
#pragma unroll
    for (int j = 0; j < kCh / 8; ++j) dst[j] = make_uint4(wv[4 * j], wv[4 * j + 1], wv[4 * j + 2], wv[4 * j + 3]);
}

int sfa_max_pairs() {
    static std::atomic<int> pairs[kMaxDevices];  // per device; 0 until known
    const int dev = current_device_slot();
    if (dev < 0) return 0;
    int known = pairs[dev].load(std::memory_order_acquire);
    if (known == 0) {
        int n = 0, sms = 0;
        if (cudaFuncSetAttribute(sfa_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSfaSmem) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, sfa_kernel, kSfaThreads, kSfaSmem) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            n = 0;
        cudaGetLastError();
        known = n * sms / 2;
        if (known > 0) pairs[dev].store(known, std::memory_order_release);
    }
    return known;
}

static cudaError_t launch_sfa_decode_and_combine(const SfaParams& p, cudaStream_t stream) {
    // the decode kernel starts its prologue while the counts finish (it waits before reading them)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.P);
    cfg.blockDim = dim3(kSfaThreads);
    cfg.dynamicSmemBytes = kSfaSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, sfa_kernel, p);
    if (e != cudaSuccess) return e;
    // An ordinary launch: with programmatic dependent launch (resident early, waiting) the
    // combine cost the sparse MLA workload 18 us per call on this part.
    // Shares of four tiles and more (so rows of a few pieces): 16 channels a thread, every block
    // resident at once; smaller shares cut rows into many pieces, merged four at a time.
    if (p.W >= 4LL * (p.P >> 1))
        sfa_combine_few<<<dim3(2 * p.R, kSfaHalf / 16), 128, 0, stream>>>(p);
    else
        sfa_combine_many<<<dim3(2 * p.R, 128 * kSfaHalf / (8 * kSfaCombineThreads)), kSfaCombineThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_sfa(const SfaParams& p, cudaStream_t stream) {
    static std::atomic<bool> configured[kMaxDevices];  // per device: the attribute is set per device
    const int dev = current_device_slot();
    if (dev < 0) return cudaErrorInvalidDevice;
    if (!configured[dev].load(std::memory_order_acquire)) {
        const cudaError_t e = cudaFuncSetAttribute(sfa_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSfaSmem);
        if (e != cudaSuccess) return e;
        configured[dev].store(true, std::memory_order_release);
    }
    cudaError_t e;
    if (p.R <= kSfaLocalRows) {
        // live tiles per row, ordered after everything before it on the stream; the decode CTAs
        // derive the split themselves
        sfa_count_rows<<<(p.R + kSfaRowCountWarps - 1) / kSfaRowCountWarps, kSfaRowCountWarps * 32, 0, stream>>>(p);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        return launch_sfa_decode_and_combine(p, stream);
    }
    // tile counts, prefix, split and piece records: one cluster, ordered after everything
    // before it on the stream
    cudaLaunchConfig_t cc = {};
    cc.gridDim = dim3(kSfaCountCtas);
    cc.blockDim = dim3(kSfaCountThreads);
    cc.stream = stream;
    cudaLaunchAttribute ca[1];
    ca[0].id = cudaLaunchAttributeClusterDimension;
    ca[0].val.clusterDim.x = kSfaCountCtas;
    ca[0].val.clusterDim.y = 1;
    ca[0].val.clusterDim.z = 1;
    cc.attrs = ca;
    cc.numAttrs = 1;
    e = cudaLaunchKernelEx(&cc, sfa_count, p);
    if (e != cudaSuccess) return e;
    return launch_sfa_decode_and_combine(p, stream);
}

}  // namespace ifa

