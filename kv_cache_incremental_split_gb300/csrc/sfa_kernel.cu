// Sparse-index MLA-absorb decode on the 5th-generation tensor cores.
//
//   out[b, n, :] = softmax_j(scale * (q[b,n] . k[i_j] + q_rope[b,n] . k_rope[i_j])) . v[i_j]
//   ("SparseFlashAttention" README, 功能说明 formula; i_j = sparse_indices[b,0,0,j]).
//
// Work: a sequence is (batch b, value half h): 128 query heads x 256 of the 512
// value channels (a full 128 x 512 fp32 accumulator would fill all of TMEM, so
// the two halves are separate sequences that share their scores' work).  A
// sequence is cut into 64-position tiles of its sparse index row; persistent
// CTAs take equal contiguous shares of all tiles, and pieces cut at CTA
// boundaries are merged by the CTA that finishes last (tagged arrival counters,
// fixed merge order).
//
// Per CTA: warp 0 gathers, warp 1 issues tcgen05.mma, warps 2-5 run the softmax.
//  * producer: Q of batch b (9 column blocks of [q | q_rope], 128 rows, 147 KB,
//    resident while b does not change) by 3-D TMA tiles; per tile, the 64 key
//    rows (9 column blocks incl. rope) and 64 value rows of half h (4 blocks) by
//    TMA tile::gather4 through block_table into a ring of 8 KB stages.  Invalid
//    positions gather an out-of-range row (zero fill, no memory traffic).
//  * MMA warp: S[128 x 64] = Q K^T (36 MMAs, M=128 N=64 K=16, both operands in
//    shared memory, S in TMEM); then O[128 x 256] += P V with P read from TMEM and
//    V (MN-major) from shared memory; tcgen05.commit releases ring stages and
//    signals S ready / O updated.
//  * softmax warps: thread = head row.  Masked scores, running max; O is rescaled
//    (tcgen05.ld/st) only when the max grows by more than 8 in log2 units, so P
//    stays below 2^8; P goes back to TMEM as 16-bit pairs.
// Every wait is bounded; on a timeout the kernel records error bit 2, drains its
// copies and MMAs, frees TMEM and returns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "decode.cuh"
#include "ptx.cuh"
#include "sfa.cuh"

namespace ifa {

namespace {

__device__ __forceinline__ float ex2f_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Cache row of sparse position `pos` of batch b, or total_rows when the position is
// past the index row, its index is outside [0, len) or its block-table entry is bad.
__device__ __forceinline__ int resolve_row(const SfaParams& p, int b, int pos, int len, bool* bad) {
    *bad = false;
    if (pos >= p.S_sp) return p.total_rows;
    const int idx = __ldg(p.indices + (long long)b * p.S_sp + pos);
    if (idx < 0 || idx >= len) return p.total_rows;
    if (idx / p.block_size >= p.bt_cols) {  // a length beyond the block table: treated as a bad entry
        *bad = true;
        return p.total_rows;
    }
    const int blk = __ldg(p.block_table + (long long)b * p.bt_cols + idx / p.block_size);
    if (blk < 0 || blk >= p.block_num) {
        *bad = true;
        return p.total_rows;
    }
    return blk * p.block_size + idx % p.block_size;
}

__device__ __forceinline__ int cta_of_tile(long long t, long long W, int P) {
    return (int)(((t + 1) * (long long)P - 1) / W);
}

}  // namespace

__global__ void __launch_bounds__(kSfaThreads, 1) sfa_kernel(const __grid_constant__ SfaParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sq = smem;                                   // [9][128 rows][128 B]
    uint8_t* ring = smem + kSfaQBytes;                    // [kSfaStages][64 rows][128 B]
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + kSfaStages * kSfaStageBytes);
    uint64_t* empty = full + kSfaStages;
    uint64_t* q_full = empty + kSfaStages;
    uint64_t* q_empty = q_full + 1;
    uint64_t* s_full = q_empty + 1;
    uint64_t* p_full = s_full + 1;
    uint64_t* o_full = p_full + 1;
    uint64_t* done_bar = o_full + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* last_flag = abort_flag + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const long long lo = (long long)blockIdx.x * p.W / p.P;
    const long long hi = (long long)(blockIdx.x + 1) * p.W / p.P;
    const int tps = p.tiles_per_seq;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kSfaStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        mbar_init(s_full, 1);
        mbar_init(p_full, 4);
        mbar_init(o_full, 1);
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        *last_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    const uint32_t S_T = tbase;          // columns [0, 64): scores
    const uint32_t P_T = tbase + 64;     // columns [64, 96): probabilities, 16-bit pairs
    const uint32_t O_T = tbase + 256;    // columns [256, 512): output accumulator

    if (warp == 0 && lo < hi) {
        // ================================================================ producer
        if (lane == 0) {
            prefetch_tensormap(&p.tmQ);
            prefetch_tensormap(&p.tmQr);
            prefetch_tensormap(&p.tmK);
            prefetch_tensormap(&p.tmKr);
            prefetch_tensormap(&p.tmV);
        }
        const uint64_t pol = policy_evict_first();
        long long it = 0;
        int epoch = 0;
        int prev_b = -1;
        for (long long g = lo; g < hi && !*abort_flag; ++g) {
            const int seq = (int)(g / tps), t = (int)(g % tps);
            const int b = seq >> 1, h = seq & 1;
            if (b != prev_b) {  // new query batch: wait until the MMAs using the old one are done
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
                prev_b = b;
            }
            const int len = __ldg(p.lens + b);
            bool bad0, bad1;
            const int row_lo = resolve_row(p, b, t * kSfaTile + lane, len, &bad0);
            const int row_hi = resolve_row(p, b, t * kSfaTile + lane + 32, len, &bad1);
            if (__any_sync(0xffffffffu, bad0 || bad1) && lane == 0) atomicOr(p.err, kErrBadBlock);
            // rows of positions 4q .. 4q+3 for the gather issued by lane q (< 16)
            int rows4[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int pos = 4 * (lane & 15) + i;
                const int a = __shfl_sync(0xffffffffu, row_lo, pos & 31);
                const int c = __shfl_sync(0xffffffffu, row_hi, pos & 31);
                rows4[i] = pos < 32 ? a : c;
            }
            for (int blk = 0; blk < kSfaQBlocks + kSfaVBlocks; ++blk, ++it) {
                const int stage = (int)(it % kSfaStages);
                const uint32_t round = (uint32_t)(it / kSfaStages);
                if (round > 0 && !mbar_wait_bounded(&empty[stage], (round - 1) & 1, kWaitLimitNs)) {
                    if (lane == 0) atomicOr(p.err, kErrTimeout);
                    *abort_flag = 1;
                    break;
                }
                if (lane == 0) mbar_arrive_expect_tx(&full[stage], kSfaStageBytes);
                __syncwarp();
                if (lane < 16) {
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
                    tma_gather4(ring + stage * kSfaStageBytes + lane * 512, map, &full[stage], x, rows4[0], rows4[1],
                                rows4[2], rows4[3], pol);
                }
                __syncwarp();
            }
        }
        // Let every issued copy land before shared memory can be released.
        if (lane == 0) {
            for (long long k = (it > kSfaStages ? it - kSfaStages : 0); k < it; ++k)
                mbar_wait_bounded(&full[k % kSfaStages], (uint32_t)(k / kSfaStages) & 1, kWaitLimitNs);
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
            int epoch = 0, prev_b = -1;
            uint32_t tile_n = 0;
            for (long long g = lo; g < hi; ++g, ++tile_n) {
                const int seq = (int)(g / tps), t = (int)(g % tps);
                const int b = seq >> 1;
                const bool first = (t == 0) || (g == lo);
                if (b != prev_b) {
                    if (!mbar_wait_bounded(q_full, epoch & 1, kWaitLimitNs)) break;
                    ++epoch;
                    prev_b = b;
                }
                tc_fence_after();
                bool ok = true;
                // ---- S = [q | q_rope] . [k | k_rope]^T
                for (int kb = 0; kb < kSfaQBlocks; ++kb, ++it) {
                    const int stage = (int)(it % kSfaStages);
                    if (!mbar_wait_bounded(&full[stage], (uint32_t)(it / kSfaStages) & 1, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint64_t ad = umma_sdesc(sq_addr + kb * 16384 + k * 32, 16, 1024);
                        const uint64_t bd = umma_sdesc(ring_addr + stage * kSfaStageBytes + k * 32, 16, 1024);
                        umma_ss(S_T, ad, bd, idesc_qk, (kb | k) != 0);
                    }
                    umma_commit(&empty[stage]);
                }
                if (!ok) break;
                umma_commit(s_full);
                // ---- O += P . V_half
                if (!mbar_wait_bounded(p_full, tile_n & 1, kWaitLimitNs)) break;
                tc_fence_after();
                for (int vb = 0; vb < kSfaVBlocks; ++vb, ++it) {
                    const int stage = (int)(it % kSfaStages);
                    if (!mbar_wait_bounded(&full[stage], (uint32_t)(it / kSfaStages) & 1, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint64_t bd = umma_sdesc(ring_addr + stage * kSfaStageBytes + k * 2048, 8192, 1024);
                        umma_ts(O_T + vb * 64, P_T + k * 8, bd, idesc_pv, !(first && k == 0));
                    }
                    umma_commit(&empty[stage]);
                }
                if (!ok) break;
                umma_commit(o_full);
                const bool last_of_b = (g + 1 == hi) || ((int)((g + 1) / tps) >> 1) != b;
                if (last_of_b) umma_commit(q_empty);
            }
            if (tile_n < (uint32_t)(hi - lo)) {
                atomicOr(p.err, kErrTimeout);
                *abort_flag = 1;
            }
            // every MMA issued so far has completed once done_bar flips
            umma_commit(done_bar);
            mbar_wait_bounded(done_bar, 0, kWaitLimitNs);
        }
        __syncwarp();
    } else if (warp >= 2 && lo < hi) {
        // ================================================================ softmax warps
        const int quad = warp & 3;                 // TMEM lane quadrant this warp may access
        const int row = quad * 32 + lane;          // query head of this thread
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const bool bf = p.is_bf16 != 0;
        const int ctid = threadIdx.x - 64;         // 0..127 over the softmax warps
        float m_used = -INFINITY, l_sum = 0.f;
        uint32_t tile_n = 0;
        for (long long g = lo; g < hi; ++g, ++tile_n) {
            const int seq = (int)(g / tps), t = (int)(g % tps);
            const int b = seq >> 1, h = seq & 1;
            const bool first = (t == 0) || (g == lo);
            const bool last = (t == tps - 1) || (g == hi - 1);
            // valid positions of this tile (the same rule the producer used)
            const int len = __ldg(p.lens + b);
            bool bad;
            const bool v_lo = resolve_row(p, b, t * kSfaTile + lane, len, &bad) != p.total_rows;
            const bool v_hi = resolve_row(p, b, t * kSfaTile + lane + 32, len, &bad) != p.total_rows;
            const uint32_t vmask_lo = __ballot_sync(0xffffffffu, v_lo);
            const uint32_t vmask_hi = __ballot_sync(0xffffffffu, v_hi);
            if (first) {
                m_used = -INFINITY;
                l_sum = 0.f;
            }
            if (!mbar_wait_bounded(s_full, tile_n & 1, kWaitLimitNs)) {
                if (lane == 0) atomicOr(p.err, kErrTimeout);
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            uint32_t sa[32], sb2[32];
            tmem_ld32(S_T + lane_off, sa);
            tmem_ld32(S_T + lane_off + 32, sb2);
            tmem_wait_ld();
            float x[64];
            float tmax = -INFINITY;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                x[j] = ((vmask_lo >> j) & 1) ? __uint_as_float(sa[j]) * p.scale_log2 : -INFINITY;
                x[j + 32] = ((vmask_hi >> j) & 1) ? __uint_as_float(sb2[j]) * p.scale_log2 : -INFINITY;
                tmax = fmaxf(tmax, fmaxf(x[j], x[j + 32]));
            }
            // P and O are free once the previous tile's P . V has completed
            if (tile_n > 0 && !mbar_wait_bounded(o_full, (tile_n - 1) & 1, kWaitLimitNs)) {
                if (lane == 0) atomicOr(p.err, kErrTimeout);
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            const float m_new = fmaxf(m_used, tmax);
            const bool need = m_new > m_used + kSfaRescaleSlack;  // also true when m_used = -inf < m_new
            if (__any_sync(0xffffffffu, need)) {
                const float alpha = need ? (m_used == -INFINITY ? 0.f : ex2f_approx(m_used - m_new)) : 1.f;
                if (!first) {
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
            const float m_use = m_used == -INFINITY ? 0.f : m_used;
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const float p0 = ex2f_approx(x[2 * c] - m_use);
                const float p1 = ex2f_approx(x[2 * c + 1] - m_use);
                l_sum += p0 + p1;
                if (bf) {
                    __nv_bfloat162 v2 = __floats2bfloat162_rn(p0, p1);
                    pk[c] = *reinterpret_cast<uint32_t*>(&v2);
                } else {
                    __half2 v2 = __floats2half2_rn(p0, p1);
                    pk[c] = *reinterpret_cast<uint32_t*>(&v2);
                }
            }
            tmem_st32(P_T + lane_off, pk);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);

            if (!last) continue;
            // ============================================================ piece epilogue
            if (!mbar_wait_bounded(o_full, tile_n & 1, kWaitLimitNs)) {
                if (lane == 0) atomicOr(p.err, kErrTimeout);
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            const long long seq_first = g - t;
            const bool complete = seq_first >= lo && seq_first + tps <= hi;
            const long long orow = ((long long)b * p.QN + row) * kSfaD + h * kSfaHalf;
            const int slot = 2 * (int)blockIdx.x + (seq_first <= lo ? 0 : 1);
            float* sp = p.partials + (long long)slot * kSfaSlotFloats;
            const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
            for (int c = 0; c < kSfaHalf / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(O_T + lane_off + c * 32, o);
                tmem_wait_ld();
                if (complete) {
                    if (row < p.QN) {
                        uint32_t w[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const float a = __uint_as_float(o[2 * j]) * inv, e = __uint_as_float(o[2 * j + 1]) * inv;
                            if (bf) {
                                __nv_bfloat162 v2 = __floats2bfloat162_rn(a, e);
                                w[j] = *reinterpret_cast<uint32_t*>(&v2);
                            } else {
                                __half2 v2 = __floats2half2_rn(a, e);
                                w[j] = *reinterpret_cast<uint32_t*>(&v2);
                            }
                        }
                        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.out) + orow + c * 32);
#pragma unroll
                        for (int j = 0; j < 4; ++j) dst[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
                    }
                } else {
                    float4* dst = reinterpret_cast<float4*>(sp + (long long)row * kSfaHalf + c * 32);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        dst[j] = make_float4(__uint_as_float(o[4 * j]), __uint_as_float(o[4 * j + 1]),
                                             __uint_as_float(o[4 * j + 2]), __uint_as_float(o[4 * j + 3]));
                }
            }
            tc_fence_before();
            if (complete) continue;
            sp[128 * kSfaHalf + row] = m_used;
            sp[128 * kSfaHalf + 128 + row] = l_sum;
            // arrive; the piece that arrives last merges all pieces of the sequence
            const int c_first = cta_of_tile(seq_first, p.W, p.P);
            const int c_last = cta_of_tile(seq_first + tps - 1, p.W, p.P);
            __threadfence();
            named_bar_sync(1, 128);
            if (ctid == 0) {
                unsigned long long* ctr = p.counters + c_first;
                const unsigned long long tag = (unsigned long long)p.gen << 32;
                unsigned long long cur = atomicAdd(ctr, 0ull);
                unsigned long long mine = 0;
                for (int tries = 0; tries < (1 << 16); ++tries) {
                    const unsigned long long want = ((cur & 0xffffffff00000000ull) == tag) ? cur + 1 : tag + 1;
                    const unsigned long long prev = atomicCAS(ctr, cur, want);
                    if (prev == cur) {
                        mine = want;
                        break;
                    }
                    cur = prev;
                }
                if (mine == 0) atomicOr(p.err, kErrTimeout);
                const int is_last = mine != 0 && (int)(mine & 0xffffffffull) == c_last - c_first + 1;
                if (is_last) *ctr = 0ull;
                *last_flag = is_last;
            }
            named_bar_sync(1, 128);
            if (*last_flag) {
                __threadfence();
                const int npieces = c_last - c_first + 1;
                const long long lo_first = (long long)c_first * p.W / p.P;
                const int slot0 = 2 * c_first + (seq_first <= lo_first ? 0 : 1);
                float M = -INFINITY;
                for (int k = 0; k < npieces; ++k) {
                    const int sl = k == 0 ? slot0 : 2 * (c_first + k);
                    M = fmaxf(M, __ldcg(p.partials + (long long)sl * kSfaSlotFloats + 128 * kSfaHalf + row));
                }
                float L = 0.f;
                for (int k = 0; k < npieces; ++k) {
                    const int sl = k == 0 ? slot0 : 2 * (c_first + k);
                    const float* pp = p.partials + (long long)sl * kSfaSlotFloats;
                    const float mk = __ldcg(pp + 128 * kSfaHalf + row);
                    if (M != -INFINITY) L += __ldcg(pp + 128 * kSfaHalf + 128 + row) * ex2f_approx(mk - M);
                }
                const float invL = L > 0.f ? 1.f / L : 0.f;
                if (row < p.QN) {
                    for (int c = 0; c < kSfaHalf; c += 8) {
                        float acc8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                        for (int k = 0; k < npieces; ++k) {
                            const int sl = k == 0 ? slot0 : 2 * (c_first + k);
                            const float* pp = p.partials + (long long)sl * kSfaSlotFloats;
                            const float mk = __ldcg(pp + 128 * kSfaHalf + row);
                            const float f = M == -INFINITY ? 0.f : ex2f_approx(mk - M) * invL;
                            const float4 a = __ldcg(reinterpret_cast<const float4*>(pp + (long long)row * kSfaHalf + c));
                            const float4 e = __ldcg(reinterpret_cast<const float4*>(pp + (long long)row * kSfaHalf + c + 4));
                            acc8[0] += f * a.x; acc8[1] += f * a.y; acc8[2] += f * a.z; acc8[3] += f * a.w;
                            acc8[4] += f * e.x; acc8[5] += f * e.y; acc8[6] += f * e.z; acc8[7] += f * e.w;
                        }
                        uint32_t w[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            if (bf) {
                                __nv_bfloat162 v2 = __floats2bfloat162_rn(acc8[2 * j], acc8[2 * j + 1]);
                                w[j] = *reinterpret_cast<uint32_t*>(&v2);
                            } else {
                                __half2 v2 = __floats2half2_rn(acc8[2 * j], acc8[2 * j + 1]);
                                w[j] = *reinterpret_cast<uint32_t*>(&v2);
                            }
                        }
                        *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.out) + orow + c) =
                            make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
            named_bar_sync(1, 128);
        }
    }
    // ==================================================================== teardown
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tbase, 512);
}

cudaError_t launch_sfa(const SfaParams& p, cudaStream_t stream) {
    static bool configured = false;
    if (!configured) {
        const cudaError_t e = cudaFuncSetAttribute(sfa_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSfaSmem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    sfa_kernel<<<p.P, kSfaThreads, kSfaSmem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace ifa
