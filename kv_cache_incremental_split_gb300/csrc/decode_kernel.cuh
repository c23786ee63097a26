// Split-KV decode kernel.  One persistent CTA per SM walks an equal share of
// the T-token tiles of all (batch, key/value head, query-head slice)
// sequences (stream-K style: variable lengths are balanced to +-1 tile).
//
// Warp NWC is the producer: TMA loads (128-byte swizzle, L2 evict-first) of
// the key and value tiles in 32-row sub-boxes (sub-boxes past the window end
// are not fetched), per-row bulk copies of the query rows at each sequence
// piece start, block-table prefetch for the next tiles, bounded waits.
// Warps 0..NWC-1 each own 16 tokens of every stage and run
//   S^T = K . Q^T      mma.sync m16n8k16, tokens on M, query heads on N
//   mask, online softmax in the exp2 domain (fp32), rescale skipped while the
//   running maxima do not move
//   O^T += V^T . P^T   ldmatrix.trans for V^T, movmatrix for P^T
// A sequence piece that starts and ends inside the CTA is normalised and
// written to the output.  A piece cut by a CTA boundary writes (O, m, l) to
// the CTA's partial slot and bumps the sequence's arrival counter; the CTA
// that arrives last merges all pieces in piece order (deterministic, no float
// atomics) and resets the counter, so one launch finishes the call.
//
// int8 key/value (antiquant): the per-channel key scale is folded into the
// query (q'[d] = q[d] * scale_K[d]) and the key offset is dropped, because it
// adds the same constant to every score of a row; the value scale and offset
// are applied once to the normalised output: out = scale_V * (o + offset_V).
// int8 bytes become exact fp16 values with a byte permute and one subtract.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "decode.cuh"
#include "ptx.cuh"

namespace ifa {

struct TileCursor {
    int b;      // batch
    int r;      // sequence within the batch: kv_head * NGS + slice
    int i;      // tile within the sequence
    int tiles;  // tiles of each sequence of batch b
};

template <int T>
__device__ __forceinline__ int tiles_of(int len) { return (len + T - 1) / T; }

template <int T>
__device__ __forceinline__ void cursor_init(TileCursor& c, const int* bd, int B, long long g) {
    const int* pre = bd + 2 * B;
    int lo = 0, hi = B;  // invariant: pre[lo] <= g < pre[hi] (pre[B] = W > g)
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if ((long long)pre[mid] <= g) lo = mid;
        else hi = mid;
    }
    c.b = lo;
    c.tiles = tiles_of<T>(bd[B + lo]);
    const long long off = g - pre[lo];
    c.r = (int)(off / c.tiles);
    c.i = (int)(off % c.tiles);
}

template <int T>
__device__ __forceinline__ void cursor_next(TileCursor& c, const int* bd, int B, int RS) {
    if (++c.i < c.tiles) return;
    c.i = 0;
    if (++c.r < RS) return;
    c.r = 0;
    do {
        ++c.b;
    } while (c.b < B && bd[B + c.b] == 0);
    c.tiles = c.b < B ? tiles_of<T>(bd[B + c.b]) : 1;
}

// CTA whose tile range [floor(c W / P), floor((c+1) W / P)) holds global tile t.
__device__ __forceinline__ int cta_of(long long t, long long W, int P) {
    return (int)(((t + 1) * (long long)P - 1) / W);
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float ld_half_as_float(const void* base, long long idx, int is_bf16) {
    const unsigned short u = __ldg(reinterpret_cast<const unsigned short*>(base) + idx);
    return is_bf16 ? __bfloat162float(__ushort_as_bfloat16(u)) : __half2float(__ushort_as_half(u));
}

__device__ __forceinline__ void st_out(void* out, long long idx, float v, int is_bf16) {
    if (is_bf16) reinterpret_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
    else reinterpret_cast<__half*>(out)[idx] = __float2half_rn(v);
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if constexpr (BF16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    } else {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
}

__device__ __forceinline__ void record_error(const DecodeParams& p, int bits) { atomicOr(p.err, bits); }

// Mask bits of one consumer thread for one tile: bit (4j + e) is set when the
// mask excludes score element e of n-tile j.  Only positions < valid are read.
template <int NT, int T>
__device__ __forceinline__ uint32_t load_mask_bits(const DecodeParams& p, const TileCursor& c, const int* bd,
                                                   int row0, int r, int q4) {
    const int B = p.B;
    const int len = bd[B + c.b];
    const int valid = min(T, len - c.i * T);
    const int h = c.r / p.NGS, gs = c.r % p.NGS;
    const int GTv = min(p.GT, p.G - gs * p.GT);
    const uint8_t* base = p.mask + (long long)c.b * p.mask_bstride + (long long)bd[c.b] + (long long)c.i * T;
    const int tl = row0 + r, th = row0 + r + 8;
    uint32_t bits = 0;
    if (p.mask_nstride == 0) {
        const uint32_t lo = tl < valid ? __ldg(base + tl) : 0u;
        const uint32_t hi = th < valid ? __ldg(base + th) : 0u;
        const uint32_t pat = (lo ? 0x3u : 0u) | (hi ? 0xCu : 0u);
#pragma unroll
        for (int j = 0; j < NT; ++j) bits |= pat << (4 * j);
    } else {
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int gg = 8 * j + 2 * q4 + (e & 1);
                const int t = (e >> 1) ? th : tl;
                if (t < valid && gg < GTv) {
                    const long long n = (long long)h * p.G + (long long)gs * p.GT + gg;
                    if (__ldg(base + n * p.mask_nstride + t)) bits |= 1u << (4 * j + e);
                }
            }
    }
    return bits;
}

template <int KV, int DPAD, int NT>
__global__ void __launch_bounds__(DecodeCfg<KV, DPAD, NT>::THREADS, 1)
    decode_kernel(const __grid_constant__ DecodeParams p) {
    using C = DecodeCfg<KV, DPAD, NT>;
    constexpr bool MMA_BF16 = (KV == KV_BF16);
    constexpr int T = C::T;
    constexpr int NWC = C::NWC;
    constexpr int CONSUMERS = NWC * 32;
    constexpr int KSTEPS = DPAD / 16;
    constexpr int MT = DPAD / 16;
    constexpr int MW = C::MW;
    static_assert(C::MERGE_BYTES >= (kMaxCtas + 1) * C::GT_PAD * 4, "merge buffer holds the piece factors");

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stages = smem;
    float* mrg_o = reinterpret_cast<float*>(smem + C::STAGES * C::STAGE_BYTES);
    float* mrg_m = mrg_o + MW * C::GT_PAD * DPAD;
    float* mrg_l = mrg_m + MW * C::GT_PAD;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES + C::MERGE_BYTES);
    uint64_t* empty = full + C::STAGES;
    int* info = reinterpret_cast<int*>(empty + C::STAGES);
    volatile int* abort_flag = info + C::STAGES;
    volatile int* last_flag = abort_flag + 1;
    volatile int* blkbuf = last_flag + 1;  // [8] block ids of the current tile's full boxes (producer)

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int* bd = p.ext_bdata ? p.ext_bdata : p.bdata_inline;
    const int B = p.B;
    const int RS = p.KV_N * p.NGS;
    const long long lo = (long long)blockIdx.x * p.W / p.P;
    const long long hi = (long long)(blockIdx.x + 1) * p.W / p.P;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NWC);
        }
        *abort_flag = 0;
        *last_flag = 0;
        fence_mbar_init();
    }
    // Query buffers start (and stay) zero outside the rows/columns the bulk copies fill.
    for (int idx = threadIdx.x; idx < C::STAGES * (C::Q_BYTES / 16); idx += C::THREADS) {
        const int s = idx / (C::Q_BYTES / 16), o = idx % (C::Q_BYTES / 16);
        reinterpret_cast<int4*>(stages + s * C::STAGE_BYTES + 2 * C::KT_BYTES)[o] = make_int4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
    __syncthreads();

    // Batches with no valid token produce all-zero rows; CTA c takes b = c, c+P, ...
    for (int b = blockIdx.x; b < B; b += p.P) {
        if (bd[B + b] != 0) continue;
        const long long base = (long long)b * p.N * p.D;
        for (int idx = threadIdx.x; idx < p.N * p.D; idx += C::THREADS) st_out(p.out, base + idx, 0.f, p.q_bf16);
    }
    if (lo >= hi) return;

    if (warp == NWC) {
        // ================================================================ producer warp
        if (lane == 0) {
            prefetch_tensormap(&p.tmK);
            prefetch_tensormap(&p.tmV);
            prefetch_tensormap(&p.tmKt);
            prefetch_tensormap(&p.tmVt);
            if (p.mask_tma) prefetch_tensormap(&p.tmM);
        }
        const uint64_t pol = policy_evict_first();
        const int br = p.box_rows;
        const int tr = p.tail_rows;
        const int nsub = T / br;  // full boxes per tile: 1..8
        const int batch_tiles = 32 / nsub;
        TileCursor cur;
        cursor_init<T>(cur, bd, B, lo);
        int my_blk = 0;
        long long it = 0;
        for (long long g = lo; g < hi; ++g, ++it) {
            const int kk = (int)((g - lo) % batch_tiles);
            if (p.paged && kk == 0) {
                // Block ids of the next batch_tiles tiles: lane l reads full box (l % nsub) of tile (l / nsub).
                TileCursor c2 = cur;
                const int adv = lane / nsub;
                const bool live = (g + adv) < hi;
                if (live)
                    for (int a = 0; a < adv; ++a) cursor_next<T>(c2, bd, B, RS);
                my_blk = -2;
                if (live) {
                    const int t0 = c2.i * T + (lane % nsub) * br;
                    if (t0 < bd[B + c2.b])
                        my_blk = __ldg(&p.block_table[(long long)c2.b * p.bt_cols + t0 / p.block_size]);
                }
            }
            const int stage = (int)(it % C::STAGES);
            const uint32_t round = (uint32_t)(it / C::STAGES);
            if (round > 0) {
                if (!mbar_wait_bounded(&empty[stage], (round - 1) & 1, kWaitLimitNs)) {
                    if (lane == 0) record_error(p, kErrTimeout);
                    *abort_flag = 1;
                }
            }
            __syncwarp();
            if (*abort_flag) break;
            const int b = cur.b;
            const int h = cur.r / p.NGS;
            const int gs = cur.r % p.NGS;
            const int valid = min(T, bd[B + b] - cur.i * T);
            uint8_t* sb = stages + stage * C::STAGE_BYTES;
            if (p.paged) {
                const int v = __shfl_sync(0xffffffffu, my_blk, (kk * nsub + lane) & 31);
                if (lane < nsub) blkbuf[lane] = v;
            }
            __syncwarp();
            if (lane == 0) {
                const bool first = (cur.i == 0) || (g == lo);
                // A full tile moves in nsub boxes of br rows; a window's last tile in boxes of tr rows
                // that stop at the first one past the window end.
                const bool tail = valid < T;
                const int rows_per = tail ? tr : br;
                const int nbox = tail ? (valid + tr - 1) / tr : nsub;
                const uint32_t box_bytes = 2u * C::NCG * 128u * (uint32_t)rows_per;
                uint32_t bytes = 0;
                int badmask = 0, rows = 0;
                if (first) {
                    rows = min(p.GT, p.G - gs * p.GT);
                    bytes += (uint32_t)rows * (uint32_t)p.D * 2u;
                }
                if (p.paged) {
                    for (int s = 0; s < nsub; ++s) {
                        const int blk = blkbuf[s];
                        if (s * br < valid && !(blk >= 0 && blk < p.block_num)) badmask |= 1 << s;
                    }
                }
                for (int k = 0; k < nbox; ++k)
                    if (!((badmask >> ((k * rows_per) / br)) & 1)) bytes += box_bytes;
                if (p.mask_tma) bytes += (uint32_t)(T + 16);
                if (badmask) record_error(p, kErrBadBlock);
                info[stage] = badmask;
                mbar_arrive_expect_tx(&full[stage], bytes);
                if (first) {
                    const char* qsrc = reinterpret_cast<const char*>(p.q) +
                                       ((long long)b * p.N + (long long)h * p.G + (long long)gs * p.GT) * p.D * 2;
                    uint8_t* qdst = sb + 2 * C::KT_BYTES;
                    for (int row = 0; row < rows; ++row)
                        bulk_g2s(qdst + row * C::QROW, qsrc + (long long)row * p.D * 2, (uint32_t)p.D * 2u, &full[stage]);
                }
                const int st = bd[b];
                if (p.mask_tma) {
                    // this tile's mask bytes, from the 16-byte boundary at or below its first position
                    const int x0 = st + cur.i * T;
                    tma_load_2d(sb + C::MASK_OFF, &p.tmM, &full[stage], x0 & ~15, p.mask_bstride ? b : 0);
                }
                const CUtensorMap* mk = tail ? &p.tmKt : &p.tmK;
                const CUtensorMap* mv = tail ? &p.tmVt : &p.tmV;
                for (int k = 0; k < nbox; ++k) {
                    const int r0 = k * rows_per;  // first row of the box within the tile
                    const int s = r0 / br;
                    if ((badmask >> s) & 1) continue;
                    int y, w;
                    if (p.paged) {
                        y = (cur.i * T + r0) % p.block_size;
                        w = blkbuf[s];
                    } else {
                        y = st + cur.i * T + r0;
                        w = b;
                    }
#pragma unroll
                    for (int cg = 0; cg < C::NCG; ++cg) {
                        const int off = cg * (T * 128) + r0 * 128;
                        tma_load_4d(sb + off, mk, &full[stage], cg * C::CG_ELEMS, y, h, w, pol);
                        tma_load_4d(sb + C::KT_BYTES + off, mv, &full[stage], cg * C::CG_ELEMS, y, h, w, pol);
                    }
                }
            }
            __syncwarp();
            cursor_next<T>(cur, bd, B, RS);
        }
        // On abort, let every issued copy land before the CTA's shared memory is released.
        if (*abort_flag && lane == 0) {
            for (long long k = (it > C::STAGES ? it - C::STAGES : 0); k < it; ++k)
                mbar_wait_bounded(&full[k % C::STAGES], (uint32_t)(k / C::STAGES) & 1, kWaitLimitNs);
        }
        return;
    }

    // ==================================================================== consumer warps
    const int r = lane >> 2;
    const int q4 = lane & 3;
    const int row0 = warp * kWarpTokens;
    const float sl2 = p.scale_log2;
    const int tid = threadIdx.x;  // 0 .. CONSUMERS-1

    uint32_t qf[KSTEPS][NT][2];
    float acc[MT][NT][4];
    float m_run[NT][2], l_run[NT][2];

    TileCursor cur;
    cursor_init<T>(cur, bd, B, lo);
    const bool mask_regs = p.has_mask && !p.mask_tma;  // masks without staging: loaded one tile ahead
    uint32_t mask_next = mask_regs ? load_mask_bits<NT, T>(p, cur, bd, row0, r, q4) : 0u;
    long long it = 0;
    for (long long g = lo; g < hi; ++g, ++it) {
        const TileCursor tc = cur;
        uint32_t mbits = mask_next;
        if (g + 1 < hi) {
            cursor_next<T>(cur, bd, B, RS);
            if (mask_regs) mask_next = load_mask_bits<NT, T>(p, cur, bd, row0, r, q4);  // one tile ahead
        }
        const int stage = (int)(it % C::STAGES);
        const uint32_t round = (uint32_t)(it / C::STAGES);
        if (!mbar_wait_bounded(&full[stage], round & 1, kWaitLimitNs)) {
            if (lane == 0) record_error(p, kErrTimeout);
            *abort_flag = 1;
        }
        __syncwarp();
        if (*abort_flag) break;

        const int b = tc.b;
        const int h = tc.r / p.NGS;
        const int gs = tc.r % p.NGS;
        const int i = tc.i;
        const int len = bd[B + b];
        const bool first = (i == 0) || (g == lo);
        const bool last = (i == tc.tiles - 1) || (g == hi - 1);
        const int GTv = min(p.GT, p.G - gs * p.GT);
        uint8_t* sb = stages + stage * C::STAGE_BYTES;
        const uint32_t kbase = smem_u32(sb);
        const uint32_t vbase = kbase + C::KT_BYTES;

        if (first) {
            const uint8_t* qb = sb + 2 * C::KT_BYTES;
#pragma unroll
            for (int ks = 0; ks < KSTEPS; ++ks) {
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    const int gg = 8 * j + r;
                    const uint8_t* qrow = qb + gg * C::QROW;
                    if constexpr (KV == KV_I8) {
                        // k-step ks covers channels 16ks..16ks+15 in the byte order ldmatrix hands out
                        // the key bytes: (4q4, 4q4+1) -> b0 and (4q4+2, 4q4+3) -> b1.
                        float qv[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int d = 16 * ks + 4 * q4 + e;
                            float x = 0.f;
                            if (d < p.D && gg < GTv) {
                                const unsigned short u = *reinterpret_cast<const unsigned short*>(qrow + d * 2);
                                x = p.q_bf16 ? __bfloat162float(__ushort_as_bfloat16(u))
                                             : __half2float(__ushort_as_half(u));
                                const long long si = p.aq_per_channel ? (long long)h * p.D + d : 0;
                                x *= ld_half_as_float(p.aq_scale, si, p.q_bf16);
                            }
                            qv[e] = x;
                        }
                        qf[ks][j][0] = pack2<false>(qv[0], qv[1]);
                        qf[ks][j][1] = pack2<false>(qv[2], qv[3]);
                    } else {
                        qf[ks][j][0] = *reinterpret_cast<const uint32_t*>(qrow + (16 * ks + 2 * q4) * 2);
                        qf[ks][j][1] = *reinterpret_cast<const uint32_t*>(qrow + (16 * ks + 8 + 2 * q4) * 2);
                    }
                }
            }
#pragma unroll
            for (int md = 0; md < MT; ++md)
#pragma unroll
                for (int j = 0; j < NT; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[md][j][e] = 0.f;
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                m_run[j][0] = m_run[j][1] = -INFINITY;
                l_run[j][0] = l_run[j][1] = 0.f;
            }
        }

        const int valid = min(T, len - i * T);
        const int badmask = info[stage];
        if (p.mask_tma) {
            const uint8_t* ms = sb + C::MASK_OFF + ((bd[b] + i * T) & 15);
            const int tl = row0 + r, th = row0 + r + 8;
            const uint32_t pat = ((tl < valid && ms[tl]) ? 0x3u : 0u) | ((th < valid && ms[th]) ? 0xCu : 0u);
            mbits = 0;
#pragma unroll
            for (int j = 0; j < NT; ++j) mbits |= pat << (4 * j);
        }
        // Rows past the window end (or in a skipped block) may hold anything, NaN
        // included: clear this warp's invalid value rows so 0 * garbage stays 0.
        if constexpr (KV != KV_I8) {
            if (valid < row0 + kWarpTokens || badmask) {
                for (int idx = lane; idx < kWarpTokens * C::NCG * 8; idx += 32) {
                    const int rr = idx / (C::NCG * 8);
                    const int c16 = idx % (C::NCG * 8);
                    const int row = row0 + rr;
                    if (row >= valid || ((badmask >> (row / p.box_rows)) & 1))
                        *reinterpret_cast<int4*>(sb + C::KT_BYTES + (c16 >> 3) * (T * 128) + row * 128 + (c16 & 7) * 16) =
                            make_int4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
        }

        // ---------------------------------------------------------- S^T = K . Q^T (two accumulator chains)
        float s[NT][4], s2[NT][4];
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[j][e] = s2[j][e] = 0.f;
        {
            const int lrow = row0 + (lane & 7) + ((lane >> 3) & 1) * 8;
            const uint32_t rbase = kbase + lrow * 128;
            const int sw = lrow & 7;
            if constexpr (KV == KV_I8) {
#pragma unroll
                for (int ks = 0; ks < KSTEPS; ks += 2) {
                    const int ch = ks + (lane >> 4);  // 16-byte chunk = 16 channels
                    const uint32_t addr = rbase + (ch >> 3) * (T * 128) + (((ch & 7) ^ sw) << 4);
                    uint32_t r0, r1, r2, r3;
                    ldsm_x4(addr, r0, r1, r2, r3);
                    r0 ^= 0x80808080u; r1 ^= 0x80808080u; r2 ^= 0x80808080u; r3 ^= 0x80808080u;
                    const uint32_t a0 = i8x2_to_f16x2(r0, 0x4140), a2 = i8x2_to_f16x2(r0, 0x4342);
                    const uint32_t a1 = i8x2_to_f16x2(r1, 0x4140), a3 = i8x2_to_f16x2(r1, 0x4342);
                    const uint32_t c0 = i8x2_to_f16x2(r2, 0x4140), c2 = i8x2_to_f16x2(r2, 0x4342);
                    const uint32_t c1 = i8x2_to_f16x2(r3, 0x4140), c3 = i8x2_to_f16x2(r3, 0x4342);
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        mma_16816<false>(s[j], a0, a1, a2, a3, qf[ks][j][0], qf[ks][j][1]);
                        mma_16816<false>(s2[j], c0, c1, c2, c3, qf[ks + 1][j][0], qf[ks + 1][j][1]);
                    }
                }
            } else {
#pragma unroll
                for (int ks = 0; ks < KSTEPS; ++ks) {
                    const int ch = 2 * ks + (lane >> 4);  // 16-byte chunk = 8 channels
                    const uint32_t addr = rbase + (ch >> 3) * (T * 128) + (((ch & 7) ^ sw) << 4);
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(addr, a0, a1, a2, a3);
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        // one n-tile: alternate two accumulators to halve the dependent chain
                        if (NT == 1 && (ks & 1)) mma_16816<MMA_BF16>(s2[j], a0, a1, a2, a3, qf[ks][j][0], qf[ks][j][1]);
                        else mma_16816<MMA_BF16>(s[j], a0, a1, a2, a3, qf[ks][j][0], qf[ks][j][1]);
                    }
                }
            }
        }

        // ---------------------------------------------------------- mask, online softmax
        const int t_lo = row0 + r, t_hi = row0 + r + 8;
        const bool ok_lo = t_lo < valid && !((badmask >> (t_lo / p.box_rows)) & 1);
        const bool ok_hi = t_hi < valid && !((badmask >> (t_hi / p.box_rows)) & 1);
        uint32_t pb[NT][2];
        float x[NT][4];
        bool moved = false;
        float mnew[NT][2];
#pragma unroll
        for (int j = 0; j < NT; ++j) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const bool ok = ((e >> 1) ? ok_hi : ok_lo) && !((mbits >> (4 * j + e)) & 1u);
                x[j][e] = ok ? (s[j][e] + s2[j][e]) * sl2 : -INFINITY;
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                float mx = fmaxf(x[j][u], x[j][u + 2]);
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                mnew[j][u] = fmaxf(m_run[j][u], mx);
                moved |= mnew[j][u] != m_run[j][u];
            }
        }
        if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const float alpha = mnew[j][u] == -INFINITY ? 1.f : ex2(m_run[j][u] - mnew[j][u]);
                    l_run[j][u] *= alpha;
#pragma unroll
                    for (int md = 0; md < MT; ++md) {
                        acc[md][j][u] *= alpha;
                        acc[md][j][u + 2] *= alpha;
                    }
                    m_run[j][u] = mnew[j][u];
                }
        }
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            float pr[4];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const float m_use = m_run[j][u] == -INFINITY ? 0.f : m_run[j][u];
                pr[u] = ex2(x[j][u] - m_use);
                pr[u + 2] = ex2(x[j][u + 2] - m_use);
                l_run[j][u] += pr[u] + pr[u + 2];
            }
            pb[j][0] = movmatrix_t(pack2<MMA_BF16>(pr[0], pr[1]));
            pb[j][1] = movmatrix_t(pack2<MMA_BF16>(pr[2], pr[3]));
        }

        // ---------------------------------------------------------- O^T += V^T . P^T
        {
            if constexpr (KV == KV_I8) {
                const int lrow = row0 + (lane & 7) + ((lane >> 3) & 1) * 8;
                const uint32_t rbase = vbase + lrow * 128;
                const int sw = lrow & 7;
#pragma unroll
                for (int c = 0; c < MT; c += 2) {
                    const int ch = c + (lane >> 4);
                    const uint32_t addr = rbase + (ch >> 3) * (T * 128) + (((ch & 7) ^ sw) << 4);
                    uint32_t r0, r1, r2, r3;
                    ldsm_x4_t(addr, r0, r1, r2, r3);
                    r0 ^= 0x80808080u; r1 ^= 0x80808080u; r2 ^= 0x80808080u; r3 ^= 0x80808080u;
                    const uint32_t a0 = i8x2_to_f16x2(r0, 0x4240), a1 = i8x2_to_f16x2(r0, 0x4341);
                    const uint32_t a2 = i8x2_to_f16x2(r1, 0x4240), a3 = i8x2_to_f16x2(r1, 0x4341);
                    const uint32_t e0 = i8x2_to_f16x2(r2, 0x4240), e1 = i8x2_to_f16x2(r2, 0x4341);
                    const uint32_t e2 = i8x2_to_f16x2(r3, 0x4240), e3 = i8x2_to_f16x2(r3, 0x4341);
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        mma_16816<false>(acc[c][j], a0, a1, a2, a3, pb[j][0], pb[j][1]);
                        mma_16816<false>(acc[c + 1][j], e0, e1, e2, e3, pb[j][0], pb[j][1]);
                    }
                }
            } else {
                const int mi = lane >> 3;
                const int lrow = row0 + (lane & 7) + (mi >> 1) * 8;
                const uint32_t rbase = vbase + lrow * 128;
                const int sw = lrow & 7;
#pragma unroll
                for (int md = 0; md < MT; ++md) {
                    const int ch = 2 * md + (mi & 1);
                    const uint32_t addr = rbase + (ch >> 3) * (T * 128) + (((ch & 7) ^ sw) << 4);
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4_t(addr, a0, a1, a2, a3);
#pragma unroll
                    for (int j = 0; j < NT; ++j) mma_16816<MMA_BF16>(acc[md][j], a0, a1, a2, a3, pb[j][0], pb[j][1]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);

        if (!last) continue;
        // ============================================================ piece epilogue
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                float v = l_run[j][u];
                v += __shfl_xor_sync(0xffffffffu, v, 4);
                v += __shfl_xor_sync(0xffffffffu, v, 8);
                v += __shfl_xor_sync(0xffffffffu, v, 16);
                l_run[j][u] = v;
            }
        // publish (m, l, O) of warp w into merge slot `slot`
        auto publish = [&](int slot) {
            if (r == 0) {
#pragma unroll
                for (int j = 0; j < NT; ++j)
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int gg = 8 * j + 2 * q4 + u;
                        mrg_m[slot * C::GT_PAD + gg] = m_run[j][u];
                        mrg_l[slot * C::GT_PAD + gg] = l_run[j][u];
                    }
            }
#pragma unroll
            for (int md = 0; md < MT; ++md)
#pragma unroll
                for (int j = 0; j < NT; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int gg = 8 * j + 2 * q4 + (e & 1);
                        const int d = (KV == KV_I8) ? 16 * md + 2 * r + (e >> 1) : 16 * md + r + 8 * (e >> 1);
                        mrg_o[(slot * C::GT_PAD + gg) * DPAD + d] = acc[md][j][e];
                    }
        };
        if constexpr (NWC > MW) {
            // first fold warps MW.. into warps 0..MW-1, in registers
            if (warp >= MW) publish(warp - MW);
            named_bar_sync(1, CONSUMERS);
            if (warp < MW) {
#pragma unroll
                for (int j = 0; j < NT; ++j)
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int gg = 8 * j + 2 * q4 + u;
                        const float mp = mrg_m[warp * C::GT_PAD + gg];
                        const float lp = mrg_l[warp * C::GT_PAD + gg];
                        const float M = fmaxf(m_run[j][u], mp);
                        const float f1 = m_run[j][u] == -INFINITY ? 0.f : ex2(m_run[j][u] - M);
                        const float f2 = mp == -INFINITY ? 0.f : ex2(mp - M);
                        l_run[j][u] = l_run[j][u] * f1 + lp * f2;
                        m_run[j][u] = M;
#pragma unroll
                        for (int md = 0; md < MT; ++md)
#pragma unroll
                            for (int hh = 0; hh < 2; ++hh) {
                                const int e = u + 2 * hh;
                                const int d = (KV == KV_I8) ? 16 * md + 2 * r + hh : 16 * md + r + 8 * hh;
                                acc[md][j][e] = acc[md][j][e] * f1 + mrg_o[(warp * C::GT_PAD + gg) * DPAD + d] * f2;
                            }
                    }
            }
            named_bar_sync(1, CONSUMERS);
        }
        if (warp < MW) publish(warp);
        named_bar_sync(1, CONSUMERS);

        const long long seq_first = g - i;
        const bool complete = seq_first >= lo && seq_first + tc.tiles <= hi;
        const int slot = 2 * (int)blockIdx.x + (seq_first <= lo ? 0 : 1);
        float* sp = p.partials + (long long)slot * p.slot_floats;
        const long long obase = ((long long)b * p.N + (long long)h * p.G + (long long)gs * p.GT) * p.D;
        for (int idx = tid; idx < GTv * p.D; idx += CONSUMERS) {
            const int gg = idx / p.D;
            const int d = idx - gg * p.D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < MW; ++w) M = fmaxf(M, mrg_m[w * C::GT_PAD + gg]);
            float L = 0.f, O = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (int w = 0; w < MW; ++w) {
                    const float f = ex2(mrg_m[w * C::GT_PAD + gg] - M);
                    L += mrg_l[w * C::GT_PAD + gg] * f;
                    O += mrg_o[(w * C::GT_PAD + gg) * DPAD + d] * f;
                }
            }
            if (complete) {
                float v = 0.f;
                if (L > 0.f) {
                    v = O / L;
                    if constexpr (KV == KV_I8) {
                        const long long si = p.aq_per_channel ? (long long)(p.KV_N + h) * p.D + d : 1;
                        v = (v + ld_half_as_float(p.aq_offset, si, p.q_bf16)) * ld_half_as_float(p.aq_scale, si, p.q_bf16);
                    }
                }
                st_out(p.out, obase + idx, v, p.q_bf16);
            } else {
                sp[gg * DPAD + d] = O;
                if (d == 0) {
                    sp[C::GT_PAD * DPAD + gg] = M;
                    sp[C::GT_PAD * DPAD + C::GT_PAD + gg] = L;
                }
            }
        }
        if (!complete) {
            // Arrive on the sequence's counter; the last piece to arrive merges all pieces.
            const int c_first = cta_of(seq_first, p.W, p.P);
            const int c_last = cta_of(seq_first + tc.tiles - 1, p.W, p.P);
            __threadfence();
            named_bar_sync(1, CONSUMERS);
            if (tid == 0) {
                // Counter word: (generation << 32) | arrivals.  A word carrying another call's tag
                // (left by an aborted call) counts as empty, so no call depends on a zeroed start.
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
                if (mine == 0) record_error(p, kErrTimeout);
                const int is_last = mine != 0 && (int)(mine & 0xffffffffull) == c_last - c_first + 1;
                if (is_last) *ctr = 0ull;  // every piece has arrived
                *last_flag = is_last;
            }
            named_bar_sync(1, CONSUMERS);
            if (*last_flag) {
                __threadfence();
                const int npieces = c_last - c_first + 1;
                const long long lo_first = (long long)c_first * p.W / p.P;
                const int slot0 = 2 * c_first + (seq_first <= lo_first ? 0 : 1);
                float* fac = mrg_o;                       // [npieces][GT_PAD] merge factors
                float* live = mrg_o + npieces * C::GT_PAD;  // [GT_PAD]
                for (int gg = tid; gg < GTv; gg += CONSUMERS) {
                    float M = -INFINITY;
                    for (int k = 0; k < npieces; ++k) {
                        const int sl = k == 0 ? slot0 : 2 * (c_first + k);
                        M = fmaxf(M, __ldcg(p.partials + (long long)sl * p.slot_floats + C::GT_PAD * DPAD + gg));
                    }
                    float L = 0.f;
                    for (int k = 0; k < npieces; ++k) {
                        const int sl = k == 0 ? slot0 : 2 * (c_first + k);
                        const float* pp = p.partials + (long long)sl * p.slot_floats;
                        const float f = M == -INFINITY ? 0.f : ex2(__ldcg(pp + C::GT_PAD * DPAD + gg) - M);
                        fac[k * C::GT_PAD + gg] = f;
                        L += __ldcg(pp + C::GT_PAD * DPAD + C::GT_PAD + gg) * f;
                    }
                    const float inv = L > 0.f ? 1.f / L : 0.f;
                    for (int k = 0; k < npieces; ++k) fac[k * C::GT_PAD + gg] *= inv;
                    live[gg] = L > 0.f ? 1.f : 0.f;
                }
                named_bar_sync(1, CONSUMERS);
                for (int idx = tid; idx < GTv * p.D; idx += CONSUMERS) {
                    const int gg = idx / p.D;
                    const int d = idx - gg * p.D;
                    float o = 0.f;
                    for (int k = 0; k < npieces; ++k) {
                        const int sl = k == 0 ? slot0 : 2 * (c_first + k);
                        o += fac[k * C::GT_PAD + gg] * __ldcg(p.partials + (long long)sl * p.slot_floats + gg * DPAD + d);
                    }
                    if constexpr (KV == KV_I8) {
                        if (live[gg] != 0.f) {
                            const long long si = p.aq_per_channel ? (long long)(p.KV_N + h) * p.D + d : 1;
                            o = (o + ld_half_as_float(p.aq_offset, si, p.q_bf16)) *
                                ld_half_as_float(p.aq_scale, si, p.q_bf16);
                        } else {
                            o = 0.f;
                        }
                    }
                    st_out(p.out, obase + idx, o, p.q_bf16);
                }
            }
        }
        named_bar_sync(1, CONSUMERS);
    }
}

template <int KV, int DPAD, int NT>
cudaError_t launch_decode(const DecodeParams& p, int grid, cudaStream_t stream) {
    using C = DecodeCfg<KV, DPAD, NT>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(decode_kernel<KV, DPAD, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    decode_kernel<KV, DPAD, NT><<<grid, C::THREADS, C::SMEM, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace ifa
