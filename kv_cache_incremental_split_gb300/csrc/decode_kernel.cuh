// Split-KV decode kernel: one persistent CTA per SM walks an equal share of
// the 64-token tiles of all (batch, key/value head, query-head slice)
// sequences.  A producer warp streams key/value tiles into a ring of shared
// memory stages with TMA (128-byte swizzle) and the query rows with bulk
// copies; four consumer warps each own 16 tokens of every stage and run
//   S^T = K . Q^T     (mma.sync m16n8k16, tokens on M, query heads on N)
//   online softmax in the exp2 domain (fp32)
//   O^T += V^T . P^T  (ldmatrix.trans for V^T, movmatrix for P^T)
// A sequence piece that starts and ends inside one CTA is normalised and
// written straight to the output; pieces cut by a CTA boundary write
// (O, m, l) partials that the combine kernel merges in a fixed order.
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

__device__ __forceinline__ int tiles_of(int len) { return (len + kTileTokens - 1) / kTileTokens; }

__device__ __forceinline__ void cursor_init(TileCursor& c, const int* bd, int B, int RS, long long g) {
    const int* pre = bd + 2 * B;
    int lo = 0, hi = B;  // invariant: pre[lo] <= g < pre[hi] (pre[B] = W > g)
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if ((long long)pre[mid] <= g) lo = mid;
        else hi = mid;
    }
    c.b = lo;
    c.tiles = tiles_of(bd[B + lo]);
    long long off = g - pre[lo];
    c.r = (int)(off / c.tiles);
    c.i = (int)(off % c.tiles);
    (void)RS;
}

__device__ __forceinline__ void cursor_next(TileCursor& c, const int* bd, int B, int RS) {
    if (++c.i < c.tiles) return;
    c.i = 0;
    if (++c.r < RS) return;
    c.r = 0;
    do {
        ++c.b;
    } while (c.b < B && bd[B + c.b] == 0);
    c.tiles = c.b < B ? tiles_of(bd[B + c.b]) : 1;
}

__device__ __forceinline__ float ld_half_as_float(const void* base, long long idx, int is_bf16) {
    const unsigned short* p = reinterpret_cast<const unsigned short*>(base) + idx;
    unsigned short u = __ldg(p);
    if (is_bf16) return __bfloat162float(__ushort_as_bfloat16(u));
    return __half2float(__ushort_as_half(u));
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

template <int KV, int DPAD, int NT>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const __grid_constant__ DecodeParams p) {
    using C = DecodeCfg<KV, DPAD, NT>;
    constexpr bool MMA_BF16 = (KV == KV_BF16);
    constexpr int T = kTileTokens;
    constexpr int KSTEPS = DPAD / 16;
    constexpr int MT = DPAD / 16;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stages = smem;
    float* mrg_o = reinterpret_cast<float*>(smem + C::STAGES * C::STAGE_BYTES);
    float* mrg_m = mrg_o + kConsumerWarps * C::GT_PAD * DPAD;
    float* mrg_l = mrg_m + kConsumerWarps * C::GT_PAD;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES + C::MERGE_BYTES);
    uint64_t* empty = full + C::STAGES;
    int* info = reinterpret_cast<int*>(empty + C::STAGES);
    volatile int* abort_flag = info + C::STAGES;

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
            mbar_init(&empty[s], kConsumerWarps);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    // Query buffers start (and stay) zero outside the rows/columns the bulk copies fill.
    for (int idx = threadIdx.x; idx < C::STAGES * (C::Q_BYTES / 16); idx += kThreads) {
        const int s = idx / (C::Q_BYTES / 16), o = idx % (C::Q_BYTES / 16);
        reinterpret_cast<int4*>(stages + s * C::STAGE_BYTES + 2 * C::KT_BYTES)[o] = make_int4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
    __syncthreads();
    pdl_launch_dependents();

    // Batches with no valid token produce all-zero rows; CTA c takes b = c, c+P, ...
    for (int b = blockIdx.x; b < B; b += p.P) {
        if (bd[B + b] != 0) continue;
        const long long base = (long long)b * p.N * p.D;
        for (int idx = threadIdx.x; idx < p.N * p.D; idx += kThreads) st_out(p.out, base + idx, 0.f, p.q_bf16);
    }
    if (lo >= hi) return;

    if (warp == kConsumerWarps) {
        // ================================================================ producer warp
        if (lane == 0) {
            prefetch_tensormap(&p.tmK);
            prefetch_tensormap(&p.tmV);
        }
        const uint64_t pol = policy_evict_first();
        const int nsub = T / p.box_rows;
        const int batch_tiles = 32 / nsub;
        const uint32_t sub_bytes = 2u * C::NCG * 128u * (uint32_t)p.box_rows;
        TileCursor cur;
        cursor_init(cur, bd, B, RS, lo);
        int my_blk = 0;
        long long it = 0;
        for (long long g = lo; g < hi; ++g, ++it) {
            const int kk = (int)((g - lo) % batch_tiles);
            if (p.paged && kk == 0) {
                // Prefetch the block ids of the next batch_tiles tiles: lane l reads
                // sub-box (l % nsub) of tile (l / nsub).
                TileCursor c2 = cur;
                const int adv = lane / nsub;
                const bool live = (g + adv) < hi;
                if (live)
                    for (int a = 0; a < adv; ++a) cursor_next(c2, bd, B, RS);
                my_blk = -2;
                if (live) {
                    const int t0 = c2.i * T + (lane % nsub) * p.box_rows;
                    if (t0 < bd[B + c2.b])
                        my_blk = __ldg(&p.block_table[(long long)c2.b * p.bt_cols + t0 / p.block_size]);
                }
            }
            const int stage = (int)(it % C::STAGES);
            const uint32_t round = (uint32_t)(it / C::STAGES);
            if (round > 0) {
                bool ok = mbar_wait_bounded(&empty[stage], (round - 1) & 1, kWaitLimitNs);
                if (!ok) {
                    if (lane == 0) record_error(p, kErrTimeout);
                    *abort_flag = 1;
                }
            }
            __syncwarp();
            if (*abort_flag) break;
            const int b = cur.b;
            const int h = cur.r / p.NGS;
            const int gs = cur.r % p.NGS;
            uint8_t* sb = stages + stage * C::STAGE_BYTES;
            int blks[4] = {0, 0, 0, 0};
            if (p.paged) {
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    if (s < nsub) blks[s] = __shfl_sync(0xffffffffu, my_blk, kk * nsub + s);
            }
            if (lane == 0) {
                const bool first = (cur.i == 0) || (g == lo);
                uint32_t bytes = 0;
                int badmask = 0;
                int loadmask = 0;
                int rows = 0;
                if (first) {
                    rows = min(p.GT, p.G - gs * p.GT);
                    bytes += (uint32_t)rows * (uint32_t)p.D * 2u;
                }
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    if (s >= nsub) break;
                    if (!p.paged || (blks[s] >= 0 && blks[s] < p.block_num)) {
                        loadmask |= 1 << s;
                        bytes += sub_bytes;
                    } else if (blks[s] != -2) {
                        badmask |= 1 << s;
                    }
                }
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
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    if (!((loadmask >> s) & 1)) continue;
                    int y, w;
                    if (p.paged) {
                        const int t0 = cur.i * T + s * p.box_rows;
                        y = t0 % p.block_size;
                        w = blks[s];
                    } else {
                        y = st + cur.i * T + s * p.box_rows;
                        w = b;
                    }
#pragma unroll
                    for (int cg = 0; cg < C::NCG; ++cg) {
                        const int off = cg * (T * 128) + s * p.box_rows * 128;
                        tma_load_4d(sb + off, &p.tmK, &full[stage], cg * C::CG_ELEMS, y, h, w, pol);
                        tma_load_4d(sb + C::KT_BYTES + off, &p.tmV, &full[stage], cg * C::CG_ELEMS, y, h, w, pol);
                    }
                }
            }
            __syncwarp();
            cursor_next(cur, bd, B, RS);
        }
        // On abort, let every issued copy land before the CTA's shared memory is released.
        if (*abort_flag && lane == 0) {
            const long long issued = it;
            for (long long k = (issued > C::STAGES ? issued - C::STAGES : 0); k < issued; ++k)
                mbar_wait_bounded(&full[k % C::STAGES], (uint32_t)(k / C::STAGES) & 1, kWaitLimitNs);
        }
        return;
    }

    // ==================================================================== consumer warps
    const int r = lane >> 2;
    const int q4 = lane & 3;
    const int row0 = warp * kWarpTokens;
    const float sl2 = p.scale_log2;

    uint32_t qf[KSTEPS][NT][2];
    float acc[MT][NT][4];
    float m_run[NT][2], l_run[NT][2];

    TileCursor cur;
    cursor_init(cur, bd, B, RS, lo);
    long long it = 0;
    for (long long g = lo; g < hi; ++g, ++it) {
        const int stage = (int)(it % C::STAGES);
        const uint32_t round = (uint32_t)(it / C::STAGES);
        if (!mbar_wait_bounded(&full[stage], round & 1, kWaitLimitNs)) {
            if (lane == 0) record_error(p, kErrTimeout);
            *abort_flag = 1;
        }
        __syncwarp();
        if (*abort_flag) break;

        const int b = cur.b;
        const int h = cur.r / p.NGS;
        const int gs = cur.r % p.NGS;
        const int i = cur.i;
        const int st = bd[b];
        const int len = bd[B + b];
        const bool first = (i == 0) || (g == lo);
        const bool last = (i == cur.tiles - 1) || (g == hi - 1);
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
                        // k-step covers physical channels 16ks..16ks+15; lane pair (4q4, 4q4+1) -> b0,
                        // (4q4+2, 4q4+3) -> b1, matching the byte order ldmatrix gives the key bytes.
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
        // Rows past the window end (or in a skipped block) may hold anything, NaN
        // included: clear this warp's invalid value rows so 0 * garbage stays 0.
        if constexpr (KV != KV_I8) {
            if (valid < row0 + kWarpTokens || badmask) {
                for (int idx = lane; idx < kWarpTokens * C::NCG * 8; idx += 32) {
                    const int rr = idx / (C::NCG * 8);
                    const int c16 = idx % (C::NCG * 8);
                    const int row = row0 + rr;
                    const bool bad = row >= valid || ((badmask >> (row / p.box_rows)) & 1);
                    if (bad)
                        *reinterpret_cast<int4*>(sb + C::KT_BYTES + (c16 >> 3) * (T * 128) + row * 128 + (c16 & 7) * 16) =
                            make_int4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
        }

        // ---------------------------------------------------------- S^T = K . Q^T
        float s[NT][4];
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[j][e] = 0.f;
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
                        mma_16816<false>(s[j], c0, c1, c2, c3, qf[ks + 1][j][0], qf[ks + 1][j][1]);
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
                    for (int j = 0; j < NT; ++j) mma_16816<MMA_BF16>(s[j], a0, a1, a2, a3, qf[ks][j][0], qf[ks][j][1]);
                }
            }
        }

        // ---------------------------------------------------------- mask, online softmax
        const int t_lo = row0 + r, t_hi = row0 + r + 8;
        bool ok_lo = t_lo < valid && !((badmask >> (t_lo / p.box_rows)) & 1);
        bool ok_hi = t_hi < valid && !((badmask >> (t_hi / p.box_rows)) & 1);
        bool okg[NT][4];
        if (p.has_mask) {
            const long long sbase = (long long)st + (long long)i * T;
            const long long mb = (long long)b * p.mask_bstride;
            if (p.mask_nstride == 0) {
                if (ok_lo) ok_lo = __ldg(p.mask + mb + sbase + t_lo) == 0;
                if (ok_hi) ok_hi = __ldg(p.mask + mb + sbase + t_hi) == 0;
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    okg[j][0] = okg[j][1] = ok_lo;
                    okg[j][2] = okg[j][3] = ok_hi;
                }
            } else {
#pragma unroll
                for (int j = 0; j < NT; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int gg = 8 * j + 2 * q4 + (e & 1);
                        const bool okt = (e >> 1) ? ok_hi : ok_lo;
                        bool ok = okt;
                        if (okt && gg < GTv) {
                            const long long n = (long long)h * p.G + (long long)gs * p.GT + gg;
                            ok = __ldg(p.mask + mb + n * p.mask_nstride + sbase + ((e >> 1) ? t_hi : t_lo)) == 0;
                        }
                        okg[j][e] = ok;
                    }
            }
        } else {
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                okg[j][0] = okg[j][1] = ok_lo;
                okg[j][2] = okg[j][3] = ok_hi;
            }
        }

        uint32_t pb[NT][2];
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            float x[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) x[e] = okg[j][e] ? s[j][e] * sl2 : -INFINITY;
            float pr[4];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                float mx = fmaxf(x[u], x[u + 2]);
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                const float m_new = fmaxf(m_run[j][u], mx);
                const float m_use = m_new == -INFINITY ? 0.f : m_new;
                const float alpha = exp2f(m_run[j][u] - m_use);
                pr[u] = exp2f(x[u] - m_use);
                pr[u + 2] = exp2f(x[u + 2] - m_use);
                l_run[j][u] = l_run[j][u] * alpha + pr[u] + pr[u + 2];
                m_run[j][u] = m_new;
#pragma unroll
                for (int md = 0; md < MT; ++md) {
                    acc[md][j][u] *= alpha;
                    acc[md][j][u + 2] *= alpha;
                }
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

        // ---------------------------------------------------------- piece epilogue
        if (last) {
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
            if (r == 0) {
#pragma unroll
                for (int j = 0; j < NT; ++j)
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int gg = 8 * j + 2 * q4 + u;
                        mrg_m[warp * C::GT_PAD + gg] = m_run[j][u];
                        mrg_l[warp * C::GT_PAD + gg] = l_run[j][u];
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
                        mrg_o[(warp * C::GT_PAD + gg) * DPAD + d] = acc[md][j][e];
                    }
            named_bar_sync(1, kConsumerWarps * 32);

            const long long seq_first = g - i;
            const bool complete = seq_first >= lo && seq_first + cur.tiles <= hi;
            const int slot = 2 * (int)blockIdx.x + (seq_first <= lo ? 0 : 1);
            float* sp = p.partials + (long long)slot * p.slot_floats;
            const long long obase = ((long long)b * p.N + (long long)h * p.G + (long long)gs * p.GT) * p.D;
            for (int idx = threadIdx.x; idx < GTv * p.D; idx += kConsumerWarps * 32) {
                const int gg = idx / p.D;
                const int d = idx - gg * p.D;
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, mrg_m[w * C::GT_PAD + gg]);
                float L = 0.f, O = 0.f;
                if (M != -INFINITY) {
#pragma unroll
                    for (int w = 0; w < kConsumerWarps; ++w) {
                        const float f = exp2f(mrg_m[w * C::GT_PAD + gg] - M);
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
            named_bar_sync(1, kConsumerWarps * 32);
        }
        cursor_next(cur, bd, B, RS);
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
    decode_kernel<KV, DPAD, NT><<<grid, kThreads, C::SMEM, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace ifa
