// Split-KV decode kernel.  One persistent CTA per SM walks an equal share of
// the T-token tiles of all (batch, key/value head, query-head slice)
// sequences (stream-K style: variable lengths are balanced to +-1 tile).
//
// Warp NWC is the producer: TMA loads (128-byte swizzle, L2 evict-first) of
// the key and value tiles (whole-tile boxes, or one box per cache block when
// paged; a window's last tile in 32-row boxes that stop past the window end),
// per-row bulk copies of the query rows at each sequence piece start, the
// tile's mask bytes when the mask is per batch, block-table prefetch for the
// next tiles, and a TileInfo record per stage that tells the consumers which
// tile they hold.  Every wait is bounded.
// Warps 0..NWC-1 each own 16 tokens of every stage and run
//   S^T = K . Q^T      mma.sync m16n8k16, tokens on M, query heads on N
//   mask, online softmax in the exp2 domain (fp32), rescale skipped while the
//   running maxima do not move
//   O^T += V^T . P^T   ldmatrix.trans for V^T, movmatrix for P^T
// At the end of a sequence piece the warps exchange (m, l) and their
// accumulator fragments through shared memory as lane-contiguous float4
// (no bank conflicts) and sum the fragments normalised by the piece's L.  A
// piece that starts and ends inside the CTA is written to the output.  A
// piece cut by a CTA boundary writes its normalised O with (M, L) per head to
// the CTA's partial slot and adds one to the sequence's arrival counter (a
// release add, nothing to wait for); the CTA that holds the sequence's first
// piece, which ends that CTA's range, waits for the others' arrivals and merges
// all pieces in piece order (deterministic, no float atomics), so one launch
// finishes the call.  The merging CTA also resets the counter, so every call
// that runs to the end leaves all counters at zero for the next one, whatever
// order calls are launched or replayed in.
//
// int8 key/value (antiquant): the per-channel key scale is folded into the
// query (q'[d] = q[d] * scale_K[d]) and the key offset is dropped, because it
// adds the same constant to every score of a row; the value scale and offset
// are applied once to the normalised output: out = scale_V * (o + offset_V).
// int8 bytes become the exact fp16 values x + 1152 with one byte permute, and
// the bias is never subtracted per element: on the key side it adds
// 1152 * sum_d q'[d] to every score of a head, which the softmax ignores; on
// the value side the normalised output comes out as o + 1152 exactly, because
// the row sums l add up the same fp16-rounded probabilities the P.V MMAs use,
// so -1152 joins offset_V.
#pragma once
#include <atomic>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "decode.cuh"
#include "ptx.cuh"

namespace ifa {

struct TileCursor {
    int b;      // batch
    int r;      // sequence within the batch: kv_head * NGS + slice
    int h, gs;  // kv head and query-head slice of r
    int i;      // tile within the sequence
    int tiles;  // tiles of each sequence of batch b
};

// What the producer tells the consumer warps about the tile in a stage.
struct TileInfo {
    int b, h, gs, i;  // batch, kv head, query-head slice, tile within the sequence
    int tiles;        // tiles of the sequence
    int valid;        // rows of the tile inside the window
    int badmask;      // full-tile boxes skipped for an out-of-range block id
    int mask_shift;   // first mask byte of the tile within the staged mask bytes
};
static_assert(sizeof(TileInfo) == 32, "two int4 per stage");

template <int T>
__device__ __forceinline__ int tiles_of(int len) { return (len + T - 1) / T; }

template <int T>
__device__ __forceinline__ void cursor_init(TileCursor& c, const int* bd, int B, int NGS, long long g) {
    const int* pre = bd + 2 * B;
    int lo = 0, hi = B;  // invariant: pre[lo] <= g < pre[hi] (pre[B] = W > g)
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if ((long long)pre[mid] <= g) lo = mid;
        else hi = mid;
    }
    c.b = lo;
    c.tiles = tiles_of<T>(bd[B + lo]);
    const int off = (int)(g - pre[lo]);  // W < 2^31
    c.r = off / c.tiles;
    c.i = off - c.r * c.tiles;
    c.h = c.r / NGS;
    c.gs = c.r - c.h * NGS;
}

template <int T>
__device__ __forceinline__ void cursor_next(TileCursor& c, const int* bd, int B, int RS, int NGS) {
    if (++c.i < c.tiles) return;
    c.i = 0;
    if (++c.gs == NGS) {
        c.gs = 0;
        ++c.h;
    }
    if (++c.r < RS) return;
    c.r = c.h = c.gs = 0;
    do {
        ++c.b;
    } while (c.b < B && bd[B + c.b] == 0);
    c.tiles = c.b < B ? tiles_of<T>(bd[B + c.b]) : 1;
}

// CTA whose tile range [bounds[c], bounds[c+1]) holds global tile t (bounds strictly increasing).
__device__ __forceinline__ int cta_of(long long t, const int* bounds, int P) {
    int lo = 0, hi = P;  // invariant: bounds[lo] <= t < bounds[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if ((long long)bounds[mid] <= t) lo = mid;
        else hi = mid;
    }
    return lo;
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

// int8 output code saturate(rint(v * scale2 + offset2)) of element idx (product and sum rounded
// apart, ties to even, NaN -> 0).
__device__ __forceinline__ void st_i8(const DecodeParams& p, long long idx, float v) {
    // idx = (b * N + n) * D + d, so the per-channel entry n * D + d is idx mod N * D
    const long long pi = p.q2_per_channel ? idx % ((long long)p.N * p.D) : 0;
    float s, o = 0.f;
    if (p.q2_bf16) {
        s = __bfloat162float(__ushort_as_bfloat16(__ldg(reinterpret_cast<const unsigned short*>(p.q2_scale) + pi)));
        if (p.q2_offset)
            o = __bfloat162float(__ushort_as_bfloat16(__ldg(reinterpret_cast<const unsigned short*>(p.q2_offset) + pi)));
    } else {
        s = __ldg(reinterpret_cast<const float*>(p.q2_scale) + pi);
        if (p.q2_offset) o = __ldg(reinterpret_cast<const float*>(p.q2_offset) + pi);
    }
    const float u = __fadd_rn(__fmul_rn(v, s), o);
    int code = 0;
    if (u == u) code = (int)fminf(fmaxf(rintf(u), -128.f), 127.f);
    reinterpret_cast<int8_t*>(p.out)[idx] = (int8_t)code;
}

// Output element idx = (b * N + n) * D + d in the output dtype, or its int8 code.
__device__ __forceinline__ void st_final(const DecodeParams& p, long long idx, float v) {
    if (p.out_i8) st_i8(p, idx, v);
    else st_out(p.out, idx, v, p.q_bf16);
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
    const int h = c.h, gs = c.gs;
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

// TL: key/value given as one tensor per batch; the producer takes each batch's descriptors from
// p.kv_maps (a separate instantiation, so the other layouts' producer keeps its parameter maps).
template <int KV, int DPAD, int NT, bool TL>
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
    constexpr int FRAG4 = C::FRAG4;
    constexpr int GT_PAD = C::GT_PAD;
    constexpr int NPOS = (FRAG4 * 32 + CONSUMERS - 1) / CONSUMERS;  // fragment positions a thread combines
    constexpr int DSTEP = (KV == KV_I8) ? 1 : 8;  // channel distance between the two halves of a fragment
    static_assert(C::BAR_BYTES >= 16 * C::STAGES + 48, "barrier area");
    static_assert(C::STAGES * 32 <= C::INFO_BYTES, "tile info area");

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stages = smem;
    uint8_t* aux = smem + C::STAGES * C::STAGE_BYTES;
    float4* mrg = reinterpret_cast<float4*>(aux);  // [MW][FRAG4][32 lanes] accumulator fragments
    float* mlm = reinterpret_cast<float*>(aux + C::MERGE_BYTES);  // [NWC][GT_PAD] running max of each warp
    float* mll = mlm + NWC * GT_PAD;                               // [NWC][GT_PAD] row sums of each warp
    int* sbd = reinterpret_cast<int*>(aux + C::MERGE_BYTES + C::ML_BYTES);  // window table copy
    int4* tinfo = reinterpret_cast<int4*>(aux + C::MERGE_BYTES + C::ML_BYTES + C::BD_BYTES);  // TileInfo per stage
    uint64_t* full = reinterpret_cast<uint64_t*>(aux + C::MERGE_BYTES + C::ML_BYTES + C::BD_BYTES + C::INFO_BYTES);
    uint64_t* empty = full + C::STAGES;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + C::STAGES);
    volatile int* blkbuf = abort_flag + 2;  // [8] block ids of the current tile's full boxes (producer)

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == NWC * 32) {  // the descriptor fetches overlap the rest of the prologue
        if constexpr (!TL) {
            prefetch_tensormap(&p.tmK);
            prefetch_tensormap(&p.tmV);
            prefetch_tensormap(&p.tmKt);
            prefetch_tensormap(&p.tmVt);
        }
        if (p.mask_tma) prefetch_tensormap(&p.tmM);
    }
    // Programmatic dependent launch: the next kernel on the stream may start its own prologue on
    // SMs this grid leaves; everything before pdl_wait_primary() below touches only launch
    // parameters and shared memory.
    pdl_launch_dependents();
    const int B = p.B;
    const int RS = p.KV_N * p.NGS;
    const long long lo = p.bounds[blockIdx.x];
    const long long hi = p.bounds[blockIdx.x + 1];
    // The window table is read every tile: keep it in shared memory when it came inline.
    // Both launch-parameter arrays are copied by one loop, so their reads overlap.
    const int* bd = p.ext_bdata ? p.ext_bdata : sbd;
    int* sbounds = sbd + 3 * kInlineB + 1;
    {
        const int nbd = p.ext_bdata ? 0 : 3 * B + 1;
        for (int x = threadIdx.x; x < nbd + p.P + 1; x += C::THREADS) {
            if (x < nbd) sbd[x] = p.bdata_inline[x];
            else sbounds[x - nbd] = p.bounds[x - nbd];
        }
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NWC);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    // Query buffers start (and stay) zero outside the rows/columns the bulk copies fill.
    for (int idx = threadIdx.x; idx < C::STAGES * (C::Q_BYTES / 16); idx += C::THREADS) {
        const int s = idx / (C::Q_BYTES / 16), o = idx % (C::Q_BYTES / 16);
        reinterpret_cast<int4*>(stages + s * C::STAGE_BYTES + 2 * C::KT_BYTES)[o] = make_int4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (threadIdx.x == NWC * 32 && !p.paged && !p.ext_bdata && lo < hi) {
        // While the previous kernel on the stream finishes, pull this CTA's first tiles of a
        // contiguous cache into L2 (a paged cache would need the block table, which may still
        // be written).  The loads after the wait below then start from L2.
        TileCursor pc;
        cursor_init<T>(pc, bd, B, p.NGS, lo);
        [[maybe_unused]] int fenced = -1;  // batch whose per-tensor maps are fenced for the TMA unit
        for (long long g = lo; g < hi && g < lo + C::PREFETCH_TILES; ++g) {
            if constexpr (TL) {
                if (pc.b != fenced) {
                    for (int m = 0; m < 4; ++m) fence_tensormap_acquire(p.kv_maps + 4 * pc.b + m);
                    fenced = pc.b;
                }
            }
            const int valid = min(T, bd[B + pc.b] - pc.i * T);
            const bool tail = valid < T;
            const int rows_per = tail ? p.tail_rows : p.box_rows;
            const int nbox = tail ? (valid + rows_per - 1) / rows_per : T / p.box_rows;
            // one tensor per batch: its own maps, batch coordinate 0
            const CUtensorMap* mk = TL ? p.kv_maps + 4 * pc.b + (tail ? 1 : 0) : (tail ? &p.tmKt : &p.tmK);
            const CUtensorMap* mv = TL ? p.kv_maps + 4 * pc.b + (tail ? 3 : 2) : (tail ? &p.tmVt : &p.tmV);
            const int wb = TL ? 0 : pc.b;
            for (int k = 0; k < nbox; ++k) {
                const int y = bd[pc.b] + pc.i * T + k * rows_per;
#pragma unroll
                for (int cg = 0; cg < C::NCG; ++cg) {
                    tma_prefetch_4d(mk, cg * C::CG_ELEMS, y, pc.h, wb);
                    tma_prefetch_4d(mv, cg * C::CG_ELEMS, y, pc.h, wb);
                }
            }
            cursor_next<T>(pc, bd, B, RS, p.NGS);
        }
    }
    // Inputs, outputs and the workspace may belong to the previous kernel on the stream until it
    // has completed.
    pdl_wait_primary();

    // Batches with no valid token produce all-zero rows; CTA c takes b = c, c+P, ...
    for (int b = blockIdx.x; b < B; b += p.P) {
        if (bd[B + b] != 0) continue;
        const long long base = (long long)b * p.N * p.D;
        for (int idx = threadIdx.x; idx < p.N * p.D; idx += C::THREADS)
            st_final(p, base + idx, 0.f);
    }
    if (lo >= hi) return;

    if (warp >= NWC) {
        // ================================================================ producer warp
        if constexpr (C::SPLIT_REGS) setmaxnreg_dec<C::PRODUCER_REGS>();
        if (warp > NWC) return;  // the rest of the producer's warpgroup only gives its registers back
        const uint64_t pol = policy_evict_first();
        const int br = p.box_rows;
        const int tr = p.tail_rows;
        const int nsub = T / br;  // full boxes per tile: 1..8
        const int batch_tiles = 32 / nsub;
        TileCursor cur;
        cursor_init<T>(cur, bd, B, p.NGS, lo);
        int my_blk = 0;
        [[maybe_unused]] int fenced = -1;  // batch whose per-tensor maps are fenced for the TMA unit
        int it = 0;  // tiles of this CTA so far (< 2^31)
        for (long long g = lo; g < hi; ++g, ++it) {
            const int kk = it % batch_tiles;
            if (p.paged && kk == 0) {
                // Block ids of the next batch_tiles tiles: lane l reads full box (l % nsub) of tile (l / nsub).
                TileCursor c2 = cur;
                const int adv = lane / nsub;
                const bool live = (g + adv) < hi;
                if (live)
                    for (int a = 0; a < adv; ++a) cursor_next<T>(c2, bd, B, RS, p.NGS);
                my_blk = -2;
                if (live) {
                    const int t0 = c2.i * T + (lane % nsub) * br;
                    if (t0 < bd[B + c2.b])
                        my_blk = __ldg(&p.block_table[(long long)c2.b * p.bt_cols + t0 / p.block_size]);
                }
            }
            const int stage = it % C::STAGES;
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
            const int h = cur.h;
            const int gs = cur.gs;
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
                    if (KV == KV_I8 && p.aq_stage) bytes += (uint32_t)p.D * 2u;
                }
                if (p.paged) {
                    for (int s = 0; s < nsub; ++s) {
                        const int blk = blkbuf[s];
                        if (s * br < valid && !(blk >= 0 && blk < p.block_num)) badmask |= 1 << s;
                    }
                }
                for (int k = 0; k < nbox; ++k)
                    if (!((badmask >> ((k * rows_per) / br)) & 1)) bytes += box_bytes;
                if (p.mask_tma) bytes += (uint32_t)(C::MASK_LOADS * kMaskBox);
                if (badmask) record_error(p, kErrBadBlock);
                const int st = bd[b];
                tinfo[2 * stage] = make_int4(b, h, gs, cur.i);
                tinfo[2 * stage + 1] = make_int4(cur.tiles, valid, badmask, (st + cur.i * T) & 15);
                mbar_arrive_expect_tx(&full[stage], bytes);
                if (first) {
                    const char* qsrc = reinterpret_cast<const char*>(p.q) +
                                       ((long long)b * p.N + (long long)h * p.G + (long long)gs * p.GT) * p.D * 2;
                    uint8_t* qdst = sb + 2 * C::KT_BYTES;
                    for (int row = 0; row < rows; ++row)
                        bulk_g2s(qdst + row * C::QROW, qsrc + (long long)row * p.D * 2, (uint32_t)p.D * 2u, &full[stage]);
                    if (KV == KV_I8 && p.aq_stage)  // the key scales of kv head h (entry 0 of the leading axis)
                        bulk_g2s(sb + C::AQ_OFF, reinterpret_cast<const char*>(p.aq_scale) + (long long)h * p.D * 2,
                                 (uint32_t)p.D * 2u, &full[stage]);
                }
                if (p.mask_tma) {
                    // this tile's mask bytes, from the 16-byte boundary at or below its first position
                    const int x0 = st + cur.i * T;
#pragma unroll
                    for (int ml = 0; ml < C::MASK_LOADS; ++ml)
                        tma_load_2d(sb + C::MASK_OFF + ml * kMaskBox, &p.tmM, &full[stage], (x0 & ~15) + ml * kMaskBox,
                                    p.mask_bstride ? b : 0);
                }
                // one tensor per batch: its own maps, batch coordinate 0
                if constexpr (TL) {
                    if (b != fenced) {
                        for (int m = 0; m < 4; ++m) fence_tensormap_acquire(p.kv_maps + 4 * b + m);
                        fenced = b;
                    }
                }
                const CUtensorMap* mk = TL ? p.kv_maps + 4 * b + (tail ? 1 : 0) : (tail ? &p.tmKt : &p.tmK);
                const CUtensorMap* mv = TL ? p.kv_maps + 4 * b + (tail ? 3 : 2) : (tail ? &p.tmVt : &p.tmV);
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
                        w = TL ? 0 : b;
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
            cursor_next<T>(cur, bd, B, RS, p.NGS);
        }
        // On abort, let every issued copy land before the CTA's shared memory is released.
        if (*abort_flag && lane == 0) {
            for (long long k = (it > C::STAGES ? it - C::STAGES : 0); k < it; ++k)
                mbar_wait_bounded(&full[k % C::STAGES], (uint32_t)(k / C::STAGES) & 1, kWaitLimitNs);
        }
        return;
    }

    // ==================================================================== consumer warps
    if constexpr (C::SPLIT_REGS) setmaxnreg_inc<C::CONSUMER_REGS>();
    const int r = lane >> 2;
    const int q4 = lane & 3;
    constexpr int MTW = C::MTW;
    const int row0 = warp * C::KWT;
    const float sl2 = p.scale_log2;
    const int tid = threadIdx.x;  // 0 .. CONSUMERS-1

    uint32_t qf[KSTEPS][NT][2];
    float acc[MT][NT][4];
    float m_run[NT][2], l_run[NT][2];
    // int8: value antiquant factors of the channels this thread writes in a piece's epilogue,
    // loaded at the piece's first tile so their latency hides behind its tiles
    float vsc[NPOS][2], vof[NPOS][2];
#pragma unroll
    for (int n = 0; n < NPOS; ++n)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) vsc[n][hh] = vof[n][hh] = 0.f;

    // Masks the producer does not stage are read by the consumers, one tile ahead.
    const bool mask_regs = p.has_mask && !p.mask_tma;
    TileCursor mcur;
    uint32_t mask_next[MTW];
#pragma unroll
    for (int mt = 0; mt < MTW; ++mt) mask_next[mt] = 0u;
    if (mask_regs) {
        cursor_init<T>(mcur, bd, B, p.NGS, lo);
#pragma unroll
        for (int mt = 0; mt < MTW; ++mt) mask_next[mt] = load_mask_bits<NT, T>(p, mcur, bd, row0 + 16 * mt, r, q4);
    }
    int it = 0;
    for (long long g = lo; g < hi; ++g, ++it) {
        uint32_t mbits[MTW];
#pragma unroll
        for (int mt = 0; mt < MTW; ++mt) mbits[mt] = mask_next[mt];
        if (mask_regs && g + 1 < hi) {
            cursor_next<T>(mcur, bd, B, RS, p.NGS);
#pragma unroll
            for (int mt = 0; mt < MTW; ++mt)  // one tile ahead
                mask_next[mt] = load_mask_bits<NT, T>(p, mcur, bd, row0 + 16 * mt, r, q4);
        }
        const int stage = it % C::STAGES;
        const uint32_t round = (uint32_t)(it / C::STAGES);
        if (!mbar_wait_bounded(&full[stage], round & 1, kWaitLimitNs)) {
            if (lane == 0) record_error(p, kErrTimeout);
            *abort_flag = 1;
        }
        __syncwarp();
        if (*abort_flag) break;

        const int4 ia = tinfo[2 * stage];
        const int4 ib = tinfo[2 * stage + 1];
        const int b = ia.x, h = ia.y, gs = ia.z, i = ia.w;
        const int tiles = ib.x, valid = ib.y, badmask = ib.z;
        const bool first = (i == 0) || (g == lo);
        const bool last = (i == tiles - 1) || (g == hi - 1);
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
                                if (p.aq_stage) {
                                    const unsigned short us = *reinterpret_cast<const unsigned short*>(sb + C::AQ_OFF + d * 2);
                                    x *= p.q_bf16 ? __bfloat162float(__ushort_as_bfloat16(us)) : __half2float(__ushort_as_half(us));
                                } else {
                                    const long long si = p.aq_per_channel ? (long long)h * p.D + d : 0;
                                    x *= ld_half_as_float(p.aq_scale, si, p.q_bf16);
                                }
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
            if constexpr (KV == KV_I8) {
#pragma unroll
                for (int n = 0; n < NPOS; ++n) {
                    const int k = tid + n * CONSUMERS;
                    if (k < FRAG4 * 32) {
                        const int d0 = 16 * ((k >> 5) / NT) + 2 * ((k & 31) >> 2);
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const int d = d0 + hh;
                            if (d < p.D) {
                                const long long si = p.aq_per_channel ? (long long)(p.KV_N + h) * p.D + d : 1;
                                vsc[n][hh] = ld_half_as_float(p.aq_scale, si, p.q_bf16);
                                vof[n][hh] = ld_half_as_float(p.aq_offset, si, p.q_bf16) - kI8Bias;  // values carry +1152
                            }
                        }
                    }
                }
            }
        }

        if (p.mask_tma) {
            const uint8_t* ms = sb + C::MASK_OFF + ib.w;
#pragma unroll
            for (int mt = 0; mt < MTW; ++mt) {
                const int tl = row0 + 16 * mt + r, th = tl + 8;
                const uint32_t pat = ((tl < valid && ms[tl]) ? 0x3u : 0u) | ((th < valid && ms[th]) ? 0xCu : 0u);
                mbits[mt] = 0;
#pragma unroll
                for (int j = 0; j < NT; ++j) mbits[mt] |= pat << (4 * j);
            }
        }
        // Rows past the window end (or in a skipped block) may hold anything, NaN
        // included: clear this warp's invalid value rows so 0 * garbage stays 0.
        if constexpr (KV != KV_I8) {
            if (valid < row0 + C::KWT || badmask) {
                for (int idx = lane; idx < C::KWT * C::NCG * 8; idx += 32) {
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
        float s[MTW][NT][4], s2[MTW][NT][4];
#pragma unroll
        for (int mt = 0; mt < MTW; ++mt)
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) s[mt][j][e] = s2[mt][j][e] = 0.f;
        if constexpr (KV == KV_I8) {
#pragma unroll
            for (int ks = 0; ks < KSTEPS; ks += 2) {
#pragma unroll
                for (int mt = 0; mt < MTW; ++mt) {
                    const int lrow = row0 + 16 * mt + (lane & 7) + ((lane >> 3) & 1) * 8;
                    const int ch = ks + (lane >> 4);  // 16-byte chunk = 16 channels
                    const uint32_t addr = kbase + lrow * 128 + (ch >> 3) * (T * 128) + (((ch & 7) ^ (lrow & 7)) << 4);
                    uint32_t r0, r1, r2, r3;
                    ldsm_x4(addr, r0, r1, r2, r3);
                    r0 ^= 0x80808080u; r1 ^= 0x80808080u; r2 ^= 0x80808080u; r3 ^= 0x80808080u;
                    const uint32_t a0 = i8x2_to_f16x2_biased(r0, 0x4140), a2 = i8x2_to_f16x2_biased(r0, 0x4342);
                    const uint32_t a1 = i8x2_to_f16x2_biased(r1, 0x4140), a3 = i8x2_to_f16x2_biased(r1, 0x4342);
                    const uint32_t c0 = i8x2_to_f16x2_biased(r2, 0x4140), c2 = i8x2_to_f16x2_biased(r2, 0x4342);
                    const uint32_t c1 = i8x2_to_f16x2_biased(r3, 0x4140), c3 = i8x2_to_f16x2_biased(r3, 0x4342);
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        mma_16816<false>(s[mt][j], a0, a1, a2, a3, qf[ks][j][0], qf[ks][j][1]);
                        mma_16816<false>(s2[mt][j], c0, c1, c2, c3, qf[ks + 1][j][0], qf[ks + 1][j][1]);
                    }
                }
            }
        } else {
#pragma unroll
            for (int ks = 0; ks < KSTEPS; ++ks) {
#pragma unroll
                for (int mt = 0; mt < MTW; ++mt) {
                    const int lrow = row0 + 16 * mt + (lane & 7) + ((lane >> 3) & 1) * 8;
                    const int ch = 2 * ks + (lane >> 4);  // 16-byte chunk = 8 channels
                    const uint32_t addr = kbase + lrow * 128 + (ch >> 3) * (T * 128) + (((ch & 7) ^ (lrow & 7)) << 4);
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(addr, a0, a1, a2, a3);
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        // one n-tile: alternate two accumulators to halve the dependent chain
                        if (NT == 1 && (ks & 1)) mma_16816<MMA_BF16>(s2[mt][j], a0, a1, a2, a3, qf[ks][j][0], qf[ks][j][1]);
                        else mma_16816<MMA_BF16>(s[mt][j], a0, a1, a2, a3, qf[ks][j][0], qf[ks][j][1]);
                    }
                }
            }
        }

        // ---------------------------------------------------------- mask, online softmax
        uint32_t pb[MTW][NT][2];
        float x[MTW][NT][4];
#pragma unroll
        for (int mt = 0; mt < MTW; ++mt) {
            const int t_lo = row0 + 16 * mt + r, t_hi = t_lo + 8;
            bool ok_lo = t_lo < valid, ok_hi = t_hi < valid;
            if (badmask) {
                ok_lo = ok_lo && !((badmask >> (t_lo / p.box_rows)) & 1);
                ok_hi = ok_hi && !((badmask >> (t_hi / p.box_rows)) & 1);
            }
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const bool ok = ((e >> 1) ? ok_hi : ok_lo) && !((mbits[mt] >> (4 * j + e)) & 1u);
                    x[mt][j][e] = ok ? (s[mt][j][e] + s2[mt][j][e]) * sl2 : -INFINITY;
                }
        }
        bool moved = false;
        float mnew[NT][2];
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                float mx = fmaxf(x[0][j][u], x[0][j][u + 2]);
#pragma unroll
                for (int mt = 1; mt < MTW; ++mt) mx = fmaxf(mx, fmaxf(x[mt][j][u], x[mt][j][u + 2]));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                mnew[j][u] = fmaxf(m_run[j][u], mx);
                moved |= mnew[j][u] != m_run[j][u];
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
        for (int mt = 0; mt < MTW; ++mt)
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                float pr[4];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const float m_use = m_run[j][u] == -INFINITY ? 0.f : m_run[j][u];
                    pr[u] = ex2(x[mt][j][u] - m_use);
                    pr[u + 2] = ex2(x[mt][j][u + 2] - m_use);
                }
                const uint32_t h0 = pack2<MMA_BF16>(pr[0], pr[1]), h1 = pack2<MMA_BF16>(pr[2], pr[3]);
                if constexpr (KV == KV_I8) {
                    // row sums of the fp16-rounded probabilities the P.V MMAs see (keeps the value bias exact)
                    const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&h0));
                    const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&h1));
                    l_run[j][0] += f0.x + f1.x;
                    l_run[j][1] += f0.y + f1.y;
                } else {
                    l_run[j][0] += pr[0] + pr[2];
                    l_run[j][1] += pr[1] + pr[3];
                }
                pb[mt][j][0] = movmatrix_t(h0);
                pb[mt][j][1] = movmatrix_t(h1);
            }

        // ---------------------------------------------------------- O^T += V^T . P^T
        if constexpr (KV == KV_I8) {
#pragma unroll
            for (int c = 0; c < MT; c += 2) {
#pragma unroll
                for (int mt = 0; mt < MTW; ++mt) {
                    const int lrow = row0 + 16 * mt + (lane & 7) + ((lane >> 3) & 1) * 8;
                    const int ch = c + (lane >> 4);
                    const uint32_t addr = vbase + lrow * 128 + (ch >> 3) * (T * 128) + (((ch & 7) ^ (lrow & 7)) << 4);
                    uint32_t r0, r1, r2, r3;
                    ldsm_x4_t(addr, r0, r1, r2, r3);
                    r0 ^= 0x80808080u; r1 ^= 0x80808080u; r2 ^= 0x80808080u; r3 ^= 0x80808080u;
                    const uint32_t a0 = i8x2_to_f16x2_biased(r0, 0x4240), a1 = i8x2_to_f16x2_biased(r0, 0x4341);
                    const uint32_t a2 = i8x2_to_f16x2_biased(r1, 0x4240), a3 = i8x2_to_f16x2_biased(r1, 0x4341);
                    const uint32_t e0 = i8x2_to_f16x2_biased(r2, 0x4240), e1 = i8x2_to_f16x2_biased(r2, 0x4341);
                    const uint32_t e2 = i8x2_to_f16x2_biased(r3, 0x4240), e3 = i8x2_to_f16x2_biased(r3, 0x4341);
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        mma_16816<false>(acc[c][j], a0, a1, a2, a3, pb[mt][j][0], pb[mt][j][1]);
                        mma_16816<false>(acc[c + 1][j], e0, e1, e2, e3, pb[mt][j][0], pb[mt][j][1]);
                    }
                }
            }
        } else {
            const int mi = lane >> 3;
#pragma unroll
            for (int md = 0; md < MT; ++md) {
#pragma unroll
                for (int mt = 0; mt < MTW; ++mt) {
                    const int lrow = row0 + 16 * mt + (lane & 7) + (mi >> 1) * 8;
                    const int ch = 2 * md + (mi & 1);
                    const uint32_t addr = vbase + lrow * 128 + (ch >> 3) * (T * 128) + (((ch & 7) ^ (lrow & 7)) << 4);
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4_t(addr, a0, a1, a2, a3);
#pragma unroll
                    for (int j = 0; j < NT; ++j)
                        mma_16816<MMA_BF16>(acc[md][j], a0, a1, a2, a3, pb[mt][j][0], pb[mt][j][1]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);

        if (!last) continue;
        // ============================================================ piece epilogue
        // Accumulator element e of (md, j) in lane (r, q4) is query head gg = 8j + 2q4 + (e & 1)
        // and channel d = 16md + r + 8(e >> 1) (int8: 16md + 2r + (e >> 1)).  Fragments travel
        // between warps as lane-contiguous float4 ("position" k = (md * NT + j) * 32 + lane),
        // and the thread that combines position k sits in lane k % 32, so it owns the same heads.
        const long long seq_first = g - i;
        const bool complete = seq_first >= lo && seq_first + tiles <= hi;
        const long long obase = ((long long)b * p.N + (long long)h * p.G + (long long)gs * p.GT) * p.D;

        // writes one combined fragment position to the output
        auto put = [&](const float4& o, int k, bool live0, bool live1, int n) {
            const int gg0 = 8 * ((k >> 5) % NT) + 2 * (k & 3);
            const int d0 = (KV == KV_I8) ? 16 * ((k >> 5) / NT) + 2 * ((k & 31) >> 2) : 16 * ((k >> 5) / NT) + ((k & 31) >> 2);
            const float v[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int gg = gg0 + (e & 1);
                const int d = d0 + (e >> 1) * DSTEP;
                if (gg < GTv && d < p.D) {
                    float y = v[e];
                    if constexpr (KV == KV_I8) y = ((e & 1) ? live1 : live0) ? (y + vof[n][e >> 1]) * vsc[n][e >> 1] : 0.f;
                    st_final(p, obase + (long long)gg * p.D + d, y);
                }
            }
        };

        // (1) row sums of this warp; every warp publishes (m, l), warps MW.. their fragments
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
                    mlm[warp * GT_PAD + 8 * j + 2 * q4 + u] = m_run[j][u];
                    mll[warp * GT_PAD + 8 * j + 2 * q4 + u] = l_run[j][u];
                }
        }
        if (warp >= MW) {
#pragma unroll
            for (int md = 0; md < MT; ++md)
#pragma unroll
                for (int j = 0; j < NT; ++j)
                    mrg[((warp - MW) * FRAG4 + md * NT + j) * 32 + lane] =
                        make_float4(acc[md][j][0], acc[md][j][1], acc[md][j][2], acc[md][j][3]);
        }
        named_bar_sync(1, CONSUMERS);

        // (2) per head: M = max over warps, L = sum of l ex2(m - M), and the weight
        //     ex2(m_w - M) / L of each warp w; lane r of a column takes warp r.  Warps
        //     0..MW-1 then fold in warp w + MW, both sides weighted.
        float Mh[NT][2], Lh[NT][2], fs[NT][2], fo[NT][2];
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int gg = 8 * j + 2 * q4 + u;
                const int wr = r % NWC;
                const float mw = mlm[wr * GT_PAD + gg];
                float M = mw;
                M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 4));
                M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 8));
                M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 16));
                const float e = mw == -INFINITY ? 0.f : ex2(mw - M);
                float L = r < NWC ? mll[wr * GT_PAD + gg] * e : 0.f;
                L += __shfl_xor_sync(0xffffffffu, L, 4);
                L += __shfl_xor_sync(0xffffffffu, L, 8);
                L += __shfl_xor_sync(0xffffffffu, L, 16);
                const float wgt = L > 0.f ? e / L : 0.f;
                Mh[j][u] = M;
                Lh[j][u] = L;
                fs[j][u] = __shfl_sync(0xffffffffu, wgt, ((warp % NWC) << 2) | q4);
                fo[j][u] = __shfl_sync(0xffffffffu, wgt, (((warp + MW) % NWC) << 2) | q4);
            }
        if (warp < MW) {
#pragma unroll
            for (int md = 0; md < MT; ++md)
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    float4* slot = mrg + (warp * FRAG4 + md * NT + j) * 32 + lane;
                    if constexpr (NWC > MW) {
                        const float4 o = *slot;
                        *slot = make_float4(acc[md][j][0] * fs[j][0] + o.x * fo[j][0], acc[md][j][1] * fs[j][1] + o.y * fo[j][1],
                                            acc[md][j][2] * fs[j][0] + o.z * fo[j][0], acc[md][j][3] * fs[j][1] + o.w * fo[j][1]);
                    } else {
                        *slot = make_float4(acc[md][j][0] * fs[j][0], acc[md][j][1] * fs[j][1], acc[md][j][2] * fs[j][0],
                                            acc[md][j][3] * fs[j][1]);
                    }
                }
        }
        named_bar_sync(1, CONSUMERS);

        // (3) sum the MW normalised fragments: the output of a whole sequence; for a sequence
        //     that CTA boundaries cut, this piece's normalised O (with M and L per head): a
        //     partial in the CTA's slot, or, for the sequence's first piece, kept in registers
        //     for the merge below.  The first piece ends its CTA's range (the sequence runs on
        //     past it), so the CTA that holds it merges: the other pieces start their CTAs'
        //     ranges or fill them, and publish long before it finishes, as a rule.
        const bool head = seq_first >= lo;
        const int slot = 2 * (int)blockIdx.x + (seq_first <= lo ? 0 : 1);
        float* sp = p.partials + (long long)slot * p.slot_floats;
        float4 own[NPOS];
#pragma unroll
        for (int n = 0; n < NPOS; ++n) {
            const int k = tid + n * CONSUMERS;
            own[n] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (k < FRAG4 * 32) {
                float4 o = mrg[k];
#pragma unroll
                for (int w = 1; w < MW; ++w) {
                    const float4 v = mrg[w * FRAG4 * 32 + k];
                    o.x += v.x; o.y += v.y; o.z += v.z; o.w += v.w;
                }
                if (complete) {
                    const int j = (k >> 5) % NT;
                    float l0 = Lh[0][0], l1 = Lh[0][1];
#pragma unroll
                    for (int jj = 1; jj < NT; ++jj)
                        if (j == jj) l0 = Lh[jj][0], l1 = Lh[jj][1];
                    put(o, k, l0 > 0.f, l1 > 0.f, n);
                } else if (head) {
                    own[n] = o;
                } else {
                    reinterpret_cast<float4*>(sp)[k] = o;
                }
            }
        }
        int publish = -1;  // int8: the counter this piece arrives on, after the last barrier
        if (!complete) {
            const int c_first = cta_of(seq_first, sbounds, p.P);
            const int c_last = cta_of(seq_first + tiles - 1, sbounds, p.P);
            const int npieces = c_last - c_first + 1;  // >= 2: the sequence runs past a range end
            unsigned int* ctr = p.counters + c_first;  // CTA c_first starts no other cut sequence
            if (!head) {
                // (4) publish: M and L beside the partial, then one release add on the sequence's
                //     counter (the partial, written by every consumer thread before a barrier, is
                //     visible before the add); nothing to wait for
                if (warp == 0 && r == 0) {
#pragma unroll
                    for (int j = 0; j < NT; ++j)
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            sp[GT_PAD * DPAD + 8 * j + 2 * q4 + u] = Mh[j][u];
                            sp[GT_PAD * DPAD + GT_PAD + 8 * j + 2 * q4 + u] = Lh[j][u];
                        }
                }
                if constexpr (KV == KV_I8) {
                    // int8 consumers are the busier side: the add follows the epilogue's last
                    // barrier below, so that its wait holds thread 0 alone (measured 0.6 us a
                    // call better here; with 16-bit caches, where the copies pace the kernel,
                    // the same order measured level or 0.3 us worse)
                    publish = c_first;
                } else {
                    named_bar_sync(1, CONSUMERS);
                    if (tid == 0) red_add_release_gpu(ctr, 1u);
                }
            } else {
                // (4) merge: wait until the other npieces - 1 pieces have published (acquire),
                //     then weigh piece k by L_k 2^(M_k - M) / sum_j L_j 2^(M_j - M), in piece
                //     order (this piece is piece 0); deterministic, no float atomics
                float* pm = reinterpret_cast<float*>(mrg);  // [npieces][GT_PAD] M, then the head's total
                float* pw = pm + npieces * GT_PAD;            // [npieces][GT_PAD] L, then the piece weights
                named_bar_sync(1, CONSUMERS);                 // step (3) has read mrg
                if (warp == 0 && r == 0) {
#pragma unroll
                    for (int j = 0; j < NT; ++j)
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            pm[8 * j + 2 * q4 + u] = Mh[j][u];
                            pw[8 * j + 2 * q4 + u] = Lh[j][u];
                        }
                }
                if (tid == 0) {
                    const uint64_t t0 = globaltimer_ns();
                    while (ld_acquire_gpu(ctr) != (unsigned int)(npieces - 1)) {
                        if (globaltimer_ns() - t0 > kWaitLimitNs) {
                            record_error(p, kErrTimeout);
                            break;
                        }
                    }
                    // every other piece has arrived: no other access to the counter in this call,
                    // so it goes back to zero for the next call (read after this grid completes)
                    *reinterpret_cast<volatile unsigned int*>(ctr) = 0u;
                }
                named_bar_sync(1, CONSUMERS);
                // pieces 1.. start the ranges of CTAs c_first + 1, ...: slot 0 of each
                auto slot_of = [&](int k) { return p.partials + (long long)(2 * (c_first + k)) * p.slot_floats; };
                // piece 1's fragments do not depend on the weights: load them now
                float4 pre1[NPOS];
#pragma unroll
                for (int n = 0; n < NPOS; ++n) {
                    const int k = tid + n * CONSUMERS;
                    pre1[n] = k < FRAG4 * 32 ? __ldcg(reinterpret_cast<const float4*>(slot_of(1)) + k)
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
                }
                for (int x2 = tid; x2 < (npieces - 1) * GT_PAD; x2 += CONSUMERS) {
                    const int k = 1 + x2 / GT_PAD, gg = x2 % GT_PAD;
                    const float* pp = slot_of(k) + GT_PAD * DPAD;
                    pm[k * GT_PAD + gg] = __ldcg(pp + gg);
                    pw[k * GT_PAD + gg] = __ldcg(pp + GT_PAD + gg);
                }
                named_bar_sync(1, CONSUMERS);
                if (tid < GT_PAD) {
                    float M = -INFINITY;
                    for (int k = 0; k < npieces; ++k) M = fmaxf(M, pm[k * GT_PAD + tid]);
                    float S = 0.f;
                    for (int k = 0; k < npieces; ++k) {
                        const float mk = pm[k * GT_PAD + tid];
                        const float wk = mk == -INFINITY ? 0.f : pw[k * GT_PAD + tid] * ex2(mk - M);
                        pw[k * GT_PAD + tid] = wk;
                        S += wk;
                    }
                    const float inv = S > 0.f ? 1.f / S : 0.f;
                    for (int k = 0; k < npieces; ++k) pw[k * GT_PAD + tid] *= inv;
                    pm[tid] = S;  // column tid is this thread's alone
                }
                named_bar_sync(1, CONSUMERS);
#pragma unroll
                for (int n = 0; n < NPOS; ++n) {
                    const int k = tid + n * CONSUMERS;
                    if (k < FRAG4 * 32) {
                        const int gg0 = 8 * ((k >> 5) % NT) + 2 * (k & 3);
                        float4 o;
                        {
                            const float w0 = pw[gg0], w1 = pw[gg0 + 1];
                            const float v0 = pw[GT_PAD + gg0], v1 = pw[GT_PAD + gg0 + 1];
                            o = make_float4(w0 * own[n].x + v0 * pre1[n].x, w1 * own[n].y + v1 * pre1[n].y,
                                            w0 * own[n].z + v0 * pre1[n].z, w1 * own[n].w + v1 * pre1[n].w);
                        }
                        int pc = 2;
                        for (; pc + 4 <= npieces; pc += 4) {
                            float4 v[4];
#pragma unroll
                            for (int t = 0; t < 4; ++t)
                                v[t] = __ldcg(reinterpret_cast<const float4*>(slot_of(pc + t)) + k);
#pragma unroll
                            for (int t = 0; t < 4; ++t) {
                                const float w0 = pw[(pc + t) * GT_PAD + gg0], w1 = pw[(pc + t) * GT_PAD + gg0 + 1];
                                o.x += w0 * v[t].x; o.y += w1 * v[t].y; o.z += w0 * v[t].z; o.w += w1 * v[t].w;
                            }
                        }
                        for (; pc < npieces; ++pc) {
                            const float4 v = __ldcg(reinterpret_cast<const float4*>(slot_of(pc)) + k);
                            const float w0 = pw[pc * GT_PAD + gg0], w1 = pw[pc * GT_PAD + gg0 + 1];
                            o.x += w0 * v.x; o.y += w1 * v.y; o.z += w0 * v.z; o.w += w1 * v.w;
                        }
                        put(o, k, pm[gg0] > 0.f, pm[gg0 + 1] > 0.f, n);
                    }
                }
            }
        }
        named_bar_sync(1, CONSUMERS);
        if (KV == KV_I8 && publish >= 0 && tid == 0) red_add_release_gpu(p.counters + publish, 1u);
    }
}

template <int KV, int DPAD, int NT, bool TL = false>
cudaError_t launch_decode(const DecodeParams& p, int grid, cudaStream_t stream) {
    using C = DecodeCfg<KV, DPAD, NT>;
    static std::atomic<bool> configured[kMaxDevices];  // per device: the attributes are set per device
    const int dev = current_device_slot();
    if (dev < 0) return cudaErrorInvalidDevice;
    if (!configured[dev].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(decode_kernel<KV, DPAD, NT, TL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM);
        if (e != cudaSuccess) return e;
        if constexpr (C::SPLIT_REGS) {
            // setmaxnreg.inc draws on the registers the block was launched with: refuse to launch
            // a build whose register count cannot cover the split (the increase would never return).
            cudaFuncAttributes fa;
            e = cudaFuncGetAttributes(&fa, decode_kernel<KV, DPAD, NT, TL>);
            if (e != cudaSuccess) return e;
            if ((long long)fa.numRegs * C::THREADS < C::REG_POOL_NEEDED) return cudaErrorInvalidConfiguration;
        }
        configured[dev].store(true, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_kernel<KV, DPAD, NT, TL>, p);
}

}  // namespace ifa
