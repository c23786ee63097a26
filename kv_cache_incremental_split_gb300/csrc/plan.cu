// Host planning shared by ifa_run and ifa_run_noalloc: parameter validation
// (constraints of the "IncreFlashAttention" README, 约束说明, and of the
// "aclnnIncreFlashAttentionV2" page, Parameters / Constraints), kernel
// variant choice, per-batch windows (actualSeqLengths, kv左padding), the
// split plan, TMA tensor-map encoding and launch-parameter filling.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "decode.cuh"

namespace ifa {

DecodeLaunchFn decode_launcher_bf16(int dpad, int nt);
DecodeLaunchFn decode_launcher_f16(int dpad, int nt);
DecodeLaunchFn decode_launcher_i8(int dpad, int nt);

DecodeLaunchFn decode_launcher_tl_bf16(int dpad, int nt);
DecodeLaunchFn decode_launcher_tl_f16(int dpad, int nt);
DecodeLaunchFn decode_launcher_tl_i8(int dpad, int nt);

DecodeLaunchFn decode_launcher(int kv_kind, int dpad, int nt, bool tensorlist) {
    if (tensorlist) {
        if (kv_kind == KV_BF16) return decode_launcher_tl_bf16(dpad, nt);
        if (kv_kind == KV_F16) return decode_launcher_tl_f16(dpad, nt);
        return decode_launcher_tl_i8(dpad, nt);
    }
    if (kv_kind == KV_BF16) return decode_launcher_bf16(dpad, nt);
    if (kv_kind == KV_F16) return decode_launcher_f16(dpad, nt);
    return decode_launcher_i8(dpad, nt);
}

template <int KV, int DPAD, int NT>
static void cfg_numbers(int* slot, int* smem, int* tile, int* threads) {
    using C = DecodeCfg<KV, DPAD, NT>;
    *slot = C::SLOT_FLOATS;
    *smem = C::SMEM;
    *tile = C::T;
    *threads = C::THREADS;
}

bool decode_cfg(int kv, int dpad, int nt, int* slot, int* smem, int* tile, int* threads) {
#define IFA_CFG(K, Dp, N)                                  \
    if (kv == K && dpad == Dp && nt == N) {                \
        cfg_numbers<K, Dp, N>(slot, smem, tile, threads);  \
        return true;                                       \
    }
    IFA_CFG(KV_BF16, 64, 1) IFA_CFG(KV_BF16, 64, 2) IFA_CFG(KV_BF16, 128, 1) IFA_CFG(KV_BF16, 128, 2)
    IFA_CFG(KV_BF16, 256, 1)
    IFA_CFG(KV_F16, 64, 1) IFA_CFG(KV_F16, 64, 2) IFA_CFG(KV_F16, 128, 1) IFA_CFG(KV_F16, 128, 2)
    IFA_CFG(KV_F16, 256, 1)
    IFA_CFG(KV_I8, 128, 1) IFA_CFG(KV_I8, 128, 2) IFA_CFG(KV_I8, 256, 1)
#undef IFA_CFG
    return false;
}

bool params_are_valid(const ifa_params& p) {
    if (p.B < 0 || p.B > 65536) return false;
    if (p.numHeads < 1 || p.numHeads > 256) return false;
    const int64_t kvn = p.numKeyValueHeads == 0 ? p.numHeads : p.numKeyValueHeads;
    if (kvn < 1 || p.numHeads % kvn != 0) return false;
    if (p.headDim < 1 || p.headDim > 512) return false;
    if (p.q_dtype != IFA_F16 && p.q_dtype != IFA_BF16) return false;
    if (p.kv_dtype == IFA_I8) {
        if (p.antiquant != IFA_ANTIQUANT_PER_CHANNEL && p.antiquant != IFA_ANTIQUANT_PER_TENSOR) return false;
        if (p.headDim % 16 != 0) return false;  // 16-byte TMA strides
    } else {
        if (p.kv_dtype != p.q_dtype) return false;
        if (p.antiquant != IFA_ANTIQUANT_NONE) return false;
    }
    if (p.headDim % 8 != 0) return false;  // 16-byte TMA strides and bulk-copy rows
    if (p.inputLayout < IFA_LAYOUT_BSH || p.inputLayout > IFA_LAYOUT_BNSD) return false;
    if (p.kvFormat == IFA_KV_CONTIG) {
        if (p.maxSeqLen < 1 || p.maxSeqLen > INT32_MAX / 2) return false;
    } else if (p.kvFormat == IFA_KV_PAGED_NBSD || p.kvFormat == IFA_KV_PAGED_BSH) {
        if (p.kvFormat == IFA_KV_PAGED_NBSD && p.inputLayout != IFA_LAYOUT_BNSD) return false;
        const int64_t align = p.kv_dtype == IFA_I8 ? 32 : 16;
        if (p.blockSize < 1 || p.blockSize > 512 || p.blockSize % align != 0) return false;
        if (p.blockNum < 1 || p.blockNum > INT32_MAX) return false;
        if (p.blockTableCols < 1 || p.blockTableCols * p.blockSize > INT32_MAX / 2) return false;
        if (p.has_kv_padding) return false;  // left padding of a paged cache is not defined
    } else if (p.kvFormat == IFA_KV_TENSORLIST) {
        if (p.B > kInlineB) return false;  // README: at most 256 tensors in the list
        if (p.maxSeqLen < 1 || p.maxSeqLen > INT32_MAX / 2) return false;
        if (p.has_kv_padding) return false;  // left padding of per-batch tensors is not defined
    } else {
        return false;
    }
    if (p.has_mask) {
        if (p.mask_dtype != IFA_BOOL && p.mask_dtype != IFA_I8 && p.mask_dtype != IFA_U8) return false;
        if (p.maskB != 1 && p.maskB != p.B) return false;
        if (p.maskN != 1 && p.maskN != p.numHeads) return false;
        if (p.maskS < 1 || p.maskS > INT32_MAX / 2) return false;
    }
    if (!std::isfinite(p.scaleValue)) return false;
    if (p.splitTiles < 0) return false;
    if (p.out_dtype == IFA_I8) {
        // README: FLOAT32 parameters, or BFLOAT16 ones with a bf16 query
        if (p.quant2 != IFA_ANTIQUANT_PER_CHANNEL && p.quant2 != IFA_ANTIQUANT_PER_TENSOR) return false;
        if (p.quant2_dtype != IFA_F32 && !(p.quant2_dtype == IFA_BF16 && p.q_dtype == IFA_BF16)) return false;
    } else if (p.quant2 != IFA_ANTIQUANT_NONE) {
        return false;
    }
    return true;
}

static int64_t gcd64(int64_t a, int64_t b) {
    while (b) {
        const int64_t t = a % b;
        a = b;
        b = t;
    }
    return a;
}

ifa_status choose_kernel(const ifa_params& p, KernelChoice* kc) {
    if (!params_are_valid(p)) return IFA_ERR_PARAM_INVALID;
    kc->KV_N = (int)(p.numKeyValueHeads == 0 ? p.numHeads : p.numKeyValueHeads);
    kc->G = (int)(p.numHeads / kc->KV_N);
    kc->kv_kind = p.kv_dtype == IFA_I8 ? KV_I8 : (p.q_dtype == IFA_BF16 ? KV_BF16 : KV_F16);
    kc->es = p.kv_dtype == IFA_I8 ? 1 : 2;
    const int cg = 128 / kc->es;
    kc->dpad = (int)((p.headDim + cg - 1) / cg * cg);
    if (kc->dpad == 192) kc->dpad = 256;
    if (kc->dpad > 256) return IFA_ERR_PARAM_INVALID;  // head dims above 256: outside this kernel set
    kc->GT = std::min(kc->G, kc->dpad >= 256 ? 8 : 16);
    kc->NT = (kc->GT + 7) / 8;
    kc->NGS = (kc->G + kc->GT - 1) / kc->GT;
    kc->launch = decode_launcher(kc->kv_kind, kc->dpad, kc->NT, p.kvFormat == IFA_KV_TENSORLIST);
    if (!kc->launch || !decode_cfg(kc->kv_kind, kc->dpad, kc->NT, &kc->slot_floats, &kc->smem, &kc->T, &kc->threads))
        return IFA_ERR_PARAM_INVALID;
    // Full tiles move in boxes as large as the tile (or the cache block); a window's last
    // tile moves in boxes of at most 32 rows, so rows past the window end are not fetched.
    kc->box_rows = kc->T;
    if (kv_paged(p)) kc->box_rows = (int)gcd64(kc->T, p.blockSize);
    kc->tail_rows = std::min(kc->box_rows, 32);
    const int tile_bytes = 2 * kc->T * kc->dpad * kc->es;
    const bool i8 = kc->kv_kind == KV_I8;
    kc->piece_cost = std::max(1, (int)((16LL * (i8 ? kPieceCostBytesI8 : kPieceCostBytes)) / tile_bytes));
    kc->cut_cost = std::max(kc->piece_cost, (int)((16LL * (i8 ? kCutCostBytesI8 : kCutCostBytes)) / tile_bytes));
    return IFA_OK;
}

ifa_status build_windows(const ifa_params& p, const KernelChoice& kc, const int64_t* lens, const int64_t* pads,
                         int64_t n_pads, int32_t* bd, int64_t* W_out, int* max_seq_tiles) {
    const int B = (int)p.B;
    const bool paged = kv_paged(p);
    const bool left_pad = p.has_kv_padding && lens != nullptr;
    const int RS = kc.KV_N * kc.NGS;
    const int64_t cap = paged ? p.blockTableCols * p.blockSize : p.maxSeqLen;
    int64_t W = 0;
    int mst = 0;
    for (int b = 0; b < B; ++b) {
        int64_t len = lens ? lens[b] : p.maxSeqLen;
        int64_t st = 0;
        if (len < 0) return IFA_ERR_PARAM_INVALID;
        if (left_pad) {
            int64_t pad = pads[n_pads == 1 ? 0 : b];
            if (pad < 0) pad = 0;  // negative kvPaddingSize counts as 0
            st = p.maxSeqLen - pad - len;
            if (st < 0 || p.maxSeqLen - pad < 0) {  // window start or end below 0: all-zero row
                st = 0;
                len = 0;
            }
        } else if (len > cap) {
            return IFA_ERR_PARAM_INVALID;
        }
        if (p.has_mask && len > 0 && st + len > p.maskS) return IFA_ERR_PARAM_INVALID;
        bd[b] = (int32_t)st;
        bd[B + b] = (int32_t)len;
        bd[2 * B + b] = (int32_t)W;
        const int tiles = (int)((len + kc.T - 1) / kc.T);
        mst = std::max(mst, tiles);
        W += (int64_t)tiles * RS;
        if (W > INT32_MAX) return IFA_ERR_PARAM_INVALID;
    }
    bd[3 * B] = (int32_t)W;
    *W_out = W;
    *max_seq_tiles = mst;
    return IFA_OK;
}

int choose_grid(const ifa_params& p, int64_t W, int max_seq_tiles, int P_max) {
    if (W == 0) return 1;
    int64_t min_share = p.splitTiles > 0 ? p.splitTiles : std::min<int64_t>(max_seq_tiles, kMinPieceTiles);
    min_share = std::max<int64_t>(min_share, 1);
    return (int)std::max<int64_t>(1, std::min<int64_t>(P_max, (W + min_share - 1) / min_share));
}

// Without splitTiles the CTA ranges balance a cost in 1/16 tiles: 16 per tile, plus
// piece_cost for a sequence that one CTA holds whole and cut_cost for each piece of a
// sequence that a range boundary cuts.  A greedy walk fills each range up to a cap X,
// closing it when the next piece would exceed X: it cuts the sequence when at least one tile
// still fits after the cut cost, and otherwise ends the range at the sequence start.  X is
// the smallest cap (binary search) with which P ranges suffice, so the costliest range is as
// cheap as this walk can make it.  The RS sequences of a batch have equal length, so a walk
// costs O(B + P).  With splitTiles the shares are equal (c W / P).  Every CTA gets at least
// one tile (P <= W), so the CTAs a sequence spans each hold one of its pieces.
namespace {
// Ranges the walk needs under cap X (stops counting past P); writes bounds[1..] when given.
int split_walk(const int32_t* bd, int B, int64_t RS, int T, int64_t Ec, int64_t Ex, int64_t X, int P,
               int32_t* bounds) {
    int n = 1;          // ranges opened so far
    int64_t cur = 0;    // cost of the open range
    int64_t g0 = 0;     // first tile of batch b
    auto close = [&](int64_t at) -> bool {
        if (bounds && n < P) bounds[n] = (int32_t)at;
        ++n;
        cur = 0;
        return n <= P;
    };
    for (int b = 0; b < B; ++b) {
        const int64_t t = ((int64_t)bd[B + b] + T - 1) / T;
        if (t == 0) continue;
        const int64_t whole = 16 * t + Ec;
        int64_t r = 0, pos = 0;  // sequences of b finished; tiles of sequence r in closed ranges
        while (r < RS) {
            if (pos == 0) {
                const int64_t fit = std::min(RS - r, std::max<int64_t>(0, X - cur) / whole);
                cur += fit * whole;
                r += fit;
                if (r == RS) break;
            }
            const int64_t g = g0 + r * t;  // first tile of sequence r
            const int64_t left = t - pos;
            const int64_t piece = 16 * left + (pos > 0 ? Ex : Ec);
            if (cur + piece <= X) {  // a continuation piece that fits
                cur += piece;
                ++r;
                pos = 0;
                continue;
            }
            const int64_t k = (X - cur - Ex) / 16;  // tiles a cut piece may take here
            if ((k >= 1 && k < left) || cur == 0) {
                if (cur == 0 && left == 1) {  // a single tile larger than the cap: take it
                    cur += piece;
                    ++r;
                    pos = 0;
                    continue;
                }
                const int64_t kk = std::max<int64_t>(1, std::min(k, left - 1));
                cur += 16 * kk + Ex;
                pos += kk;
                if (!close(g + pos)) return n;
            } else {
                if (!close(g + pos)) return n;  // pos is 0: the range ends at the sequence start
            }
        }
        g0 += RS * t;
    }
    return n;
}
}  // namespace

void build_bounds(const ifa_params& p, const KernelChoice& kc, const int32_t* bd, int64_t W, int P, int32_t* bounds) {
    const int B = (int)p.B;
    bounds[0] = 0;
    bounds[P] = (int32_t)W;
    if (p.splitTiles > 0 || P == 1) {
        for (int c = 1; c < P; ++c) bounds[c] = (int32_t)((int64_t)c * W / P);
        return;
    }
    const int64_t RS = (int64_t)kc.KV_N * kc.NGS;
    const int64_t Ec = kc.piece_cost, Ex = std::max<int64_t>(kc.cut_cost, kc.piece_cost);
    int64_t nseq = 0;
    for (int b = 0; b < B; ++b)
        if (bd[B + b] > 0) nseq += RS;
    const int64_t base = 16 * W + Ec * nseq;
    // Every range but the last ends with less than Ex + 16 of its cap unused, so P ranges of at
    // least the mean cost with a cut at every boundary, plus that slack, always suffice.
    int64_t lo = std::max<int64_t>(1, base / P), hi = (base + 2 * Ex * (int64_t)P) / P + Ex + 17;
    while (lo < hi) {
        const int64_t mid = lo + (hi - lo) / 2;
        if (split_walk(bd, B, RS, kc.T, Ec, Ex, mid, P, nullptr) <= P) hi = mid;
        else lo = mid + 1;
    }
    for (int c = 1; c < P; ++c) bounds[c] = (int32_t)W;
    split_walk(bd, B, RS, kc.T, Ec, Ex, lo, P, bounds);
    for (int c = 1; c < P; ++c) bounds[c] = std::max(bounds[c], bounds[c - 1] + 1);
    for (int c = P - 1; c >= 1; --c) bounds[c] = std::min(bounds[c], bounds[c + 1] - 1);
}

static bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

ifa_status check_run_pointers(const ifa_params& p, const void* query, const void* key, const void* value,
                              const void* attenMask, const int64_t* actualSeqLengths, const int64_t* kvPaddingSize,
                              int64_t n_kv_padding, const int32_t* blockTable, const void* antiquantScale,
                              const void* antiquantOffset, const void* quantScale2, const void* quantOffset2,
                              const void* attentionOut) {
    const bool paged = kv_paged(p);
    if (!query || !key || !value || !attentionOut) return IFA_ERR_PARAM_NULLPTR;
    if (p.has_mask && !attenMask) return IFA_ERR_PARAM_NULLPTR;
    if (paged && (!blockTable || !actualSeqLengths)) return IFA_ERR_PARAM_NULLPTR;
    if (p.antiquant != IFA_ANTIQUANT_NONE && (!antiquantScale || !antiquantOffset)) return IFA_ERR_PARAM_NULLPTR;
    if (p.has_kv_padding && !kvPaddingSize) return IFA_ERR_PARAM_NULLPTR;
    if (!aligned(query, 16) || !aligned(key, 16) || !aligned(value, 16) || !aligned(attentionOut, 16))
        return IFA_ERR_PARAM_INVALID;
    if (blockTable && !aligned(blockTable, 4)) return IFA_ERR_PARAM_INVALID;
    if (p.antiquant != IFA_ANTIQUANT_NONE && (!aligned(antiquantScale, 2) || !aligned(antiquantOffset, 2)))
        return IFA_ERR_PARAM_INVALID;
    if (p.has_kv_padding && actualSeqLengths && n_kv_padding != 1 && n_kv_padding != p.B)
        return IFA_ERR_PARAM_INVALID;
    if (p.out_dtype == IFA_I8) {
        if (!quantScale2) return IFA_ERR_PARAM_NULLPTR;
        const uintptr_t a = p.quant2_dtype == IFA_F32 ? 4 : 2;
        if (!aligned(quantScale2, a) || (quantOffset2 && !aligned(quantOffset2, a))) return IFA_ERR_PARAM_INVALID;
    }
    return IFA_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return (EncodeTiledFn) nullptr;
        }
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

bool encode_kv_map(const ifa_params& p, const KernelChoice& kc, const void* base, int box_rows, CUtensorMap* map) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const uint64_t E = (uint64_t)kc.es, D = (uint64_t)p.headDim, KVN = (uint64_t)kc.KV_N;
    const bool contig = p.kvFormat == IFA_KV_CONTIG;
    const bool bnsd_like = p.kvFormat == IFA_KV_PAGED_NBSD || (contig && p.inputLayout == IFA_LAYOUT_BNSD);
    const uint64_t S = contig ? (uint64_t)p.maxSeqLen : (uint64_t)p.blockSize;
    cuuint64_t dims[4] = {D, S, KVN, contig ? (uint64_t)p.B : (uint64_t)p.blockNum};
    cuuint64_t strides[3];
    if (bnsd_like) {  // (..., KV_N, S, D)
        strides[0] = D * E;
        strides[1] = S * D * E;
        strides[2] = KVN * S * D * E;
    } else {  // (..., S, KV_N, D)
        strides[0] = KVN * D * E;
        strides[1] = D * E;
        strides[2] = S * KVN * D * E;
    }
    cuuint32_t box[4] = {(cuuint32_t)(128 / kc.es), (cuuint32_t)box_rows, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUtensorMapDataType dt = kc.kv_kind == KV_I8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : (kc.kv_kind == KV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                            : CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
    return enc(map, dt, 4, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_kv_maps(const ifa_params& p, const KernelChoice& kc, const void* key, const void* value, DecodeParams& dp) {
    return encode_kv_map(p, kc, key, kc.box_rows, &dp.tmK) && encode_kv_map(p, kc, value, kc.box_rows, &dp.tmV) &&
           encode_kv_map(p, kc, key, kc.tail_rows, &dp.tmKt) && encode_kv_map(p, kc, value, kc.tail_rows, &dp.tmVt);
}

bool encode_mask_map(const ifa_params& p, const KernelChoice& kc, const void* mask, DecodeParams& dp) {
    dp.mask_tma = 0;
    if (!p.has_mask || p.maskN != 1 || p.maskS % 16 != 0 || (reinterpret_cast<uintptr_t>(mask) % 16) != 0) return true;
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    // A tile's mask bytes plus the up-to-15-byte lead from rounding its start down to 16 bytes
    // come in one to three kMaskBox-byte boxes.
    cuuint64_t dims[2] = {(cuuint64_t)p.maskS, (cuuint64_t)p.maskB};
    cuuint64_t strides[1] = {(cuuint64_t)p.maskS};
    cuuint32_t box[2] = {(cuuint32_t)kMaskBox, 1};
    cuuint32_t estr[2] = {1, 1};
    if (enc(&dp.tmM, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(mask), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    dp.mask_tma = 1;
    return true;
}

void fill_decode_params(DecodeParams& dp, const ifa_params& p, const KernelChoice& kc, const void* query,
                        const void* attenMask, const int32_t* blockTable, const void* antiquantScale,
                        const void* antiquantOffset, const void* quantScale2, const void* quantOffset2,
                        void* attentionOut, int64_t W, int P) {
    dp.q = query;
    dp.out = attentionOut;
    dp.mask = reinterpret_cast<const uint8_t*>(attenMask);
    dp.block_table = blockTable;
    dp.aq_scale = antiquantScale;
    dp.aq_offset = antiquantOffset;
    dp.W = W;
    dp.P = P;
    dp.B = (int)p.B;
    dp.N = (int)p.numHeads;
    dp.KV_N = kc.KV_N;
    dp.D = (int)p.headDim;
    dp.G = kc.G;
    dp.GT = kc.GT;
    dp.NGS = kc.NGS;
    dp.q_bf16 = p.q_dtype == IFA_BF16;
    dp.paged = kv_paged(p);
    dp.block_size = (int)p.blockSize;
    dp.bt_cols = (int)p.blockTableCols;
    dp.block_num = (int)p.blockNum;
    dp.box_rows = kc.box_rows;
    dp.tail_rows = kc.tail_rows;
    dp.has_mask = p.has_mask != 0;
    dp.mask_bstride = (p.has_mask && p.maskB > 1) ? p.maskN * p.maskS : 0;
    dp.mask_nstride = (p.has_mask && p.maskN > 1) ? p.maskS : 0;
    dp.aq_per_channel = p.antiquant == IFA_ANTIQUANT_PER_CHANNEL;
    // a bulk copy moves a key scale row: 16-byte aligned source (rows are D * 2 bytes, D % 8 == 0)
    dp.aq_stage = dp.aq_per_channel && aligned(antiquantScale, 16);
    dp.scale_log2 = (float)(p.scaleValue * 1.4426950408889634);
    dp.slot_floats = kc.slot_floats;
    dp.out_i8 = p.out_dtype == IFA_I8;
    dp.q2_per_channel = dp.out_i8 && p.quant2 == IFA_ANTIQUANT_PER_CHANNEL;
    dp.q2_bf16 = dp.out_i8 && p.quant2_dtype == IFA_BF16;
    dp.q2_scale = dp.out_i8 ? quantScale2 : nullptr;
    dp.q2_offset = dp.out_i8 ? quantOffset2 : nullptr;
}

}  // namespace ifa
