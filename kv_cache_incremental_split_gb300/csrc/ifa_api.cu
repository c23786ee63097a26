// C ABI of the decode-attention library: validation, split planning, tensor
// map encoding and kernel launches.  Parameter checks follow the constraints
// of the "IncreFlashAttention" README (约束说明) and the
// "aclnnIncreFlashAttentionV2" page (Parameters, Constraints, Return Value).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "../../include/ifa.h"
#include "decode.cuh"

namespace ifa {
DecodeLaunchFn decode_launcher_bf16(int dpad, int nt);
DecodeLaunchFn decode_launcher_f16(int dpad, int nt);
DecodeLaunchFn decode_launcher_i8(int dpad, int nt);

DecodeLaunchFn decode_launcher(int kv_kind, int dpad, int nt) {
    if (kv_kind == KV_BF16) return decode_launcher_bf16(dpad, nt);
    if (kv_kind == KV_F16) return decode_launcher_f16(dpad, nt);
    return decode_launcher_i8(dpad, nt);
}

template <int KV, int DPAD, int NT>
static void cfg_numbers(int* slot, int* smem) {
    *slot = DecodeCfg<KV, DPAD, NT>::SLOT_FLOATS;
    *smem = DecodeCfg<KV, DPAD, NT>::SMEM;
}

static bool cfg_lookup(int kv, int dpad, int nt, int* slot, int* smem) {
#define IFA_CFG(K, Dp, N)                      \
    if (kv == K && dpad == Dp && nt == N) {    \
        cfg_numbers<K, Dp, N>(slot, smem);     \
        return true;                           \
    }
    IFA_CFG(KV_BF16, 64, 1) IFA_CFG(KV_BF16, 64, 2) IFA_CFG(KV_BF16, 128, 1) IFA_CFG(KV_BF16, 128, 2)
    IFA_CFG(KV_BF16, 256, 1)
    IFA_CFG(KV_F16, 64, 1) IFA_CFG(KV_F16, 64, 2) IFA_CFG(KV_F16, 128, 1) IFA_CFG(KV_F16, 128, 2)
    IFA_CFG(KV_F16, 256, 1)
    IFA_CFG(KV_I8, 128, 1) IFA_CFG(KV_I8, 128, 2) IFA_CFG(KV_I8, 256, 1)
#undef IFA_CFG
    return false;
}
}  // namespace ifa

using namespace ifa;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

struct ifa_plan {
    ifa_params prm;
    int KV_N, G, GT, NGS, NT, DPAD, kv_kind, es;
    int num_sms, P_max, device;
    int slot_floats, box_rows;
    size_t partial_bytes, ext_offset, ws_bytes;
    int* d_err;
    DecodeLaunchFn launch;
    const void* last_k;
    const void* last_v;
    DecodeParams* dp;
    CombineParams* cp;
    int64_t last_launches;
    std::vector<int32_t> bdata;
};

static int64_t gcd64(int64_t a, int64_t b) {
    while (b) {
        int64_t t = a % b;
        a = b;
        b = t;
    }
    return a;
}

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

extern "C" const char* ifa_status_string(ifa_status s) {
    switch (s) {
    case IFA_OK: return "success";
    case IFA_ERR_PARAM_NULLPTR: return "a required pointer is NULL (161001)";
    case IFA_ERR_PARAM_INVALID: return "a parameter is outside the supported range (161002)";
    case IFA_ERR_RUNTIME: return "a CUDA runtime call failed (361001)";
    default: return "unknown status";
    }
}

static bool valid_params(const ifa_params& p) {
    if (p.B < 0 || p.B > 65536) return false;
    if (p.numHeads < 1 || p.numHeads > 256) return false;
    const int64_t kvn = p.numKeyValueHeads == 0 ? p.numHeads : p.numKeyValueHeads;
    if (kvn < 1 || p.numHeads % kvn != 0) return false;
    if (p.headDim < 1 || p.headDim > 512) return false;
    if (p.q_dtype != IFA_F16 && p.q_dtype != IFA_BF16) return false;
    if (p.kv_dtype == IFA_I8) {
        if (p.antiquant != IFA_ANTIQUANT_PER_CHANNEL && p.antiquant != IFA_ANTIQUANT_PER_TENSOR) return false;
        if (p.headDim % 16 != 0) return false;
    } else {
        if (p.kv_dtype != p.q_dtype) return false;
        if (p.antiquant != IFA_ANTIQUANT_NONE) return false;
    }
    if (p.headDim % 8 != 0) return false;
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
    return true;
}

extern "C" ifa_status ifa_create(const ifa_params* params, ifa_plan** plan, size_t* workspace_bytes) {
    if (!params || !plan || !workspace_bytes) return IFA_ERR_PARAM_NULLPTR;
    *plan = nullptr;
    *workspace_bytes = 0;
    if (!valid_params(*params)) return IFA_ERR_PARAM_INVALID;
    const ifa_params& p = *params;

    ifa_plan* pl = new (std::nothrow) ifa_plan();
    if (!pl) return IFA_ERR_RUNTIME;
    pl->prm = p;
    pl->KV_N = (int)(p.numKeyValueHeads == 0 ? p.numHeads : p.numKeyValueHeads);
    pl->G = (int)(p.numHeads / pl->KV_N);
    pl->kv_kind = p.kv_dtype == IFA_I8 ? KV_I8 : (p.q_dtype == IFA_BF16 ? KV_BF16 : KV_F16);
    pl->es = p.kv_dtype == IFA_I8 ? 1 : 2;
    const int cg_elems = 128 / pl->es;
    pl->DPAD = (int)((p.headDim + cg_elems - 1) / cg_elems * cg_elems);
    if (pl->DPAD == 192) pl->DPAD = 256;
    if (pl->DPAD > 256) {  // head dims above 256 are outside this build's kernel set
        delete pl;
        return IFA_ERR_PARAM_INVALID;
    }
    const int max_nt = pl->DPAD >= 256 ? 1 : 2;
    const int gt_max = 8 * max_nt;
    pl->GT = std::min(pl->G, gt_max);
    pl->NT = (pl->GT + 7) / 8;
    pl->NGS = (pl->G + pl->GT - 1) / pl->GT;
    pl->launch = decode_launcher(pl->kv_kind, pl->DPAD, pl->NT);
    int smem = 0;
    if (!pl->launch || !cfg_lookup(pl->kv_kind, pl->DPAD, pl->NT, &pl->slot_floats, &smem)) {
        delete pl;
        return IFA_ERR_PARAM_INVALID;
    }
    pl->box_rows = kTileTokens;
    if (p.kvFormat != IFA_KV_CONTIG) pl->box_rows = (int)gcd64(kTileTokens, p.blockSize);

    if (cudaGetDevice(&pl->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&pl->num_sms, cudaDevAttrMultiProcessorCount, pl->device) != cudaSuccess) {
        cudaGetLastError();
        delete pl;
        return IFA_ERR_RUNTIME;
    }
    pl->P_max = std::max(1, std::min(kMaxCtas, pl->num_sms));
    pl->partial_bytes = align_up((size_t)2 * pl->P_max * pl->slot_floats * sizeof(float), 256);
    pl->ext_offset = pl->partial_bytes;
    pl->ws_bytes = pl->partial_bytes;
    if (p.B > kInlineB) pl->ws_bytes += align_up((size_t)(3 * p.B + 1) * sizeof(int32_t), 256);
    if (cudaMalloc(&pl->d_err, sizeof(int)) != cudaSuccess || cudaMemset(pl->d_err, 0, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        delete pl;
        return IFA_ERR_RUNTIME;
    }
    pl->dp = new (std::nothrow) DecodeParams();
    pl->cp = new (std::nothrow) CombineParams();
    if (!pl->dp || !pl->cp) {
        cudaFree(pl->d_err);
        delete pl->dp;
        delete pl->cp;
        delete pl;
        return IFA_ERR_RUNTIME;
    }
    pl->last_k = pl->last_v = nullptr;
    pl->last_launches = 0;
    *plan = pl;
    *workspace_bytes = pl->ws_bytes;
    return IFA_OK;
}

extern "C" int64_t ifa_last_launch_count(const ifa_plan* plan) { return plan ? plan->last_launches : 0; }

extern "C" ifa_status ifa_destroy(ifa_plan* plan) {
    if (!plan) return IFA_OK;
    cudaFree(plan->d_err);
    delete plan->dp;
    delete plan->cp;
    delete plan;
    return IFA_OK;
}

extern "C" ifa_status ifa_get_device_errors(ifa_plan* plan, void* stream, int64_t* flags) {
    if (!plan || !flags) return IFA_ERR_PARAM_NULLPTR;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int h = 0;
    if (cudaMemcpyAsync(&h, plan->d_err, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemsetAsync(plan->d_err, 0, sizeof(int), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return IFA_ERR_RUNTIME;
    }
    *flags = h;
    return IFA_OK;
}

static bool encode_map(const ifa_plan* pl, const void* base, CUtensorMap* map) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    const ifa_params& p = pl->prm;
    const uint64_t es = (uint64_t)pl->es;
    const uint64_t D = (uint64_t)p.headDim, KVN = (uint64_t)pl->KV_N;
    cuuint64_t dims[4], strides[3];
    const bool bnsd_like = (p.kvFormat == IFA_KV_PAGED_NBSD) ||
                           (p.kvFormat == IFA_KV_CONTIG && p.inputLayout == IFA_LAYOUT_BNSD);
    const uint64_t S = p.kvFormat == IFA_KV_CONTIG ? (uint64_t)p.maxSeqLen : (uint64_t)p.blockSize;
    const uint64_t outer = p.kvFormat == IFA_KV_CONTIG ? (uint64_t)p.B : (uint64_t)p.blockNum;
    dims[0] = D;
    dims[1] = S;
    dims[2] = KVN;
    dims[3] = outer;
    if (bnsd_like) {
        strides[0] = D * es;          // token
        strides[1] = S * D * es;      // kv head
        strides[2] = KVN * S * D * es;
    } else {
        strides[0] = KVN * D * es;
        strides[1] = D * es;
        strides[2] = S * KVN * D * es;
    }
    cuuint32_t box[4] = {(cuuint32_t)(128 / es), (cuuint32_t)pl->box_rows, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUtensorMapDataType dt = pl->kv_kind == KV_I8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                             : (pl->kv_kind == KV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                       : CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
    CUresult r = enc(map, dt, 4, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

static bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

extern "C" ifa_status ifa_run(ifa_plan* pl, const void* query, const void* key, const void* value,
                              const void* attenMask, const int64_t* actualSeqLengths,
                              const int64_t* kvPaddingSize, int64_t n_kv_padding, const int32_t* blockTable,
                              const void* antiquantScale, const void* antiquantOffset, void* attentionOut,
                              void* workspace, size_t workspace_bytes, void* stream) {
    if (!pl) return IFA_ERR_PARAM_NULLPTR;
    const ifa_params& p = pl->prm;
    const bool paged = p.kvFormat != IFA_KV_CONTIG;
    if (!query || !key || !value || !attentionOut) return IFA_ERR_PARAM_NULLPTR;
    if (p.has_mask && !attenMask) return IFA_ERR_PARAM_NULLPTR;
    if (paged && (!blockTable || !actualSeqLengths)) return IFA_ERR_PARAM_NULLPTR;
    if (p.antiquant != IFA_ANTIQUANT_NONE && (!antiquantScale || !antiquantOffset)) return IFA_ERR_PARAM_NULLPTR;
    if (p.has_kv_padding && !kvPaddingSize) return IFA_ERR_PARAM_NULLPTR;
    if (pl->ws_bytes > 0 && !workspace) return IFA_ERR_PARAM_NULLPTR;
    if (workspace_bytes < pl->ws_bytes) return IFA_ERR_PARAM_INVALID;
    if (!aligned(query, 16) || !aligned(key, 16) || !aligned(value, 16) || !aligned(attentionOut, 16) ||
        (workspace && !aligned(workspace, 16)))
        return IFA_ERR_PARAM_INVALID;
    if (blockTable && !aligned(blockTable, 4)) return IFA_ERR_PARAM_INVALID;
    if (p.antiquant != IFA_ANTIQUANT_NONE && (!aligned(antiquantScale, 2) || !aligned(antiquantOffset, 2)))
        return IFA_ERR_PARAM_INVALID;
    const bool left_pad = p.has_kv_padding && actualSeqLengths != nullptr;
    if (left_pad && n_kv_padding != 1 && n_kv_padding != p.B) return IFA_ERR_PARAM_INVALID;
    const int B = (int)p.B;
    pl->last_launches = 0;
    if (B == 0) return IFA_OK;

    // ---- per-batch windows (IncreFlashAttention README: actualSeqLengths, kv左padding)
    const int RS = pl->KV_N * pl->NGS;
    std::vector<int32_t>& bd = pl->bdata;
    bd.assign((size_t)3 * B + 1, 0);
    int64_t W = 0;
    int max_seq_tiles = 0;
    const int64_t cap = paged ? p.blockTableCols * p.blockSize : p.maxSeqLen;
    for (int b = 0; b < B; ++b) {
        int64_t len = actualSeqLengths ? actualSeqLengths[b] : p.maxSeqLen;
        int64_t st = 0;
        if (len < 0) return IFA_ERR_PARAM_INVALID;
        if (left_pad) {
            int64_t pad = kvPaddingSize[n_kv_padding == 1 ? 0 : b];
            if (pad < 0) pad = 0;
            st = p.maxSeqLen - pad - len;
            const int64_t en = p.maxSeqLen - pad;
            if (st < 0 || en < 0) {
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
        const int tiles = (int)((len + kTileTokens - 1) / kTileTokens);
        max_seq_tiles = std::max(max_seq_tiles, tiles);
        W += (int64_t)tiles * RS;
        if (W > INT32_MAX) return IFA_ERR_PARAM_INVALID;
    }
    bd[3 * B] = (int32_t)W;

    // ---- split plan: P CTAs with equal shares of the W tiles
    int64_t tpc;
    if (p.splitTiles > 0) {
        tpc = p.splitTiles;
    } else {
        tpc = (W + pl->P_max - 1) / pl->P_max;
        tpc = std::max<int64_t>(tpc, std::min(max_seq_tiles, 4));
        tpc = std::max<int64_t>(tpc, 1);
    }
    int P = W == 0 ? 1 : (int)std::min<int64_t>(pl->P_max, (W + tpc - 1) / tpc);

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    DecodeParams& dp = *pl->dp;
    if (key != pl->last_k) {
        if (!encode_map(pl, key, &dp.tmK)) return IFA_ERR_RUNTIME;
        pl->last_k = key;
    }
    if (value != pl->last_v) {
        if (!encode_map(pl, value, &dp.tmV)) return IFA_ERR_RUNTIME;
        pl->last_v = value;
    }
    dp.q = query;
    dp.out = attentionOut;
    dp.mask = reinterpret_cast<const uint8_t*>(attenMask);
    dp.block_table = blockTable;
    dp.aq_scale = antiquantScale;
    dp.aq_offset = antiquantOffset;
    dp.partials = reinterpret_cast<float*>(workspace);
    dp.err = pl->d_err;
    dp.W = W;
    dp.P = P;
    dp.B = B;
    dp.N = (int)p.numHeads;
    dp.KV_N = pl->KV_N;
    dp.D = (int)p.headDim;
    dp.G = pl->G;
    dp.GT = pl->GT;
    dp.NGS = pl->NGS;
    dp.q_bf16 = p.q_dtype == IFA_BF16;
    dp.paged = paged;
    dp.block_size = (int)p.blockSize;
    dp.bt_cols = (int)p.blockTableCols;
    dp.block_num = (int)p.blockNum;
    dp.box_rows = pl->box_rows;
    dp.has_mask = p.has_mask != 0;
    dp.mask_bstride = (p.has_mask && p.maskB > 1) ? p.maskN * p.maskS : 0;
    dp.mask_nstride = (p.has_mask && p.maskN > 1) ? p.maskS : 0;
    dp.aq_per_channel = p.antiquant == IFA_ANTIQUANT_PER_CHANNEL;
    dp.scale_log2 = (float)(p.scaleValue * 1.4426950408889634);
    dp.slot_floats = pl->slot_floats;
    if (B <= kInlineB) {
        std::memcpy(dp.bdata_inline, bd.data(), bd.size() * sizeof(int32_t));
        dp.ext_bdata = nullptr;
    } else {
        int32_t* ext = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(workspace) + pl->ext_offset);
        if (cudaMemcpyAsync(ext, bd.data(), bd.size() * sizeof(int32_t), cudaMemcpyHostToDevice, s) != cudaSuccess) {
            cudaGetLastError();
            return IFA_ERR_RUNTIME;
        }
        dp.ext_bdata = ext;
    }
    if (pl->launch(dp, P, s) != cudaSuccess) {
        cudaGetLastError();
        return IFA_ERR_RUNTIME;
    }
    pl->last_launches = 1;

    // ---- combine jobs: sequences cut by a CTA boundary
    CombineParams& cp = *pl->cp;
    cp.njobs = 0;
    int max_pieces = 1;
    auto seq_of = [&](int64_t tile, int64_t* first_tile) -> int64_t {
        int lo = 0, hi = B;
        while (hi - lo > 1) {
            int mid = (lo + hi) / 2;
            if (bd[2 * B + mid] <= tile) lo = mid;
            else hi = mid;
        }
        const int64_t tiles = (bd[B + lo] + kTileTokens - 1) / kTileTokens;
        const int64_t off = tile - bd[2 * B + lo];
        const int64_t r = off / tiles;
        *first_tile = bd[2 * B + lo] + r * tiles;
        return (int64_t)lo * RS + r;
    };
    for (int c = 0; c + 1 < P; ++c) {
        const int64_t bnd = (int64_t)(c + 1) * W / P;
        if (bnd <= 0 || bnd >= W) continue;
        int64_t f1, f2;
        const int64_t s1 = seq_of(bnd - 1, &f1);
        const int64_t s2 = seq_of(bnd, &f2);
        if (s1 != s2) continue;
        if (cp.njobs > 0 && cp.jobs[cp.njobs - 1].seq == (int)s1) {
            cp.jobs[cp.njobs - 1].c_last = c + 1;
        } else {
            CombineJob& j = cp.jobs[cp.njobs++];
            j.seq = (int)s1;
            j.c_first = c;
            j.c_last = c + 1;
            const int64_t lo_c = (int64_t)c * W / P;
            j.first_odd = f1 <= lo_c ? 0 : 1;
        }
        max_pieces = std::max(max_pieces, cp.jobs[cp.njobs - 1].c_last - cp.jobs[cp.njobs - 1].c_first + 1);
    }
    if (cp.njobs > 0) {
        cp.out = attentionOut;
        cp.partials = reinterpret_cast<const float*>(workspace);
        cp.aq_scale = antiquantScale;
        cp.aq_offset = antiquantOffset;
        cp.N = (int)p.numHeads;
        cp.D = (int)p.headDim;
        cp.G = pl->G;
        cp.GT = pl->GT;
        cp.NGS = pl->NGS;
        cp.KV_N = pl->KV_N;
        cp.q_bf16 = p.q_dtype == IFA_BF16;
        cp.kv_i8 = pl->kv_kind == KV_I8;
        cp.aq_per_channel = p.antiquant == IFA_ANTIQUANT_PER_CHANNEL;
        cp.slot_floats = pl->slot_floats;
        cp.d_pad = pl->DPAD;
        cp.gt_pad = 8 * pl->NT;
        if (launch_combine(cp, max_pieces, s) != cudaSuccess) {
            cudaGetLastError();
            return IFA_ERR_RUNTIME;
        }
        pl->last_launches = 2;
    }
    return IFA_OK;
}

// Shared with the fixed-scratch entry point (ifa_noalloc.cu).
namespace ifa {
bool params_are_valid(const ifa_params& p) { return valid_params(p); }
bool decode_cfg(int kv, int dpad, int nt, int* slot_floats, int* smem) {
    return cfg_lookup(kv, dpad, nt, slot_floats, smem);
}
void* tensor_map_encoder() { return reinterpret_cast<void*>(get_encode_fn()); }
}  // namespace ifa
