// ifa_run_noalloc: the decode-attention call for callers that cannot allocate
// device memory.  Some callers cannot call cudaMalloc at all: code running
// inside a memory pool or allocator they do not own, runtimes that forbid
// allocation on their inference path, or code that must not grow the device
// footprint after start-up.  This entry point needs no plan, no workspace and
// no allocation: the split-KV partials live in one file-scope device array of
// fixed size, shared by every call in the process.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/ifa.h"
#include "decode.cuh"

namespace ifa {
bool params_are_valid(const ifa_params& p);
bool decode_cfg(int kv, int dpad, int nt, int* slot_floats, int* smem);
void* tensor_map_encoder();
}  // namespace ifa

using namespace ifa;

namespace {

constexpr size_t kScratchBytes = IFA_NOALLOC_SCRATCH_BYTES;
constexpr size_t kErrWordBytes = 256;               // first 256 bytes: device error word
constexpr int kMaxDevices = 64;

// The scratch every ifa_run_noalloc call on a device shares.  In host code this
// name is only a stand-in; the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Device address of the scratch array on the current device, looked up once per
// device (the first call on a device does this set-up).
unsigned char* scratch_on_current_device(int device) {
    static std::mutex mu;
    static unsigned char* addr[kMaxDevices] = {};
    if (device < 0 || device >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[device]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        addr[device] = static_cast<unsigned char*>(p);
    }
    return addr[device];
}

int64_t gcd(int64_t a, int64_t b) {
    while (b) {
        const int64_t t = a % b;
        a = b;
        b = t;
    }
    return a;
}

bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool encode(const ifa_params& p, int kvn, int es, int box_rows, int kv_kind, const void* base, CUtensorMap* map) {
    EncodeTiledFn enc = reinterpret_cast<EncodeTiledFn>(tensor_map_encoder());
    if (!enc) return false;
    const uint64_t E = (uint64_t)es, D = (uint64_t)p.headDim, KVN = (uint64_t)kvn;
    const bool contig = p.kvFormat == IFA_KV_CONTIG;
    const bool bnsd_like = p.kvFormat == IFA_KV_PAGED_NBSD || (contig && p.inputLayout == IFA_LAYOUT_BNSD);
    const uint64_t S = contig ? (uint64_t)p.maxSeqLen : (uint64_t)p.blockSize;
    cuuint64_t dims[4] = {D, S, KVN, contig ? (uint64_t)p.B : (uint64_t)p.blockNum};
    cuuint64_t strides[3];
    if (bnsd_like) {
        strides[0] = D * E;
        strides[1] = S * D * E;
        strides[2] = KVN * S * D * E;
    } else {
        strides[0] = KVN * D * E;
        strides[1] = D * E;
        strides[2] = S * KVN * D * E;
    }
    cuuint32_t box[4] = {(cuuint32_t)(128 / es), (cuuint32_t)box_rows, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUtensorMapDataType dt = kv_kind == KV_I8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : (kv_kind == KV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                         : CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
    return enc(map, dt, 4, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" ifa_status ifa_run_noalloc(const ifa_params* params, const void* query, const void* key,
                                      const void* value, const void* attenMask, const int64_t* actualSeqLengths,
                                      const int64_t* kvPaddingSize, int64_t n_kv_padding,
                                      const int32_t* blockTable, const void* antiquantScale,
                                      const void* antiquantOffset, void* attentionOut, int32_t* deviceErrorFlags,
                                      void* stream) {
    if (!params) return IFA_ERR_PARAM_NULLPTR;
    const ifa_params& p = *params;
    if (!params_are_valid(p)) return IFA_ERR_PARAM_INVALID;
    if (p.B > IFA_NOALLOC_MAX_BATCH) return IFA_ERR_PARAM_INVALID;  // windows must fit the launch parameters
    const bool paged = p.kvFormat != IFA_KV_CONTIG;
    if (!query || !key || !value || !attentionOut) return IFA_ERR_PARAM_NULLPTR;
    if (p.has_mask && !attenMask) return IFA_ERR_PARAM_NULLPTR;
    if (paged && (!blockTable || !actualSeqLengths)) return IFA_ERR_PARAM_NULLPTR;
    if (p.antiquant != IFA_ANTIQUANT_NONE && (!antiquantScale || !antiquantOffset)) return IFA_ERR_PARAM_NULLPTR;
    if (p.has_kv_padding && !kvPaddingSize) return IFA_ERR_PARAM_NULLPTR;
    if (!aligned_to(query, 16) || !aligned_to(key, 16) || !aligned_to(value, 16) || !aligned_to(attentionOut, 16))
        return IFA_ERR_PARAM_INVALID;
    if (blockTable && !aligned_to(blockTable, 4)) return IFA_ERR_PARAM_INVALID;
    if (deviceErrorFlags && !aligned_to(deviceErrorFlags, 4)) return IFA_ERR_PARAM_INVALID;
    if (p.antiquant != IFA_ANTIQUANT_NONE && (!aligned_to(antiquantScale, 2) || !aligned_to(antiquantOffset, 2)))
        return IFA_ERR_PARAM_INVALID;
    const bool left_pad = p.has_kv_padding && actualSeqLengths != nullptr;
    if (left_pad && n_kv_padding != 1 && n_kv_padding != p.B) return IFA_ERR_PARAM_INVALID;

    // ---- kernel configuration (same rules as ifa_create)
    const int KV_N = (int)(p.numKeyValueHeads == 0 ? p.numHeads : p.numKeyValueHeads);
    const int G = (int)(p.numHeads / KV_N);
    const int kv_kind = p.kv_dtype == IFA_I8 ? KV_I8 : (p.q_dtype == IFA_BF16 ? KV_BF16 : KV_F16);
    const int es = p.kv_dtype == IFA_I8 ? 1 : 2;
    const int cg = 128 / es;
    int dpad = (int)((p.headDim + cg - 1) / cg * cg);
    if (dpad == 192) dpad = 256;
    if (dpad > 256) return IFA_ERR_PARAM_INVALID;
    const int GT = std::min(G, dpad >= 256 ? 8 : 16);
    const int NT = (GT + 7) / 8;
    const int NGS = (G + GT - 1) / GT;
    int slot_floats = 0, smem = 0;
    DecodeLaunchFn launch = decode_launcher(kv_kind, dpad, NT);
    if (!launch || !decode_cfg(kv_kind, dpad, NT, &slot_floats, &smem)) return IFA_ERR_PARAM_INVALID;
    const int box_rows = paged ? (int)gcd(kTileTokens, p.blockSize) : kTileTokens;

    const int B = (int)p.B;
    if (B == 0) return IFA_OK;

    int device = 0, sms = 0;
    if (cudaGetDevice(&device) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
        cudaGetLastError();
        return IFA_ERR_RUNTIME;
    }
    unsigned char* scratch = scratch_on_current_device(device);
    if (!scratch) return IFA_ERR_RUNTIME;
    // The partial slots (2 per CTA) must fit the fixed scratch: cap the grid accordingly.
    const size_t slot_bytes = (size_t)slot_floats * sizeof(float);
    const int p_fit = (int)std::min<size_t>(kMaxCtas, (kScratchBytes - kErrWordBytes) / (2 * slot_bytes));
    if (p_fit < 1) return IFA_ERR_PARAM_INVALID;
    const int P_max = std::max(1, std::min({kMaxCtas, sms, p_fit}));

    // ---- per-batch windows, in the launch parameters
    static_assert(IFA_NOALLOC_MAX_BATCH <= kInlineB, "windows travel inline");
    DecodeParams dp;
    std::memset(&dp, 0, sizeof(dp));
    int* bd = dp.bdata_inline;
    const int RS = KV_N * NGS;
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
            if (st < 0 || p.maxSeqLen - pad < 0) {
                st = 0;
                len = 0;
            }
        } else if (len > cap) {
            return IFA_ERR_PARAM_INVALID;
        }
        if (p.has_mask && len > 0 && st + len > p.maskS) return IFA_ERR_PARAM_INVALID;
        bd[b] = (int)st;
        bd[B + b] = (int)len;
        bd[2 * B + b] = (int)W;
        const int tiles = (int)((len + kTileTokens - 1) / kTileTokens);
        max_seq_tiles = std::max(max_seq_tiles, tiles);
        W += (int64_t)tiles * RS;
        if (W > INT32_MAX) return IFA_ERR_PARAM_INVALID;
    }
    bd[3 * B] = (int)W;

    int64_t tpc = p.splitTiles > 0 ? p.splitTiles
                                   : std::max<int64_t>({(W + P_max - 1) / P_max,
                                                        (int64_t)std::min(max_seq_tiles, 4), (int64_t)1});
    const int P = W == 0 ? 1 : (int)std::min<int64_t>(P_max, (W + tpc - 1) / tpc);

    if (!encode(p, KV_N, es, box_rows, kv_kind, key, &dp.tmK) ||
        !encode(p, KV_N, es, box_rows, kv_kind, value, &dp.tmV))
        return IFA_ERR_RUNTIME;
    float* partials = reinterpret_cast<float*>(scratch + kErrWordBytes);
    dp.q = query;
    dp.out = attentionOut;
    dp.mask = reinterpret_cast<const uint8_t*>(attenMask);
    dp.block_table = blockTable;
    dp.aq_scale = antiquantScale;
    dp.aq_offset = antiquantOffset;
    dp.partials = partials;
    dp.err = deviceErrorFlags ? deviceErrorFlags : reinterpret_cast<int*>(scratch);
    dp.ext_bdata = nullptr;
    dp.W = W;
    dp.P = P;
    dp.B = B;
    dp.N = (int)p.numHeads;
    dp.KV_N = KV_N;
    dp.D = (int)p.headDim;
    dp.G = G;
    dp.GT = GT;
    dp.NGS = NGS;
    dp.q_bf16 = p.q_dtype == IFA_BF16;
    dp.paged = paged;
    dp.block_size = (int)p.blockSize;
    dp.bt_cols = (int)p.blockTableCols;
    dp.block_num = (int)p.blockNum;
    dp.box_rows = box_rows;
    dp.has_mask = p.has_mask != 0;
    dp.mask_bstride = (p.has_mask && p.maskB > 1) ? p.maskN * p.maskS : 0;
    dp.mask_nstride = (p.has_mask && p.maskN > 1) ? p.maskS : 0;
    dp.aq_per_channel = p.antiquant == IFA_ANTIQUANT_PER_CHANNEL;
    dp.scale_log2 = (float)(p.scaleValue * 1.4426950408889634);
    dp.slot_floats = slot_floats;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (launch(dp, P, s) != cudaSuccess) {
        cudaGetLastError();
        return IFA_ERR_RUNTIME;
    }

    // ---- sequences cut by a CTA boundary are merged by the combine kernel
    CombineParams cp;
    std::memset(&cp, 0, sizeof(cp));
    int max_pieces = 1;
    auto seq_at = [&](int64_t tile, int64_t* first_tile) -> int64_t {
        int lo = 0, hi = B;
        while (hi - lo > 1) {
            const int mid = (lo + hi) / 2;
            if (bd[2 * B + mid] <= tile) lo = mid;
            else hi = mid;
        }
        const int64_t tiles = (bd[B + lo] + kTileTokens - 1) / kTileTokens;
        const int64_t r = (tile - bd[2 * B + lo]) / tiles;
        *first_tile = bd[2 * B + lo] + r * tiles;
        return (int64_t)lo * RS + r;
    };
    for (int c = 0; c + 1 < P; ++c) {
        const int64_t bnd = (int64_t)(c + 1) * W / P;
        if (bnd <= 0 || bnd >= W) continue;
        int64_t f1, f2;
        const int64_t s1 = seq_at(bnd - 1, &f1);
        if (s1 != seq_at(bnd, &f2)) continue;
        if (cp.njobs > 0 && cp.jobs[cp.njobs - 1].seq == (int)s1) {
            cp.jobs[cp.njobs - 1].c_last = c + 1;
        } else {
            CombineJob& j = cp.jobs[cp.njobs++];
            j.seq = (int)s1;
            j.c_first = c;
            j.c_last = c + 1;
            j.first_odd = f1 <= (int64_t)c * W / P ? 0 : 1;
        }
        max_pieces = std::max(max_pieces, cp.jobs[cp.njobs - 1].c_last - cp.jobs[cp.njobs - 1].c_first + 1);
    }
    if (cp.njobs > 0) {
        cp.out = attentionOut;
        cp.partials = partials;
        cp.aq_scale = antiquantScale;
        cp.aq_offset = antiquantOffset;
        cp.N = (int)p.numHeads;
        cp.D = (int)p.headDim;
        cp.G = G;
        cp.GT = GT;
        cp.NGS = NGS;
        cp.KV_N = KV_N;
        cp.q_bf16 = p.q_dtype == IFA_BF16;
        cp.kv_i8 = kv_kind == KV_I8;
        cp.aq_per_channel = p.antiquant == IFA_ANTIQUANT_PER_CHANNEL;
        cp.slot_floats = slot_floats;
        cp.d_pad = dpad;
        cp.gt_pad = 8 * NT;
        if (launch_combine(cp, max_pieces, s) != cudaSuccess) {
            cudaGetLastError();
            return IFA_ERR_RUNTIME;
        }
    }
    return IFA_OK;
}
