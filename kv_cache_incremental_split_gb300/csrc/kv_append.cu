// KV-cache append (ifa_kv_append): the key and value rows of one new token per batch are
// written at that batch's position in the cache, in the cache's own layout, as the
// incremental decode step grows the cache (IncreFlashAttention README, incremental
// inference).  int8 caches receive codes that the antiquant reading (code + offset) * scale
// maps back to the new values.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "../../include/ifa.h"
#include "decode.cuh"

namespace ifa {
namespace {

struct AppendArgs {
    const uint16_t* k_new;
    const uint16_t* v_new;
    const int64_t* pos;
    const int32_t* block_table;
    const uint16_t* aq_scale;
    const uint16_t* aq_offset;
    void* k_cache;
    void* v_cache;
    int* err;
    int KV_N, D, chunks;  // chunks: 8-element groups of one token row (KV_N * D / 8)
    int layout, kv_format;
    long long Smax;
    int block_size, bt_cols, block_num;
    int bf16, int8_cache, per_channel;
};

__device__ __forceinline__ float half_bits(uint16_t u, int bf16) {
    return bf16 ? __bfloat162float(__ushort_as_bfloat16(u)) : __half2float(__ushort_as_half(u));
}

// Code of x read back as (code + offset) * scale: rint(x / scale - offset) in single precision
// (ties to even), saturated to [-128, 127]; NaN gives 0.
__device__ __forceinline__ int quantize(float x, float scale, float offset) {
    const float u = __fsub_rn(__fdiv_rn(x, scale), offset);
    if (u != u) return 0;
    const float r = fminf(fmaxf(rintf(u), -128.f), 127.f);
    return (int)r;
}

// One CTA per batch; thread i moves 8-element groups i, i + blockDim, ... of the key row then
// the value row.  Element (h, d) of batch b's new token sits at (b * KV_N + h) * D + d.
__global__ void __launch_bounds__(256) kv_append_kernel(const AppendArgs a) {
    const int b = blockIdx.x;
    const long long t = __ldg(a.pos + b);
    long long blk = 0;
    bool ok = t >= 0;
    if (a.kv_format == IFA_KV_CONTIG) {
        ok = ok && t < a.Smax;
    } else {
        ok = ok && t / a.block_size < a.bt_cols;
        if (ok) {
            blk = __ldg(a.block_table + (long long)b * a.bt_cols + t / a.block_size);
            ok = blk >= 0 && blk < a.block_num;
        }
    }
    if (!ok) {
        if (threadIdx.x == 0 && a.err) atomicOr(a.err, kErrBadBlock);
        return;
    }
    const long long slot = a.kv_format == IFA_KV_CONTIG ? 0 : t % a.block_size;
    for (int w = threadIdx.x; w < 2 * a.chunks; w += blockDim.x) {
        const int which = w >= a.chunks;  // 0 key, 1 value
        const int c = w - which * a.chunks;
        const int e0 = c * 8;              // first element of the group within the token row
        const int h = e0 / a.D, d = e0 - h * a.D;
        long long dst;
        if (a.kv_format == IFA_KV_CONTIG) {
            if (a.layout == IFA_LAYOUT_BNSD) dst = (((long long)b * a.KV_N + h) * a.Smax + t) * a.D + d;
            else dst = (((long long)b * a.Smax + t) * a.KV_N + h) * a.D + d;  // BSND and BSH
        } else if (a.kv_format == IFA_KV_PAGED_NBSD) {
            dst = ((blk * a.KV_N + h) * a.block_size + slot) * a.D + d;
        } else {
            dst = ((blk * a.block_size + slot) * a.KV_N + h) * a.D + d;  // (blocknum, blockSize, H)
        }
        const uint16_t* src = (which ? a.v_new : a.k_new) + ((long long)b * a.KV_N * a.D + e0);
        const uint4 raw = *reinterpret_cast<const uint4*>(src);
        void* cache = which ? a.v_cache : a.k_cache;
        if (!a.int8_cache) {
            *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(cache) + dst) = raw;
            continue;
        }
        const uint16_t* x = reinterpret_cast<const uint16_t*>(&raw);
        uint32_t packed[2] = {0u, 0u};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const long long pi = a.per_channel ? ((long long)which * a.KV_N + h) * a.D + d + j : which;
            const float s = half_bits(__ldg(a.aq_scale + pi), a.bf16);
            const float o = half_bits(__ldg(a.aq_offset + pi), a.bf16);
            const int q = quantize(half_bits(x[j], a.bf16), s, o);
            packed[j >> 2] |= (uint32_t)(q & 0xff) << (8 * (j & 3));
        }
        *reinterpret_cast<uint2*>(reinterpret_cast<int8_t*>(cache) + dst) = make_uint2(packed[0], packed[1]);
    }
}

bool aligned(const void* p, uintptr_t a) { return p && (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool append_valid(const ifa_append_params& p) {
    if (p.B < 0 || p.B > (1 << 20)) return false;
    if (p.numKeyValueHeads < 1 || p.numKeyValueHeads > 256) return false;
    if (p.new_dtype != IFA_F16 && p.new_dtype != IFA_BF16) return false;
    const bool i8 = p.kv_dtype == IFA_I8;
    if (!i8 && p.kv_dtype != p.new_dtype) return false;
    if (i8 != (p.antiquant != IFA_ANTIQUANT_NONE)) return false;
    if (p.antiquant < IFA_ANTIQUANT_NONE || p.antiquant > IFA_ANTIQUANT_PER_TENSOR) return false;
    if (p.headDim < 8 || p.headDim > 512 || p.headDim % (i8 ? 16 : 8) != 0) return false;
    if (p.kvFormat == IFA_KV_CONTIG) {
        if (p.inputLayout < IFA_LAYOUT_BSH || p.inputLayout > IFA_LAYOUT_BNSD) return false;
        if (p.maxSeqLen < 1) return false;
    } else if (p.kvFormat == IFA_KV_PAGED_NBSD || p.kvFormat == IFA_KV_PAGED_BSH) {
        if (p.blockSize < 1 || p.blockSize > 1024 || p.blockNum < 1 || p.blockTableCols < 1) return false;
        if (p.blockTableCols > INT32_MAX / 2 || p.blockNum > INT32_MAX) return false;
    } else {
        return false;
    }
    return true;
}

}  // namespace
}  // namespace ifa

using namespace ifa;

extern "C" ifa_status ifa_kv_append(const ifa_append_params* params, const void* keyNew, const void* valueNew,
                                    const int64_t* positions, const int32_t* blockTable, const void* antiquantScale,
                                    const void* antiquantOffset, void* keyCache, void* valueCache,
                                    int32_t* deviceErrorFlags, void* stream) {
    if (!params) return IFA_ERR_PARAM_NULLPTR;
    const ifa_append_params& p = *params;
    if (!append_valid(p)) return IFA_ERR_PARAM_INVALID;
    const bool paged = p.kvFormat != IFA_KV_CONTIG;
    const bool i8 = p.kv_dtype == IFA_I8;
    if (!keyNew || !valueNew || !positions || !keyCache || !valueCache) return IFA_ERR_PARAM_NULLPTR;
    if (paged && !blockTable) return IFA_ERR_PARAM_NULLPTR;
    if (i8 && (!antiquantScale || !antiquantOffset)) return IFA_ERR_PARAM_NULLPTR;
    if (!aligned(keyNew, 16) || !aligned(valueNew, 16) || !aligned(keyCache, 16) || !aligned(valueCache, 16) ||
        !aligned(positions, 8) || (paged && !aligned(blockTable, 4)) ||
        (i8 && (!aligned(antiquantScale, 2) || !aligned(antiquantOffset, 2))) ||
        (deviceErrorFlags && !aligned(deviceErrorFlags, 4)))
        return IFA_ERR_PARAM_INVALID;
    if (p.B == 0) return IFA_OK;
    AppendArgs a;
    std::memset(&a, 0, sizeof(a));
    a.k_new = static_cast<const uint16_t*>(keyNew);
    a.v_new = static_cast<const uint16_t*>(valueNew);
    a.pos = positions;
    a.block_table = blockTable;
    a.aq_scale = static_cast<const uint16_t*>(antiquantScale);
    a.aq_offset = static_cast<const uint16_t*>(antiquantOffset);
    a.k_cache = keyCache;
    a.v_cache = valueCache;
    a.err = deviceErrorFlags;
    a.KV_N = (int)p.numKeyValueHeads;
    a.D = (int)p.headDim;
    a.chunks = a.KV_N * a.D / 8;
    a.layout = p.inputLayout;
    a.kv_format = p.kvFormat;
    a.Smax = paged ? 0 : p.maxSeqLen;
    a.block_size = paged ? (int)p.blockSize : 1;
    a.bt_cols = paged ? (int)p.blockTableCols : 0;
    a.block_num = paged ? (int)p.blockNum : 0;
    a.bf16 = p.new_dtype == IFA_BF16;
    a.int8_cache = i8;
    a.per_channel = p.antiquant == IFA_ANTIQUANT_PER_CHANNEL;
    kv_append_kernel<<<(unsigned)p.B, 256, 0, static_cast<cudaStream_t>(stream)>>>(a);
    if (cudaGetLastError() != cudaSuccess) return IFA_ERR_RUNTIME;
    return IFA_OK;
}
