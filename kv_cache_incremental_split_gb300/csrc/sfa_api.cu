// C ABI of the sparse MLA-absorb decode (sfa_workspace_size, sfa_run).  The
// checks follow the "SparseFlashAttention" README's 参数说明 and 约束说明 for
// the decode case this library implements (BSND or TND queries, PA_BSND, BSND
// or TND key/value, KV_N = 1, D = 512, Dr = 64, token-wise or block-wise
// sparsity, sparse_mode 0 or 3, MLA-absorb, optional softmax_max/softmax_sum).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "../../include/ifa.h"
#include "decode.cuh"
#include "sfa.cuh"

using namespace ifa;

static_assert(kSfaStartOffset + sizeof(SfaStart) * kMaxCtas <= kSfaPartialOffset, "workspace layout");

namespace {

bool sfa_valid(const sfa_params& p) {
    if (p.B < 0 || p.B > 65536) return false;
    if (p.layout_query == SFA_LAYOUT_BSND) {
        if (p.Q_S < 1 || p.Q_S > 1024 || p.B * p.Q_S > (1 << 20)) return false;
    } else if (p.layout_query == SFA_LAYOUT_TND) {
        if (p.Q_T < 0 || p.Q_T > (1 << 20) || (p.B < 1 && p.Q_T > 0)) return false;
    } else {
        return false;
    }
    if (p.Q_N < 1 || p.Q_N > 128) return false;
    if (p.KV_N != 1 || p.D != kSfaD || p.Dr != kSfaDr) return false;
    if (p.sparse_size < 1 || p.sparse_size > INT32_MAX / 2) return false;
    // token-wise (1) or block-wise: a power of two up to 128 (that divides block_size when paged)
    if (p.sparse_block_size < 1 || p.sparse_block_size > 128 || (p.sparse_block_size & (p.sparse_block_size - 1)) != 0)
        return false;
    if (p.layout_kv == SFA_KV_PA_BSND) {
        if (p.block_size < 16 || p.block_size > 1024 || p.block_size % 16 != 0) return false;
        if (p.block_num < 1 || p.block_table_cols < 1) return false;
        if (p.block_num * p.block_size >= INT32_MAX) return false;
        if (p.block_table_cols > INT32_MAX / 2) return false;
        if (p.block_size % p.sparse_block_size != 0) return false;
    } else if (p.layout_kv == SFA_KV_BSND) {
        if (p.KV_S < 1 || p.KV_S >= INT32_MAX || p.B * p.KV_S >= INT32_MAX) return false;
    } else if (p.layout_kv == SFA_KV_TND) {
        if (p.KV_S < 1 || p.KV_S >= INT32_MAX) return false;
    } else {
        return false;
    }
    if (p.sparse_size * p.sparse_block_size > INT32_MAX / 2) return false;
    if (p.sparse_mode != 0 && p.sparse_mode != 3) return false;
    if (p.dtype != IFA_BF16 && p.dtype != IFA_F16) return false;
    if (!std::isfinite(p.scale_value)) return false;
    return true;
}

int sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return sms;
}

bool aligned(const void* p, uintptr_t a) { return p && (reinterpret_cast<uintptr_t>(p) % a) == 0; }

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
    static EncodeTiledFn fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return (EncodeTiledFn) nullptr;
        }
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

bool encode(CUtensorMap* map, bool bf16, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
            const cuuint32_t* box) {
    EncodeTiledFn enc = encoder();
    if (!enc) return false;
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, rank,
               const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" ifa_status sfa_workspace_size(const sfa_params* params, size_t* workspace_bytes) {
    if (!params || !workspace_bytes) return IFA_ERR_PARAM_NULLPTR;
    *workspace_bytes = 0;
    if (!sfa_valid(*params)) return IFA_ERR_PARAM_INVALID;
    const int sms = sm_count();
    if (sms <= 0) return IFA_ERR_RUNTIME;
    const int P_max = std::min(kMaxCtas, sms);
    const int64_t R = params->layout_query == SFA_LAYOUT_TND ? params->Q_T : params->B * params->Q_S;
    *workspace_bytes = kSfaPartialOffset + (size_t)2 * P_max * kSfaSlotFloats * sizeof(float) +
                       ((size_t)(2 * R + 1) * sizeof(int) + 15) / 16 * 16 + (size_t)R * sizeof(SfaPieces);
    return IFA_OK;
}

extern "C" ifa_status sfa_run(const sfa_params* params, const void* query, const void* query_rope, const void* key,
                              const void* key_rope, const void* value, const int32_t* sparse_indices,
                              const int32_t* block_table, const int32_t* actual_seq_lengths_kv,
                              const int32_t* actual_seq_lengths_query, void* attention_out, float* softmax_max,
                              float* softmax_sum, void* workspace, size_t workspace_bytes, int32_t* deviceErrorFlags,
                              void* stream) {
    if (!params) return IFA_ERR_PARAM_NULLPTR;
    const sfa_params& p = *params;
    if (!sfa_valid(p)) return IFA_ERR_PARAM_INVALID;
    const bool paged = p.layout_kv == SFA_KV_PA_BSND;
    if (!query || !query_rope || !key || !key_rope || !value || !sparse_indices || !attention_out || !workspace)
        return IFA_ERR_PARAM_NULLPTR;
    if (paged && !block_table) return IFA_ERR_PARAM_NULLPTR;
    if (p.layout_kv != SFA_KV_BSND && !actual_seq_lengths_kv) return IFA_ERR_PARAM_NULLPTR;
    if (p.layout_query == SFA_LAYOUT_TND && !actual_seq_lengths_query) return IFA_ERR_PARAM_NULLPTR;
    if ((softmax_max == nullptr) != (softmax_sum == nullptr)) return IFA_ERR_PARAM_NULLPTR;
    if (!aligned(query, 16) || !aligned(query_rope, 16) || !aligned(key, 16) || !aligned(key_rope, 16) ||
        !aligned(value, 16) || !aligned(attention_out, 16) || !aligned(workspace, 16) || !aligned(sparse_indices, 4))
        return IFA_ERR_PARAM_INVALID;
    if ((paged && !aligned(block_table, 4)) || (actual_seq_lengths_kv && !aligned(actual_seq_lengths_kv, 4)) ||
        (actual_seq_lengths_query && !aligned(actual_seq_lengths_query, 4)) ||
        (softmax_max && (!aligned(softmax_max, 4) || !aligned(softmax_sum, 4))))
        return IFA_ERR_PARAM_INVALID;
    if (deviceErrorFlags && !aligned(deviceErrorFlags, 4)) return IFA_ERR_PARAM_INVALID;
    size_t need = 0;
    const ifa_status st = sfa_workspace_size(&p, &need);
    if (st != IFA_OK) return st;
    if (workspace_bytes < need) return IFA_ERR_PARAM_INVALID;
    const int64_t R = p.layout_query == SFA_LAYOUT_TND ? p.Q_T : p.B * p.Q_S;  // query rows, each its own problem
    if (p.B == 0 || R == 0) return IFA_OK;

    const int sms = sm_count();
    const int P_max = std::min(kMaxCtas, sms);
    SfaParams sp;
    std::memset(&sp, 0, sizeof(sp));
    const bool bf = p.dtype == IFA_BF16;
    const uint64_t es = 2;
    const uint64_t rows = (uint64_t)(paged ? p.block_num * p.block_size
                                           : (p.layout_kv == SFA_KV_BSND ? p.B * p.KV_S : p.KV_S));
    {
        cuuint64_t dq[3] = {(cuuint64_t)kSfaD, (cuuint64_t)p.Q_N, (cuuint64_t)R};
        cuuint64_t sq[2] = {kSfaD * es, (cuuint64_t)p.Q_N * kSfaD * es};
        cuuint32_t bq[3] = {64, 128, 1};
        cuuint64_t dr[3] = {(cuuint64_t)kSfaDr, (cuuint64_t)p.Q_N, (cuuint64_t)R};
        cuuint64_t sr[2] = {kSfaDr * es, (cuuint64_t)p.Q_N * kSfaDr * es};
        cuuint64_t dk[2] = {(cuuint64_t)kSfaD, rows};
        cuuint64_t sk[1] = {kSfaD * es};
        cuuint64_t dkr[2] = {(cuuint64_t)kSfaDr, rows};
        cuuint64_t skr[1] = {kSfaDr * es};
        cuuint32_t bg[2] = {64, 1};
        if (!encode(&sp.tmQ, bf, query, 3, dq, sq, bq) || !encode(&sp.tmQr, bf, query_rope, 3, dr, sr, bq) ||
            !encode(&sp.tmK, bf, key, 2, dk, sk, bg) || !encode(&sp.tmKr, bf, key_rope, 2, dkr, skr, bg) ||
            !encode(&sp.tmV, bf, value, 2, dk, sk, bg))
            return IFA_ERR_RUNTIME;
        if (p.sparse_block_size >= 8) {
            // a selected block is sparse_block_size consecutive rows of one cache block
            cuuint32_t bb[2] = {64, (cuuint32_t)std::min<int64_t>(p.sparse_block_size, kSfaTile)};
            if (!encode(&sp.tmKb, bf, key, 2, dk, sk, bb) || !encode(&sp.tmKrb, bf, key_rope, 2, dkr, skr, bb) ||
                !encode(&sp.tmVb, bf, value, 2, dk, sk, bb))
                return IFA_ERR_RUNTIME;
        }
    }
    const int tps = (int)((p.sparse_size * p.sparse_block_size + kSfaTile - 1) / kSfaTile);
    // tiles of the query rows (each runs once per value half, on the two CTAs of a pair)
    const long long W = (long long)R * tps;
    if (W > INT32_MAX) return IFA_ERR_PARAM_INVALID;
    // pairs: as many as fit at once, with contiguous shares of at least min(tiles per row, kSfaMinShareTiles) tiles
    const int fit = std::min(P_max / 2, sfa_max_pairs());
    if (fit < 1) return IFA_ERR_RUNTIME;
    const long long min_share = std::max(1, std::min(tps, kSfaMinShareTiles));
    const int P = 2 * (int)std::max<long long>(1, std::min<long long>(fit, (W + min_share - 1) / min_share));

    unsigned char* ws = static_cast<unsigned char*>(workspace);
    sp.indices = sparse_indices;
    sp.block_table = block_table;
    sp.lens = actual_seq_lengths_kv;
    sp.lens_q = actual_seq_lengths_query;
    sp.lse_max = softmax_max;
    sp.lse_sum = softmax_sum;
    sp.B = (int)p.B;
    sp.q_tnd = p.layout_query == SFA_LAYOUT_TND;
    sp.kv_layout = p.layout_kv;
    sp.kv_s = paged ? 0 : (int)p.KV_S;
    sp.out = attention_out;
    sp.partials = reinterpret_cast<float*>(ws + kSfaPartialOffset);
    sp.starts = reinterpret_cast<SfaStart*>(ws + kSfaStartOffset);
    sp.eff = reinterpret_cast<int*>(ws + kSfaPartialOffset + (size_t)2 * P_max * kSfaSlotFloats * sizeof(float));
    sp.pre = sp.eff + R;
    sp.pieces = reinterpret_cast<SfaPieces*>(reinterpret_cast<unsigned char*>(sp.eff) +
                                             ((size_t)(2 * R + 1) * sizeof(int) + 15) / 16 * 16);
    sp.err = deviceErrorFlags ? deviceErrorFlags : reinterpret_cast<int*>(ws);
    sp.W = W;
    sp.P = P;
    sp.R = (int)R;
    sp.QS = p.layout_query == SFA_LAYOUT_TND ? 1 : (int)p.Q_S;
    sp.causal = p.sparse_mode == 3;
    sp.QN = (int)p.Q_N;
    sp.S_sp = (int)p.sparse_size;
    sp.sbs_log2 = 0;
    while ((1LL << sp.sbs_log2) < p.sparse_block_size) ++sp.sbs_log2;
    sp.tiles_per_seq = tps;
    sp.block_size = paged ? (int)p.block_size : 1;
    sp.bt_cols = paged ? (int)p.block_table_cols : 0;
    sp.block_num = paged ? (int)p.block_num : 0;
    sp.total_rows = (int)rows;
    sp.is_bf16 = bf;
    sp.scale_log2 = (float)(p.scale_value * 1.4426950408889634);
    if (launch_sfa(sp, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return IFA_ERR_RUNTIME;
    }
    return IFA_OK;
}
