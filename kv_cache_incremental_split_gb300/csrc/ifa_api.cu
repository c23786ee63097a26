// C ABI of the decode-attention library: the two-phase plan/run API of the
// "aclnnIncreFlashAttentionV2" page (Function Prototype, Return Value),
// built on the shared host planner (plan.cu) and the split-KV decode kernel.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "../../include/ifa.h"
#include "decode.cuh"

using namespace ifa;

struct ifa_plan {
    ifa_params prm;
    KernelChoice kc;
    int num_sms, P_max, device;
    size_t partial_bytes, ws_bytes;
    int* d_state;  // [0]: device error word; from byte 8 on: kMaxCtas arrival counters
    const void* last_k;
    const void* last_v;
    const void* last_mask;
    DecodeParams* dp;
    int64_t last_launches;
    std::vector<int32_t> bdata;
    // one tensor per batch: 4 TMA descriptors per batch on the device, their host copy, and the
    // pointers and extents they were encoded for
    CUtensorMap* d_maps;
    std::vector<CUtensorMap> h_maps;
    std::vector<const void*> list_k, list_v;
    std::vector<int64_t> list_s;
};

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

extern "C" ifa_status ifa_create(const ifa_params* params, ifa_plan** plan, size_t* workspace_bytes) {
    if (!params || !plan || !workspace_bytes) return IFA_ERR_PARAM_NULLPTR;
    *plan = nullptr;
    *workspace_bytes = 0;
    KernelChoice kc;
    const ifa_status st = choose_kernel(*params, &kc);
    if (st != IFA_OK) return st;

    ifa_plan* pl = new (std::nothrow) ifa_plan();
    if (!pl) return IFA_ERR_RUNTIME;
    pl->prm = *params;
    pl->kc = kc;
    if (cudaGetDevice(&pl->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&pl->num_sms, cudaDevAttrMultiProcessorCount, pl->device) != cudaSuccess) {
        cudaGetLastError();
        delete pl;
        return IFA_ERR_RUNTIME;
    }
    pl->P_max = std::max(1, std::min(kMaxCtas, pl->num_sms));
    pl->partial_bytes = align_up((size_t)2 * pl->P_max * kc.slot_floats * sizeof(float), 256);
    pl->ws_bytes = pl->partial_bytes;
    if (params->B > kInlineB) pl->ws_bytes += align_up((size_t)(3 * params->B + 1) * sizeof(int32_t), 256);
    const size_t state_bytes = 8 + (size_t)kMaxCtas * sizeof(unsigned int);
    if (cudaMalloc(&pl->d_state, state_bytes) != cudaSuccess ||
        cudaMemset(pl->d_state, 0, state_bytes) != cudaSuccess) {
        cudaGetLastError();
        delete pl;
        return IFA_ERR_RUNTIME;
    }
    pl->dp = new (std::nothrow) DecodeParams();
    if (!pl->dp) {
        cudaFree(pl->d_state);
        delete pl;
        return IFA_ERR_RUNTIME;
    }
    pl->last_k = pl->last_v = pl->last_mask = nullptr;
    pl->last_launches = 0;
    pl->d_maps = nullptr;
    if (params->kvFormat == IFA_KV_TENSORLIST && params->B > 0) {
        if (cudaMalloc(&pl->d_maps, (size_t)4 * params->B * sizeof(CUtensorMap)) != cudaSuccess) {
            cudaGetLastError();
            cudaFree(pl->d_state);
            delete pl->dp;
            delete pl;
            return IFA_ERR_RUNTIME;
        }
    }
    *plan = pl;
    *workspace_bytes = pl->ws_bytes;
    return IFA_OK;
}

extern "C" int64_t ifa_last_launch_count(const ifa_plan* plan) { return plan ? plan->last_launches : 0; }

extern "C" ifa_status ifa_destroy(ifa_plan* plan) {
    if (!plan) return IFA_OK;
    cudaFree(plan->d_state);
    if (plan->d_maps) cudaFree(plan->d_maps);
    delete plan->dp;
    delete plan;
    return IFA_OK;
}

extern "C" ifa_status ifa_get_device_errors(ifa_plan* plan, void* stream, int64_t* flags) {
    if (!plan || !flags) return IFA_ERR_PARAM_NULLPTR;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int h = 0;
    if (cudaMemcpyAsync(&h, plan->d_state, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return IFA_ERR_RUNTIME;
    }
    // A call that gave up on a wait (bit 2) may have left arrival counters behind: clear them
    // with the error word, so the next call starts from zero counters again.
    const size_t clear = (h & kErrTimeout) ? 8 + (size_t)kMaxCtas * sizeof(unsigned int) : sizeof(int);
    if (cudaMemsetAsync(plan->d_state, 0, clear, s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return IFA_ERR_RUNTIME;
    }
    *flags = h;
    return IFA_OK;
}

// The call after argument checks: windows, split, descriptors, launch.  kv_maps: the per-batch
// descriptors of a tensor-list call (the key/value maps of the contiguous or paged cache
// otherwise).
static ifa_status run_planned(ifa_plan* pl, const void* query, const void* key, const void* value,
                              const void* attenMask, const int64_t* actualSeqLengths, const int64_t* kvPaddingSize,
                              int64_t n_kv_padding, const int32_t* blockTable, const void* antiquantScale,
                              const void* antiquantOffset, const void* quantScale2, const void* quantOffset2,
                              void* attentionOut, void* workspace, size_t workspace_bytes, void* stream,
                              const CUtensorMap* kv_maps) {
    const ifa_params& p = pl->prm;
    ifa_status st = IFA_OK;
    if (pl->ws_bytes > 0 && !workspace) return IFA_ERR_PARAM_NULLPTR;
    if (workspace_bytes < pl->ws_bytes) return IFA_ERR_PARAM_INVALID;
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) % 16) != 0) return IFA_ERR_PARAM_INVALID;
    pl->last_launches = 0;
    const int B = (int)p.B;
    if (B == 0) return IFA_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (B > kInlineB) {
        // Beyond kInlineB batches the windows reach the device by a copy from pageable host
        // memory that the plan reuses, which a CUDA graph cannot hold: under capture the call
        // is refused before it touches the stream, so the capture stays usable.
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) {
            cudaGetLastError();
            return IFA_ERR_RUNTIME;
        }
        if (cap != cudaStreamCaptureStatusNone) return IFA_ERR_PARAM_INVALID;
    }

    std::vector<int32_t>& bd = pl->bdata;
    bd.assign((size_t)3 * B + 1, 0);
    int64_t W = 0;
    int max_seq_tiles = 0;
    st = build_windows(p, pl->kc, actualSeqLengths, kvPaddingSize, n_kv_padding, bd.data(), &W, &max_seq_tiles);
    if (st != IFA_OK) return st;
    const int P = choose_grid(p, W, max_seq_tiles, pl->P_max);

    DecodeParams& dp = *pl->dp;
    if (!kv_maps && (key != pl->last_k || value != pl->last_v)) {
        pl->last_k = pl->last_v = nullptr;
        if (!encode_kv_maps(p, pl->kc, key, value, dp)) return IFA_ERR_RUNTIME;
        pl->last_k = key;
        pl->last_v = value;
    }
    if (attenMask != pl->last_mask || !p.has_mask) {
        pl->last_mask = nullptr;
        if (!encode_mask_map(p, pl->kc, attenMask, dp)) return IFA_ERR_RUNTIME;
        pl->last_mask = attenMask;
    }
    fill_decode_params(dp, p, pl->kc, query, attenMask, blockTable, antiquantScale, antiquantOffset, quantScale2,
                       quantOffset2, attentionOut, W, P);
    build_bounds(p, pl->kc, bd.data(), W, P, dp.bounds);
    dp.kv_maps = kv_maps;
    dp.partials = reinterpret_cast<float*>(workspace);
    dp.err = pl->d_state;
    dp.counters = reinterpret_cast<unsigned int*>(reinterpret_cast<char*>(pl->d_state) + 8);
    if (B <= kInlineB) {
        std::memcpy(dp.bdata_inline, bd.data(), bd.size() * sizeof(int32_t));
        dp.ext_bdata = nullptr;
    } else {
        // Pageable source: the copy is staged before cudaMemcpyAsync returns, so bd may be reused.
        int32_t* ext = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(workspace) + pl->partial_bytes);
        if (cudaMemcpyAsync(ext, bd.data(), bd.size() * sizeof(int32_t), cudaMemcpyHostToDevice, s) != cudaSuccess) {
            cudaGetLastError();
            return IFA_ERR_RUNTIME;
        }
        dp.ext_bdata = ext;
    }
    if (pl->kc.launch(dp, P, s) != cudaSuccess) {
        cudaGetLastError();
        return IFA_ERR_RUNTIME;
    }
    pl->last_launches = 1;
    return IFA_OK;
}

extern "C" ifa_status ifa_run(ifa_plan* pl, const void* query, const void* key, const void* value,
                              const void* attenMask, const int64_t* actualSeqLengths,
                              const int64_t* kvPaddingSize, int64_t n_kv_padding, const int32_t* blockTable,
                              const void* antiquantScale, const void* antiquantOffset, const void* quantScale2,
                              const void* quantOffset2, void* attentionOut, void* workspace, size_t workspace_bytes,
                              void* stream) {
    if (!pl) return IFA_ERR_PARAM_NULLPTR;
    const ifa_params& p = pl->prm;
    if (p.kvFormat == IFA_KV_TENSORLIST) return IFA_ERR_PARAM_INVALID;  // ifa_run_tensorlist
    const ifa_status st = check_run_pointers(p, query, key, value, attenMask, actualSeqLengths, kvPaddingSize,
                                             n_kv_padding, blockTable, antiquantScale, antiquantOffset, quantScale2,
                                             quantOffset2, attentionOut);
    if (st != IFA_OK) return st;
    return run_planned(pl, query, key, value, attenMask, actualSeqLengths, kvPaddingSize, n_kv_padding, blockTable,
                       antiquantScale, antiquantOffset, quantScale2, quantOffset2, attentionOut, workspace,
                       workspace_bytes, stream, nullptr);
}

extern "C" ifa_status ifa_run_tensorlist(ifa_plan* pl, const void* query, const void* const* keyList,
                                         const void* const* valueList, const int64_t* kvSeqLens, const void* attenMask,
                                         const int64_t* actualSeqLengths, const void* antiquantScale,
                                         const void* antiquantOffset, const void* quantScale2,
                                         const void* quantOffset2, void* attentionOut, void* workspace,
                                         size_t workspace_bytes, void* stream) {
    if (!pl) return IFA_ERR_PARAM_NULLPTR;
    const ifa_params& p = pl->prm;
    if (p.kvFormat != IFA_KV_TENSORLIST) return IFA_ERR_PARAM_INVALID;
    const int B = (int)p.B;
    if (B > 0 && (!keyList || !valueList || !kvSeqLens)) return IFA_ERR_PARAM_NULLPTR;
    // the per-tensor pointers stand in for key/value in the common checks (NULL and alignment)
    const void* k0 = B > 0 ? keyList[0] : query;
    const void* v0 = B > 0 ? valueList[0] : query;
    ifa_status st = check_run_pointers(p, query, k0, v0, attenMask, actualSeqLengths, nullptr, 0, nullptr,
                                       antiquantScale, antiquantOffset, quantScale2, quantOffset2, attentionOut);
    if (st != IFA_OK) return st;
    bool same = (int)pl->list_k.size() == B;
    for (int b = 0; b < B; ++b) {
        if (!keyList[b] || !valueList[b]) return IFA_ERR_PARAM_NULLPTR;
        if ((reinterpret_cast<uintptr_t>(keyList[b]) % 16) || (reinterpret_cast<uintptr_t>(valueList[b]) % 16))
            return IFA_ERR_PARAM_INVALID;
        if (kvSeqLens[b] < 1 || kvSeqLens[b] > p.maxSeqLen) return IFA_ERR_PARAM_INVALID;
        if (actualSeqLengths && (actualSeqLengths[b] < 0 || actualSeqLengths[b] > kvSeqLens[b]))
            return IFA_ERR_PARAM_INVALID;
        same = same && pl->list_k[b] == keyList[b] && pl->list_v[b] == valueList[b] && pl->list_s[b] == kvSeqLens[b];
    }
    // a missing actualSeqLengths means each tensor's own S_b
    std::vector<int64_t> lens;
    if (!actualSeqLengths && B > 0) lens.assign(kvSeqLens, kvSeqLens + B);
    const int64_t* use_lens = actualSeqLengths ? actualSeqLengths : (B > 0 ? lens.data() : nullptr);
    if (B > 0 && !same) {
        // The descriptor copy reads pageable host memory, which a CUDA graph cannot replay:
        // under capture the lists must be those of the plan's previous call.
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(reinterpret_cast<cudaStream_t>(stream), &cap) != cudaSuccess) {
            cudaGetLastError();
            return IFA_ERR_RUNTIME;
        }
        if (cap != cudaStreamCaptureStatusNone) return IFA_ERR_PARAM_INVALID;
        // batch b's tensor is a one-batch contiguous cache of extent S_b: encode its four maps
        pl->list_k.clear();
        pl->h_maps.assign((size_t)4 * B, CUtensorMap{});
        ifa_params one = p;
        one.B = 1;
        one.kvFormat = IFA_KV_CONTIG;
        for (int b = 0; b < B; ++b) {
            one.maxSeqLen = kvSeqLens[b];
            CUtensorMap* m = &pl->h_maps[(size_t)4 * b];
            if (!encode_kv_map(one, pl->kc, keyList[b], pl->kc.box_rows, m) ||
                !encode_kv_map(one, pl->kc, keyList[b], pl->kc.tail_rows, m + 1) ||
                !encode_kv_map(one, pl->kc, valueList[b], pl->kc.box_rows, m + 2) ||
                !encode_kv_map(one, pl->kc, valueList[b], pl->kc.tail_rows, m + 3))
                return IFA_ERR_RUNTIME;
        }
        // Pageable source: the copy is staged before cudaMemcpyAsync returns, so h_maps may change.
        if (cudaMemcpyAsync(pl->d_maps, pl->h_maps.data(), pl->h_maps.size() * sizeof(CUtensorMap),
                            cudaMemcpyHostToDevice, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
            cudaGetLastError();
            return IFA_ERR_RUNTIME;
        }
        pl->list_k.assign(keyList, keyList + B);
        pl->list_v.assign(valueList, valueList + B);
        pl->list_s.assign(kvSeqLens, kvSeqLens + B);
    }
    return run_planned(pl, query, k0, v0, attenMask, use_lens, nullptr, 0, nullptr, antiquantScale, antiquantOffset,
                       quantScale2, quantOffset2, attentionOut, workspace, workspace_bytes, stream, pl->d_maps);
}
