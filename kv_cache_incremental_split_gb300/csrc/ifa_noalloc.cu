// ifa_run_noalloc: the decode-attention call for callers that cannot allocate
// device memory.  Some callers cannot call cudaMalloc at all: code running
// inside a memory pool or allocator they do not own, runtimes that forbid
// allocation on their inference path, or code that must not grow the device
// footprint after start-up.  This entry point needs no plan, no workspace and
// no allocation: the split-KV state lives in one file-scope device array of
// fixed size, shared by every call in the process.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/ifa.h"
#include "decode.cuh"

using namespace ifa;

namespace {

constexpr size_t kScratchBytes = IFA_NOALLOC_SCRATCH_BYTES;
// Layout of the scratch: [0, 256) device error word; [256, 256 + 4*kMaxCtas) the arrival
// counters (zero at load time; the CTA that merges each cut sequence resets its counter, so
// every call that runs to the end leaves them at zero); from kPartialOffset on, the partial
// slots.
constexpr size_t kCounterOffset = 256;
constexpr size_t kPartialOffset = 4096;
static_assert(kCounterOffset + sizeof(unsigned int) * kMaxCtas <= kPartialOffset, "scratch layout");

// The scratch every ifa_run_noalloc call on a device shares.  In host code this
// name is only a stand-in; the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of the scratch array on the current device, looked up once per device (the
// first call on a device does this set-up).
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

}  // namespace

extern "C" ifa_status ifa_run_noalloc(const ifa_params* params, const void* query, const void* key,
                                      const void* value, const void* attenMask, const int64_t* actualSeqLengths,
                                      const int64_t* kvPaddingSize, int64_t n_kv_padding,
                                      const int32_t* blockTable, const void* antiquantScale,
                                      const void* antiquantOffset, const void* quantScale2,
                                      const void* quantOffset2, void* attentionOut, int32_t* deviceErrorFlags,
                                      void* stream) {
    if (!params) return IFA_ERR_PARAM_NULLPTR;
    const ifa_params& p = *params;
    KernelChoice kc;
    ifa_status st = choose_kernel(p, &kc);
    if (st != IFA_OK) return st;
    if (p.B > IFA_NOALLOC_MAX_BATCH) return IFA_ERR_PARAM_INVALID;  // windows must fit the launch parameters
    if (p.kvFormat == IFA_KV_TENSORLIST) return IFA_ERR_PARAM_INVALID;  // per-tensor descriptors need device memory
    st = check_run_pointers(p, query, key, value, attenMask, actualSeqLengths, kvPaddingSize, n_kv_padding,
                            blockTable, antiquantScale, antiquantOffset, quantScale2, quantOffset2, attentionOut);
    if (st != IFA_OK) return st;
    if (deviceErrorFlags && (reinterpret_cast<uintptr_t>(deviceErrorFlags) % 4) != 0) return IFA_ERR_PARAM_INVALID;
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
    const size_t slot_bytes = (size_t)kc.slot_floats * sizeof(float);
    const int p_fit = (int)std::min<size_t>(kMaxCtas, (kScratchBytes - kPartialOffset) / (2 * slot_bytes));
    if (p_fit < 1) return IFA_ERR_PARAM_INVALID;
    const int P_max = std::max(1, std::min({kMaxCtas, sms, p_fit}));

    static_assert(IFA_NOALLOC_MAX_BATCH <= kInlineB, "windows travel in the launch parameters");
    DecodeParams dp;
    std::memset(&dp, 0, sizeof(dp));
    int64_t W = 0;
    int max_seq_tiles = 0;
    st = build_windows(p, kc, actualSeqLengths, kvPaddingSize, n_kv_padding, dp.bdata_inline, &W, &max_seq_tiles);
    if (st != IFA_OK) return st;
    const int P = choose_grid(p, W, max_seq_tiles, P_max);
    if (!encode_kv_maps(p, kc, key, value, dp) || !encode_mask_map(p, kc, attenMask, dp)) return IFA_ERR_RUNTIME;
    fill_decode_params(dp, p, kc, query, attenMask, blockTable, antiquantScale, antiquantOffset, quantScale2,
                       quantOffset2, attentionOut, W, P);
    build_bounds(p, kc, dp.bdata_inline, W, P, dp.bounds);
    dp.partials = reinterpret_cast<float*>(scratch + kPartialOffset);
    dp.counters = reinterpret_cast<unsigned int*>(scratch + kCounterOffset);
    dp.err = deviceErrorFlags ? deviceErrorFlags : reinterpret_cast<int*>(scratch);
    dp.ext_bdata = nullptr;
    if (kc.launch(dp, P, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return IFA_ERR_RUNTIME;
    }
    return IFA_OK;
}
