// Instantiations of the split-KV decode kernel for bf16 key/value given as one tensor per batch.
#include "decode_kernel.cuh"

namespace ifa {
DecodeLaunchFn decode_launcher_tl_bf16(int dpad, int nt) {
    if (dpad == 64) return nt == 1 ? launch_decode<KV_BF16, 64, 1, true> : launch_decode<KV_BF16, 64, 2, true>;
    if (dpad == 128) return nt == 1 ? launch_decode<KV_BF16, 128, 1, true> : launch_decode<KV_BF16, 128, 2, true>;
    if (dpad == 256 && nt == 1) return launch_decode<KV_BF16, 256, 1, true>;
    return nullptr;
}
}  // namespace ifa
