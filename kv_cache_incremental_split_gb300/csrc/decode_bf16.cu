// Instantiations of the split-KV decode kernel for bf16 key/value.
#include "decode_kernel.cuh"

namespace ifa {
DecodeLaunchFn decode_launcher_bf16(int dpad, int nt) {
    if (dpad == 64) return nt == 1 ? launch_decode<KV_BF16, 64, 1> : launch_decode<KV_BF16, 64, 2>;
    if (dpad == 128) return nt == 1 ? launch_decode<KV_BF16, 128, 1> : launch_decode<KV_BF16, 128, 2>;
    if (dpad == 256 && nt == 1) return launch_decode<KV_BF16, 256, 1>;
    return nullptr;
}
}  // namespace ifa
