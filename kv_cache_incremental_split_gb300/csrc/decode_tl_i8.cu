// Instantiations of the split-KV decode kernel for i8 key/value given as one tensor per batch.
#include "decode_kernel.cuh"

namespace ifa {
DecodeLaunchFn decode_launcher_tl_i8(int dpad, int nt) {
    if (dpad == 128) return nt == 1 ? launch_decode<KV_I8, 128, 1, true> : launch_decode<KV_I8, 128, 2, true>;
    if (dpad == 256 && nt == 1) return launch_decode<KV_I8, 256, 1, true>;
    return nullptr;
}
}  // namespace ifa
