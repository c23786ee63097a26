// Instantiations of the split-KV decode kernel for i8 key/value.
#include "decode_kernel.cuh"

namespace ifa {
DecodeLaunchFn decode_launcher_i8(int dpad, int nt) {
    if (dpad == 128) return nt == 1 ? launch_decode<KV_I8, 128, 1> : launch_decode<KV_I8, 128, 2>;
    if (dpad == 256 && nt == 1) return launch_decode<KV_I8, 256, 1>;
    return nullptr;
}
}  // namespace ifa
