// Host-only driver for the split planner (build_windows, choose_grid, build_bounds):
// reads one problem per line on stdin and prints the CTA tile bounds.  Compiled by
// tests/test_plan_host.py against kv_cache_incremental_split_gb300/csrc/plan.cu; the
// kernel launchers are stubs, nothing touches a GPU.
//
// input line:  B N KV_N D kv_dtype(0 bf16, 2 int8) split_tiles P_max len_0 ... len_{B-1}
// output line: W P T piece_cost cut_cost bounds_0 ... bounds_P   (or "error <status>");
//              the costs are in 1/16 tiles
#include <cstdio>
#include <cstring>
#include <iostream>
#include <sstream>
#include <string>
#include <vector>

#include "decode.cuh"

namespace ifa {
static cudaError_t stub_launch(const DecodeParams&, int, cudaStream_t) { return cudaSuccess; }
DecodeLaunchFn decode_launcher_bf16(int, int) { return stub_launch; }
DecodeLaunchFn decode_launcher_f16(int, int) { return stub_launch; }
DecodeLaunchFn decode_launcher_i8(int, int) { return stub_launch; }
DecodeLaunchFn decode_launcher_tl_bf16(int, int) { return stub_launch; }
DecodeLaunchFn decode_launcher_tl_f16(int, int) { return stub_launch; }
DecodeLaunchFn decode_launcher_tl_i8(int, int) { return stub_launch; }
}  // namespace ifa

using namespace ifa;

int main() {
    std::string line;
    while (std::getline(std::cin, line)) {
        std::istringstream in(line);
        long long B, N, KVN, D, kv, split, pmax;
        if (!(in >> B >> N >> KVN >> D >> kv >> split >> pmax)) continue;
        std::vector<int64_t> lens(B);
        long long smax = 1;
        for (auto& l : lens) {
            in >> l;
            smax = l > smax ? l : smax;
        }
        ifa_params p;
        std::memset(&p, 0, sizeof(p));
        p.B = B;
        p.numHeads = N;
        p.numKeyValueHeads = KVN;
        p.headDim = D;
        p.maxSeqLen = smax;
        p.q_dtype = kv == 2 ? IFA_F16 : IFA_BF16;
        p.kv_dtype = kv == 2 ? IFA_I8 : IFA_BF16;
        p.inputLayout = IFA_LAYOUT_BNSD;
        p.kvFormat = IFA_KV_CONTIG;
        p.antiquant = kv == 2 ? IFA_ANTIQUANT_PER_TENSOR : IFA_ANTIQUANT_NONE;
        p.scaleValue = 0.1;
        p.splitTiles = split;
        KernelChoice kc;
        ifa_status st = choose_kernel(p, &kc);
        if (st != IFA_OK) {
            std::printf("error %d\n", (int)st);
            continue;
        }
        std::vector<int32_t> bd(3 * B + 1);
        int64_t W = 0;
        int mst = 0;
        st = build_windows(p, kc, lens.data(), nullptr, 0, bd.data(), &W, &mst);
        if (st != IFA_OK) {
            std::printf("error %d\n", (int)st);
            continue;
        }
        const int P = choose_grid(p, W, mst, (int)pmax);
        std::vector<int32_t> bounds(P + 1);
        if (W > 0) build_bounds(p, kc, bd.data(), W, P, bounds.data());
        std::printf("%lld %d %d %d %d", (long long)W, P, kc.T, kc.piece_cost, kc.cut_cost);
        for (int c = 0; c <= P; ++c) std::printf(" %d", W > 0 ? bounds[c] : 0);
        std::printf("\n");
    }
    return 0;
}
