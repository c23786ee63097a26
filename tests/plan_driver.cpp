// Host-only driver for the split planner (build_windows, choose_grid, build_bounds):
// reads one problem per line on stdin and prints the CTA tile bounds.  Compiled by
// tests/test_plan_host.py against kv_cache_incremental_split_gb300/csrc/plan.cu; the
// kernel launchers are stubs, nothing touches a GPU.
//
// input line:  B N KV_N D kv_dtype(0 bf16, 2 int8) split_tiles P_max len_0 ... len_{B-1}
// output line: W P T piece_cost cut_cost bounds_0 ... bounds_P   (or "error <status>");
//              the costs are in 1/16 tiles
// Windows only (N = 8, KV_N = 2, D = 128, bf16, BNSD):
// input line:  w B Smax paged(0/1) bt_cols block_size n_pads pad_0 .. pad_{n_pads-1} len_0 .. len_{B-1}
//              (n_pads 0: no kvPaddingSize; a length of -9 stands for "no actualSeqLengths")
// output line: W T st_0 .. st_{B-1} len_0 .. len_{B-1}   (or "error <status>")
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

static void windows_line(std::istringstream& in) {
    long long B, smax, paged, cols, bs, npads;
    if (!(in >> B >> smax >> paged >> cols >> bs >> npads)) return;
    std::vector<int64_t> pads(npads), lens(B);
    for (auto& x : pads) in >> x;
    bool no_lens = false;
    for (auto& l : lens) {
        in >> l;
        no_lens = no_lens || l == -9;
    }
    ifa_params p;
    std::memset(&p, 0, sizeof(p));
    p.B = B;
    p.numHeads = 8;
    p.numKeyValueHeads = 2;
    p.headDim = 128;
    p.maxSeqLen = smax;
    p.q_dtype = IFA_BF16;
    p.kv_dtype = IFA_BF16;
    p.inputLayout = IFA_LAYOUT_BNSD;
    p.kvFormat = paged ? IFA_KV_PAGED_NBSD : IFA_KV_CONTIG;
    p.blockSize = bs;
    p.blockNum = paged ? cols * B : 0;
    p.blockTableCols = paged ? cols : 0;
    p.has_kv_padding = npads > 0;
    p.antiquant = IFA_ANTIQUANT_NONE;
    p.scaleValue = 0.1;
    KernelChoice kc;
    ifa_status st = choose_kernel(p, &kc);
    if (st != IFA_OK) {
        std::printf("error %d\n", (int)st);
        return;
    }
    std::vector<int32_t> bd(3 * B + 1);
    int64_t W = 0;
    int mst = 0;
    st = build_windows(p, kc, no_lens ? nullptr : lens.data(), npads ? pads.data() : nullptr, npads, bd.data(), &W,
                       &mst);
    if (st != IFA_OK) {
        std::printf("error %d\n", (int)st);
        return;
    }
    std::printf("%lld %d", (long long)W, kc.T);
    for (long long b = 0; b < 2 * B; ++b) std::printf(" %d", bd[b]);
    std::printf("\n");
}

int main() {
    std::string line;
    while (std::getline(std::cin, line)) {
        std::istringstream in(line);
        if (!line.empty() && line[0] == 'w') {
            std::string tag;
            in >> tag;
            windows_line(in);
            continue;
        }
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
