// Log-sum-exp combine of split-KV partials: one CTA per sequence that the
// partial kernel's CTA boundaries cut into pieces.  For every query head g of
// the sequence: M = max_k m_k, L = sum_k l_k 2^(m_k - M),
// out = sum_k O_k 2^(m_k - M) / L, summed in piece order (deterministic), and
// zero when no token survived.  int8 key/value: out = scale_V * (o + offset_V).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "decode.cuh"
#include "ptx.cuh"

namespace ifa {

__device__ __forceinline__ float ld_q16(const void* base, long long idx, int is_bf16) {
    const unsigned short u = __ldg(reinterpret_cast<const unsigned short*>(base) + idx);
    return is_bf16 ? __bfloat162float(__ushort_as_bfloat16(u)) : __half2float(__ushort_as_half(u));
}

__global__ void __launch_bounds__(256) combine_kernel(const __grid_constant__ CombineParams p) {
    pdl_wait_primary();
    extern __shared__ float fsm[];
    const CombineJob jb = p.jobs[blockIdx.x];
    const int npieces = jb.c_last - jb.c_first + 1;
    const int RS = p.KV_N * p.NGS;
    const int b = jb.seq / RS;
    const int rr = jb.seq % RS;
    const int h = rr / p.NGS;
    const int gs = rr % p.NGS;
    const int GTv = min(p.GT, p.G - gs * p.GT);
    const int mo = p.gt_pad * p.d_pad;
    float* live = fsm + npieces * p.gt_pad;

    for (int g = threadIdx.x; g < GTv; g += blockDim.x) {
        float M = -INFINITY;
        for (int k = 0; k < npieces; ++k) {
            const int slot = k == 0 ? 2 * jb.c_first + jb.first_odd : 2 * (jb.c_first + k);
            M = fmaxf(M, p.partials[(long long)slot * p.slot_floats + mo + g]);
        }
        float L = 0.f;
        for (int k = 0; k < npieces; ++k) {
            const int slot = k == 0 ? 2 * jb.c_first + jb.first_odd : 2 * (jb.c_first + k);
            const float* sp = p.partials + (long long)slot * p.slot_floats;
            const float f = (M == -INFINITY) ? 0.f : exp2f(sp[mo + g] - M);
            fsm[k * p.gt_pad + g] = f;
            L += sp[mo + p.gt_pad + g] * f;
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        for (int k = 0; k < npieces; ++k) fsm[k * p.gt_pad + g] *= inv;
        live[g] = L > 0.f ? 1.f : 0.f;
    }
    __syncthreads();

    const long long obase = ((long long)b * p.N + (long long)h * p.G + (long long)gs * p.GT) * p.D;
    for (int idx = threadIdx.x; idx < GTv * p.D; idx += blockDim.x) {
        const int g = idx / p.D;
        const int d = idx - g * p.D;
        float o = 0.f;
        for (int k = 0; k < npieces; ++k) {
            const int slot = k == 0 ? 2 * jb.c_first + jb.first_odd : 2 * (jb.c_first + k);
            o += fsm[k * p.gt_pad + g] * p.partials[(long long)slot * p.slot_floats + g * p.d_pad + d];
        }
        if (p.kv_i8) {
            if (live[g] != 0.f) {
                const long long si = p.aq_per_channel ? (long long)(p.KV_N + h) * p.D + d : 1;
                o = (o + ld_q16(p.aq_offset, si, p.q_bf16)) * ld_q16(p.aq_scale, si, p.q_bf16);
            } else {
                o = 0.f;
            }
        }
        if (p.q_bf16) reinterpret_cast<__nv_bfloat16*>(p.out)[obase + idx] = __float2bfloat16_rn(o);
        else reinterpret_cast<__half*>(p.out)[obase + idx] = __float2half_rn(o);
    }
}

cudaError_t launch_combine(const CombineParams& p, int max_pieces, cudaStream_t stream) {
    const size_t smem = (size_t)(max_pieces + 1) * p.gt_pad * sizeof(float);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.njobs);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, combine_kernel, p);
}

}  // namespace ifa
