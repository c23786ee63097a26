// PTX wrappers that only the sparse decode kernels use: a CTA pair's cluster barrier, TMA copies
// multicast to both CTAs of the cluster, and the multicast form of tcgen05.commit.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace ifa {

// Every thread of every CTA of the cluster arrives; global and shared memory writes made before
// it are visible to the cluster's threads after it.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// tma_gather4 into the shared memory of every CTA of the cluster in cta_mask, at dst's offset;
// each destination CTA's barrier at bar's offset receives its bytes.
__device__ __forceinline__ void tma_gather4_mc(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int r0, int r1,
                                               int r2, int r3, uint16_t cta_mask, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes.multicast::cluster"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8, %9;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(smem_u32(bar)),
        "h"(cta_mask), "l"(policy)
        : "memory");
}

// tma_load_2d into every CTA of the cluster in cta_mask (same offsets, as above).
__device__ __forceinline__ void tma_load_2d_mc(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                               uint16_t cta_mask) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "h"(cta_mask)
        : "memory");
}

// Arrive on the barrier at bar's offset in every CTA of the cluster in cta_mask once every
// tcgen05.mma this thread issued so far has completed.
__device__ __forceinline__ void umma_commit_mc(uint64_t* bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

}  // namespace ifa
