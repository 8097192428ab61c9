// TMA loads with cluster multicast (one box written into the shared memory of
// several CTAs of the cluster).  Kept apart from ptx.cuh: only the kernel
// units of clusters that share operands include this header, and only the
// single-GPU library links them.  Every tensor map these loads read covers
// memory of the GPU the kernel runs on.
#pragma once

#include "ptx.cuh"

namespace gb300 {

// Multicast variants: the box lands at the same shared-memory offset in every
// CTA of `cta_mask`, and each destination's barrier at the offset of `bar`
// receives the completion.  With cta_group::2 the completion goes to the
// barrier in the even (leader) CTA of each destination's pair.
__device__ __forceinline__ void tma_load_3d_mc(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                               int32_t c0, int32_t c1, int32_t c2,
                                               uint16_t cta_mask, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".multicast::cluster.L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6, %7;"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2),
         "h"(cta_mask), "l"(pol)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d_pair_mc(uint32_t dst, const CUtensorMap* map,
                                                    uint32_t cluster_bar, int32_t c0, int32_t c1,
                                                    int32_t c2, uint16_t cta_mask, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".multicast::cluster.cta_group::2.L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6, %7;"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(cluster_bar), "r"(c0), "r"(c1),
         "r"(c2), "h"(cta_mask), "l"(pol)
      : "memory");
}

template <int CG>
struct OperandLoad<CG, true> {
  __device__ static __forceinline__ void load(uint32_t dst, const CUtensorMap* map,
                                              uint32_t bar, int32_t c0, int32_t c1, int32_t c2,
                                              uint16_t cta_mask, uint64_t pol) {
    if constexpr (CG == 1) tma_load_3d_mc(dst, map, bar, c0, c1, c2, cta_mask, pol);
    else tma_load_3d_pair_mc(dst, map, bar, c0, c1, c2, cta_mask, pol);
  }
};

}  // namespace gb300
