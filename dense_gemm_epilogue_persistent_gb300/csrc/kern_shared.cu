// Persistent-GEMM variants whose cluster holds GB300_MC x GB300_NC CTA groups
// that share operands through TMA multicast (B along M when GB300_MC = 2, A
// along N when GB300_NC = 2).  Compiled once per input width (GB300_AB) and
// cluster shape; linked only into the single-GPU library.
#include "ptx_multicast.cuh"
#include "gemm_kernel.cuh"
#include "kernels.h"

namespace gb300 {

const void* GB300_SHARED_NAME(GB300_AB, GB300_MC, GB300_NC)(int cta_group, int ka) {
  if (cta_group == 1 && ka == 1)
    return (const void*)&persistent_gemm_kernel<1, GB300_AB, 1, GB300_MC, GB300_NC, 1, 0>;
  if (cta_group == 1 && ka == 2)
    return (const void*)&persistent_gemm_kernel<1, GB300_AB, 2, GB300_MC, GB300_NC, 1, 0>;
  if (cta_group == 2 && ka == 2)
    return (const void*)&persistent_gemm_kernel<2, GB300_AB, 2, GB300_MC, GB300_NC, 1, 0>;
  return nullptr;
}

}  // namespace gb300
