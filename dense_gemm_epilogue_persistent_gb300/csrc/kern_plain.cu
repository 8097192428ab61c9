// Persistent-GEMM variants whose cluster is one CTA group (a single CTA, or a
// CTA pair for cta_group 2): no operand is shared, no load multicasts.
// Compiled once per input width, GB300_AB = 2 (fp16/bf16, tcgen05 kind::f16),
// 1 (fp8, kind::f8f6f4) or 4 (tf32 in fp32 storage, kind::tf32), per count of
// epilogue warps per tensor-memory lane quarter, GB300_EPW = 1 or 2, and with
// or without stream-K items, GB300_SK = 0 or 1.
#include "gemm_kernel.cuh"
#include "kernels.h"

namespace gb300 {

const void* GB300_PLAIN_NAME(GB300_AB, GB300_EPW, GB300_SK)(int cta_group, int ka) {
  if (cta_group == 1 && ka == 1)
    return (const void*)&persistent_gemm_kernel<1, GB300_AB, 1, 1, 1, GB300_EPW, GB300_SK>;
  if (cta_group == 1 && ka == 2)
    return (const void*)&persistent_gemm_kernel<1, GB300_AB, 2, 1, 1, GB300_EPW, GB300_SK>;
  if (cta_group == 2 && ka == 2)
    return (const void*)&persistent_gemm_kernel<2, GB300_AB, 2, 1, 1, GB300_EPW, GB300_SK>;
  return nullptr;
}

}  // namespace gb300
