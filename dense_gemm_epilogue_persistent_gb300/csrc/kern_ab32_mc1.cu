// tf32-input (fp32 storage, tcgen05 kind::tf32) variants of the persistent GEMM with 1 CTA
// group(s) per cluster.
#include "gemm_kernel.cuh"
#include "kernels.h"

namespace gb300 {

const void* kernel_ab32_mc1(int cta_group, int tile_n) {
  if (cta_group == 1 && tile_n == 128) return (const void*)&persistent_gemm_kernel<1, 128, 4, 1>;
  if (cta_group == 1 && tile_n == 256) return (const void*)&persistent_gemm_kernel<1, 256, 4, 1>;
  if (cta_group == 2 && tile_n == 128) return (const void*)&persistent_gemm_kernel<2, 128, 4, 1>;
  if (cta_group == 2 && tile_n == 256) return (const void*)&persistent_gemm_kernel<2, 256, 4, 1>;
  return nullptr;
}

}  // namespace gb300
