// Kernel variants compiled into the library, looked up by the host planner.
#pragma once

namespace gb300 {

// Kernel entry for 16-bit (ab_bytes = 2) or 8-bit (ab_bytes = 1) inputs, CTA
// group 1 or 2, tile width 128 or 256; nullptr if that variant is not built.
const void* kernel_ab16(int cta_group, int tile_n);
const void* kernel_ab8(int cta_group, int tile_n);

}  // namespace gb300
