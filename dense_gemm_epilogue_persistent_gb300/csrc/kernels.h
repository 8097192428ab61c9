// Kernel variants compiled into the library, looked up by the host planner.
#pragma once

namespace gb300 {

// Kernel entry for 16-bit (ab_bytes = 2), 8-bit (ab_bytes = 1) or tf32
// (ab_bytes = 4) inputs, CTA
// group 1 or 2, tile width 128 or 256, and mc CTA groups per cluster sharing B
// through TMA multicast (1 or 2); nullptr if that variant is not built.
const void* kernel_ab16_mc1(int cta_group, int tile_n);
const void* kernel_ab16_mc2(int cta_group, int tile_n);
const void* kernel_ab8_mc1(int cta_group, int tile_n);
const void* kernel_ab8_mc2(int cta_group, int tile_n);
const void* kernel_ab32_mc1(int cta_group, int tile_n);
const void* kernel_ab32_mc2(int cta_group, int tile_n);

// 128-byte swizzle atoms along K per ring stage.  Two atoms (8 MMAs per
// barrier round trip) keep the tensor pipe fed far better than one; the only
// variant kept at one is the single-CTA 128x256 tile, whose 96 KB two-atom
// stage would leave room for just two stages.
constexpr int k_atoms(int cta_group, int tile_n) { return (cta_group == 1 && tile_n == 256) ? 1 : 2; }

inline const void* kernel_for(int ab_bytes, int cta_group, int tile_n, int mc) {
  if (ab_bytes == 2) return mc == 1 ? kernel_ab16_mc1(cta_group, tile_n)
                                    : mc == 2 ? kernel_ab16_mc2(cta_group, tile_n) : nullptr;
  if (ab_bytes == 1) return mc == 1 ? kernel_ab8_mc1(cta_group, tile_n)
                                    : mc == 2 ? kernel_ab8_mc2(cta_group, tile_n) : nullptr;
  if (ab_bytes == 4) return mc == 1 ? kernel_ab32_mc1(cta_group, tile_n)
                                    : mc == 2 ? kernel_ab32_mc2(cta_group, tile_n) : nullptr;
  return nullptr;
}

}  // namespace gb300
