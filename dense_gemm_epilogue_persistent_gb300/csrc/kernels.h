// Kernel variants compiled into the library, looked up by the host planner.
#pragma once

namespace gb300 {

// A variant is fixed by the input width (ab_bytes: 2 for fp16/bf16, 1 for fp8,
// 4 for tf32), the CTA group (cta_group 1: single CTAs, 2: CTA pairs), the
// 128-byte K atoms per ring stage (ka: 1 or 2), the cluster's CTA groups
// along M (mc, sharing B) and along N (nc, sharing A), each 1 or 2, and the
// epilogue warps per tensor-memory lane quarter (epw: 1, or 2 for clusters of
// one CTA group) and stream-K items (sk: 0, or 1 for clusters of one CTA
// group).  The tile width is a launch parameter.
//
// kern_plain.cu, compiled once per input width, epw and sk, holds the clusters
// of one CTA group; kern_shared.cu, compiled once per input width and
// (mc, nc), holds the operand-sharing clusters, whose TMA loads multicast.
// Only the single-GPU library links the latter (GB300_MULTICAST = 1).
#define GB300_PLAIN_ENTRIES(X)                                                          \
  X(2, 1, 0) X(1, 1, 0) X(4, 1, 0) X(2, 2, 0) X(1, 2, 0) X(4, 2, 0) X(2, 1, 1) X(1, 1, 1) \
  X(4, 1, 1) X(2, 2, 1) X(1, 2, 1) X(4, 2, 1)
#define GB300_SHARED_ENTRIES(X) \
  X(2, 2, 1) X(2, 1, 2) X(2, 2, 2) X(1, 2, 1) X(1, 1, 2) X(1, 2, 2) X(4, 2, 1) X(4, 1, 2) X(4, 2, 2)

// (two levels, so that macro arguments are expanded before they are pasted)
#define GB300_PLAIN_NAME_(ab, epw, sk) kernel_plain_ab##ab##_e##epw##_s##sk
#define GB300_PLAIN_NAME(ab, epw, sk) GB300_PLAIN_NAME_(ab, epw, sk)
#define GB300_SHARED_NAME_(ab, mc, nc) kernel_shared_ab##ab##_m##mc##_n##nc
#define GB300_SHARED_NAME(ab, mc, nc) GB300_SHARED_NAME_(ab, mc, nc)

#define GB300_DECLARE_PLAIN(ab, epw, sk) \
  const void* GB300_PLAIN_NAME(ab, epw, sk)(int cta_group, int ka);
#define GB300_DECLARE_SHARED(ab, mc, nc) \
  const void* GB300_SHARED_NAME(ab, mc, nc)(int cta_group, int ka);
GB300_PLAIN_ENTRIES(GB300_DECLARE_PLAIN)
GB300_SHARED_ENTRIES(GB300_DECLARE_SHARED)
#undef GB300_DECLARE_PLAIN
#undef GB300_DECLARE_SHARED

#ifndef GB300_MULTICAST
#define GB300_MULTICAST 0
#endif

// 128-byte swizzle atoms along K per ring stage the planner gives a single CTA
// of width tile_n: two atoms (8 MMAs per barrier round trip) keep the tensor
// pipe fed far better than one, unless a two-atom stage is so large that
// fewer than three stages fit (128 x 160 and wider single-CTA tiles).
// CTA pairs always take two.
constexpr int k_atoms(int cta_group, int tile_n) {
  return (cta_group == 1 && tile_n > 128) ? 1 : 2;
}

inline const void* kernel_for(int ab_bytes, int cta_group, int ka, int mc, int nc, int epw = 1,
                              int sk = 0) {
  if (mc == 1 && nc == 1) {
#define GB300_PICK_PLAIN(ab, e, k) \
  if (ab_bytes == ab && epw == e && sk == k) return GB300_PLAIN_NAME(ab, e, k)(cta_group, ka);
    GB300_PLAIN_ENTRIES(GB300_PICK_PLAIN)
#undef GB300_PICK_PLAIN
    return nullptr;
  }
  if (epw != 1 || sk != 0) return nullptr;
#if GB300_MULTICAST
#define GB300_PICK_SHARED(ab, m, n) \
  if (ab_bytes == ab && mc == m && nc == n) return GB300_SHARED_NAME(ab, m, n)(cta_group, ka);
  GB300_SHARED_ENTRIES(GB300_PICK_SHARED)
#undef GB300_PICK_SHARED
#endif
  return nullptr;
}

}  // namespace gb300
