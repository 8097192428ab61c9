// Host side of the C ABI declared in include/gemm_gb300.h: argument
// validation, kernel-configuration planning, TMA tensor-map encoding and the
// cluster launch of the persistent kernel.
//
// Validation follows the "Constraints" list of "custom_epilogue_dense_gemm.py"
// (A and B share one type; the contiguous dimension of every tensor is 16-byte
// aligned) and the cuBLASDx Blackwell card's "alignment_unfulfilled" error;
// the shared-memory ring accounting follows that card's "Depth and shared
// memory" bullets (stage = (M*K + N*K) * sizeof(input); 8 bytes per barrier,
// two per stage and two per tensor-memory stage; a 4-byte tensor-memory
// handle) and its opt-in limit check against
// cudaDevAttrMaxSharedMemoryPerBlockOptin before launching.
#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "gemm_gb300.h"
#include "gemm_kernel.cuh"
#include "kernels.h"

#define GEMM_API extern "C" __attribute__((visibility("default")))

namespace {

using gb300::KernelParams;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

constexpr uint64_t kDefaultTimeoutNs = 4000000000ull;
constexpr int kMaxStages = 12;
constexpr int kMaxEpiSlots = 6;
// Default L2 priorities: evict-first for every TMA copy (A/B loads, C/X loads,
// D/Y stores).  Interleaved sustained sweeps on GB300 found it best or tied
// on all five benchmark shapes (fp8 3000x5000x4096: +11% over evict-normal);
// 1500-launch runs under the power cap on 8192^3 (fp16 custom epilogue / bf16)
// give 1450 / 1602 TFLOP/s against 1401 / 1559 with evict-normal A/B loads and
// 1432 / 1600 with evict-last ones; separate A and B policies (A kept longer, since
// the tile order reuses A row-panels across the waves of a strip) were all worse:
// A normal / B first 1410 / 1560, A 25 %-evict-last / B first 1410 / 1570,
// A first / B normal 1370 / 1546, against 1468 / 1625 in the same runs.
constexpr int kDefaultL2Hints = 2 | (2 << 2) | (2 << 4);
constexpr int kDefaultEpiWaitNs = 0;
// base alignment + abort flag + watchdog-test barrier + the epilogue warps'
// ring-batch barriers (one per warp and chunk of a tile) + the two stream-K
// barriers
constexpr int kSmemSlack = 1024 + 16 + 8 * gb300::kMaxEpiWarps * gb300::kMaxChunks + 16;

struct VariantState {
  bool smem_attr_set = false;  // max dynamic smem attribute raised to the opt-in limit
  int occ_smem = 0;            // dynamic smem size of the last occupancy query
  int max_clusters = 0;        // resident clusters at that size
};

// Everything a launch needs, prepared once per distinct call.  A call whose
// arguments (every field of the problem, byte for byte) and forced
// configuration equal a cached entry's launches from it without planning or
// encoding tensor maps again.
struct LaunchKey {
  gemm_problem_t problem;
  uint64_t config_gen;       // bumped by gemm_set_config
};

struct LaunchEntry {
  bool valid = false;
  LaunchKey key;
  gemm_config_t cfg{};
  const void* kern = nullptr;
  int cluster_ctas = 0;
  CUtensorMap maps[6];       // A, B, C, X, D, Y
  KernelParams kp{};
};

constexpr int kLaunchCacheEntries = 4;

// NVTX ranges in the "gemm_gb300" domain around every entry point that
// enqueues work (and around planning and tensor-map encoding on a launch-cache
// miss), so that a profiler's timeline and its range filters (ncu --nvtx
// --nvtx-include "gemm_gb300@gemm_run/") can pick the library's calls out.
// Without a tool attached each push and pop returns at once.
nvtxDomainHandle_t nvtx_domain() {
  static const nvtxDomainHandle_t d = nvtxDomainCreateA("gemm_gb300");
  return d;
}

struct NvtxRange {
  explicit NvtxRange(const char* name) {
    nvtxEventAttributes_t a{};
    a.version = NVTX_VERSION;
    a.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
    a.messageType = NVTX_MESSAGE_TYPE_ASCII;
    a.message.ascii = name;
    nvtxDomainRangePushEx(nvtx_domain(), &a);
  }
  ~NvtxRange() { nvtxDomainRangePop(nvtx_domain()); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

}  // namespace

struct gemm_handle {
  int device = 0;
  int sm_count = 0;
  int smem_optin = 0;
  EncodeTiledFn encode = nullptr;
  uint32_t* d_status = nullptr;
  bool forced = false;
  gemm_config_t forced_cfg{};
  gemm_config_t last{};
  uint64_t timeout_ns = kDefaultTimeoutNs;
  VariantState variants[3][2][2][2][2][2][2];   // [ab 16/8/32][cta_group][k atoms][mc][nc][epw][sk]
  int clusters_by_size[9] = {0, 0, 0, 0, 0, 0, 0, 0, 0};   // resident clusters of 1, 2, 4, 8 CTAs
  uint64_t config_gen = 0;
  LaunchEntry cache[kLaunchCacheEntries];
  int cache_next = 0;
  std::mutex mu;
  void* ws = nullptr;          // gemm_run_host's device copies of its host buffers
  size_t ws_bytes = 0;
  std::mutex ws_mu;
  unsigned long long* d_stats = nullptr;   // ring statistics (statistics build only)
  // Stream-K workspace: one 128 x 256 fp32 partial slot and one flag per SM
  // (null: stream-K is never planned for this handle).
  float* sk_partials = nullptr;
  uint32_t* sk_flags = nullptr;
};

namespace {

int dtype_bytes(int dt) {
  switch (dt) {
    case GEMM_F32: return 4;
    case GEMM_F16: return 2;
    case GEMM_BF16: return 2;
    case GEMM_E4M3: return 1;
    case GEMM_E5M2: return 1;
    case GEMM_TF32: return 4;
  }
  return 0;
}

bool is_epi_type(int dt) { return dt == GEMM_F32 || dt == GEMM_F16 || dt == GEMM_BF16; }
bool is_fp8(int dt) { return dt == GEMM_E4M3 || dt == GEMM_E5M2; }
bool is_ab_type(int dt) {
  return dt == GEMM_F16 || dt == GEMM_BF16 || is_fp8(dt) || dt == GEMM_TF32;
}
// B's type: the descriptor's b when set (0 = GEMM_F32 means "same as ab").
int b_type(const gemm_dtypes_t& t) { return t.b == GEMM_F32 ? t.ab : t.b; }
bool is_layout(int v) { return v == GEMM_K_MAJOR || v == GEMM_MN_MAJOR; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool reads_c(const gemm_problem_t& p) { return p.beta != 0.0f; }
bool reads_x(const gemm_problem_t& p) { return p.X != nullptr && p.x_factor != 0.0f; }

gemm_status_t validate(const gemm_problem_t* pp) {
  if (!pp) return GEMM_ERR_INVALID_ARG;
  const gemm_problem_t& p = *pp;
  const gemm_dtypes_t& t = p.dtypes;
  if (p.M < 0 || p.N < 0 || p.K < 0 || p.L < 0) return GEMM_ERR_INVALID_ARG;
  const int64_t kMax = INT32_MAX;
  if (p.M > kMax || p.N > kMax || p.K > kMax || p.L > kMax) return GEMM_ERR_INVALID_ARG;
  if (!is_layout(p.layoutA) || !is_layout(p.layoutB) || !is_layout(t.cdxy_major))
    return GEMM_ERR_INVALID_ARG;
  if (!is_ab_type(t.ab) || !is_epi_type(t.c) || !is_epi_type(t.d) || !is_epi_type(t.x) ||
      !is_epi_type(t.y))
    return GEMM_ERR_UNSUPPORTED_DTYPE;
  // A and B share one type, except fp8 pairs (the tensor core's f8f6f4 kind
  // takes E4M3 and E5M2 in any pairing).
  if (t.b != GEMM_F32 && !(is_fp8(t.ab) && is_fp8(t.b))) return GEMM_ERR_UNSUPPORTED_DTYPE;
  if (t.epilogue != GEMM_EPI_LINEAR && t.epilogue != GEMM_EPI_RELU) return GEMM_ERR_INVALID_ARG;
  // Accumulator: fp32, or fp16 for fp16 and fp8 inputs (cuBLASDx Blackwell
  // card, "Precision": half with a half or float accumulator, bfloat16 and
  // tf32 with float only, fp8 with half or float).
  if (t.acc != GEMM_F32 && t.acc != GEMM_F16) return GEMM_ERR_UNSUPPORTED_DTYPE;
  if (t.acc == GEMM_F16 && t.ab != GEMM_F16 && !is_fp8(t.ab)) return GEMM_ERR_UNSUPPORTED_DTYPE;
  // tf32 operands are K-major only (cuBLASDx Blackwell card, "Arrangement").
  if (t.ab == GEMM_TF32 && (p.layoutA != GEMM_K_MAJOR || p.layoutB != GEMM_K_MAJOR))
    return GEMM_ERR_UNSUPPORTED_DTYPE;
  if (p.M == 0 || p.N == 0 || p.L == 0) return GEMM_OK;   // nothing to compute

  // Sizes the kernel indexes with 32-bit tile ids and 64-bit element offsets.
  if (cdiv(p.M, 128) * cdiv(p.N, 128) * p.L > kMax) return GEMM_ERR_INVALID_ARG;
  if ((double)p.M * (double)p.N * (double)p.L > 9.0e15) return GEMM_ERR_INVALID_ARG;

  // Outputs and epilogue inputs: packed, one major order.
  const bool m_major = t.cdxy_major == GEMM_MN_MAJOR;
  const int64_t ld = m_major ? p.M : p.N;
  if (!p.D) return GEMM_ERR_INVALID_ARG;
  if (reads_c(p) && !p.C) return GEMM_ERR_INVALID_ARG;
  auto cd_ok = [&](const void* ptr, int dt) {
    return aligned16(ptr) && (ld * dtype_bytes(dt)) % 16 == 0;
  };
  if (!cd_ok(p.D, t.d)) return GEMM_ERR_MISALIGNED;
  if (p.Y && !cd_ok(p.Y, t.y)) return GEMM_ERR_MISALIGNED;
  if (reads_c(p) && !cd_ok(p.C, t.c)) return GEMM_ERR_MISALIGNED;
  if (reads_x(p) && !cd_ok(p.X, t.x)) return GEMM_ERR_MISALIGNED;
  if (p.C && p.C == p.D && reads_c(p) && t.c != t.d) return GEMM_ERR_INVALID_ARG;

  if (p.K > 0) {
    if (!p.A || !p.B) return GEMM_ERR_INVALID_ARG;
    const int64_t es = dtype_bytes(t.ab);
    const int64_t a_min = p.layoutA == GEMM_K_MAJOR ? p.K : p.M;
    const int64_t b_min = p.layoutB == GEMM_K_MAJOR ? p.K : p.N;
    if (p.lda < a_min || p.ldb < b_min) return GEMM_ERR_INVALID_ARG;
    if (!aligned16(p.A) || !aligned16(p.B)) return GEMM_ERR_MISALIGNED;
    if ((p.lda * es) % 16 != 0 || (p.ldb * es) % 16 != 0) return GEMM_ERR_MISALIGNED;
    // Tensor-map limits: strides below 2^40 bytes.
    const int64_t a_rows = p.layoutA == GEMM_K_MAJOR ? p.M : p.K;
    const int64_t b_rows = p.layoutB == GEMM_K_MAJOR ? p.N : p.K;
    const double lim = 1099511627776.0;   // 2^40
    if ((double)p.lda * es * a_rows >= lim || (double)p.ldb * es * b_rows >= lim)
      return GEMM_ERR_INVALID_ARG;
  }
  return GEMM_OK;
}

// A/B ring bytes per CTA: stages x (A stage + B stage) + 8 bytes per
// mbarrier (full and empty per stage, full and empty per accumulator stage)
// + 4 bytes of tensor-memory address.  A stage holds `ka` 128-byte-wide K
// atoms of 128 A rows and tile_n / cta_group B rows.
int ring_bytes(int cta_group, int tile_n, int ka, int stages) {
  const int stage = (128 * 128 + (tile_n / cta_group) * 128) * ka;
  return stages * stage + 8 * (2 * stages + 2 * gb300::kAccStages) + 4;
}

// Bytes of one epilogue slot: C/D region + X/Y region, each 128 x 32
// elements of the wider type stored there.
int epi_slot_bytes(const gemm_problem_t& p) {
  const int sub = 128 * gb300::kEpiChunk;
  int cd = dtype_bytes(p.dtypes.d);
  if (reads_c(p)) cd = std::max(cd, dtype_bytes(p.dtypes.c));
  int xy = 0;
  if (reads_x(p)) xy = dtype_bytes(p.dtypes.x);
  if (p.Y) xy = std::max(xy, dtype_bytes(p.dtypes.y));
  return sub * (cd + xy);
}

// Dynamic shared memory of one CTA: A/B ring, epilogue slots, every mbarrier
// (full/empty per stage, full/empty per accumulator stage, one per epilogue
// warp and slot), tensor-memory address and abort flag, plus 1 KiB of
// alignment slack.
int total_smem(int cg, int bn, int ka, int stages, int slots, int slot_bytes) {
  return ring_bytes(cg, bn, ka, stages) + slots * slot_bytes + 8 * 4 * slots + 4 + kSmemSlack;
}

// Tile widths: multiples of 32 from 64 to 256 (the custom-epilogue example's
// "Constraints" allow MMA tile N from 32 to 256 in steps of 32; 32 is left
// out, its tiles are too thin to feed the tensor pipe from shared memory).
bool valid_tile_n(int bn) { return bn >= 64 && bn <= 256 && bn % 32 == 0; }

bool variant_supports(const gemm_problem_t& p, int cg, int bn, int mc, int nc) {
  if (cg != 1 && cg != 2) return false;
  if (!valid_tile_n(bn)) return false;
  if ((mc != 1 && mc != 2) || (nc != 1 && nc != 2)) return false;
  const int ab_bytes = dtype_bytes(p.dtypes.ab);
  const int atom = 128 / ab_bytes;
  // MN-major operands are staged (and multicast) in swizzle atoms of `atom`
  // rows: a CTA's B part (tile_n / cta_group / mc rows) and A part (128 / nc
  // rows) must be whole atoms.
  if (p.layoutB == GEMM_MN_MAJOR && (bn / cg / mc) % atom != 0) return false;
  if (p.layoutA == GEMM_MN_MAJOR && (128 / nc) % atom != 0) return false;
  return true;
}

// Relative cost of running `tiles` tiles of one variant: waves of tiles times
// the time of one tile, in units of one 128-byte-K-atom k-block of a 256 x 256
// CTA-pair tile.  A tile takes the longer of its main loop and its epilogue,
// plus a fixed cost (pipeline fill, hand-offs, the tail of the epilogue).
// Main loop per k-block: the tile's share of tensor work (tile_n / 256) plus a
// feed overhead that grows as the tile narrows (each CTA still stages 128 A
// rows per k-block):
//   CTA pairs                        tile_n/256 + 0.22 (256 - tile_n)/128
//   single CTAs, 2 atoms per stage   tile_n/256 + 0.18 (256 - tile_n)/128
//   single CTAs, 1 atom per stage    1.15 tile_n/256
// fixed per tile: pairs 15.0 - 1.9 (tile_n - 128)/128, single CTAs 11.0 -
// 0.4 (tile_n - 128)/128; epilogue: tile_n/32 chunks per CTA, each 2.5 + 0.08
// per KB the chunk moves (C and X read, D and Y written, 128 x 32 elements
// each); a last wave split into half-width items (tail_split) costs ~0.8 of a
// wave.  Constants fitted on GB300 to a sweep of all 14 widths x CTA groups
// over 11 workloads (256^3 to 8192^3; 16-bit, fp8, mixed fp8, tf32 inputs;
// fp32 and fp16 accumulators; fp32 and 16-bit epilogues with and without C, X,
// Y; ragged and batched shapes): the pick is the measured fastest variant on
// 10 of them and within 0.2 % on the eleventh.  (With per-warp epilogue
// pipelines the number of C/X slots no longer changes the cost.)
//
// Two epilogue warps per accumulator lane quarter (epw = 2) run two chunk
// chains per quarter side by side: in a GB300 sweep of the same widths with
// the two epilogues alternating, the 10-warp CTAs took 0.85-0.95 of the time
// where the epilogue is the longer side or stands alone (fp8 with 16-bit C, X
// and D; single-wave 2048^3 and 256^3), about 1.0 (0.98-1.03 between runs)
// where the two sides are close (fp8 with 16-bit C and D) and 1.00-1.02 where
// the main loop dominates (8192^3, tf32, fp16 accumulators, batched).
// Modelled as the epilogue x 0.55, the fixed part x 0.9 and the main loop x
// 1.015, offered only where it pays (two_epilogue_warps_pay).
//
// When every cluster runs one tile at most (a single partial wave), a CTA
// pair costs a further 4 units (2048^3: 128 x 256 single-CTA tiles 19.4-19.5
// us against 19.5-20.2 us for 256 x 256 pairs with ten warps, 21.3 against
// 21.6 us with six).
struct TileCost {
  double waves, main_loop, epilogue, fixed;
  bool single_wave;
  int cta_group;
};

TileCost tile_cost(int64_t tiles, int64_t k_blocks, int cg, int ka, int bn, int64_t clusters,
                   double epi_kb, bool can_split) {
  clusters = std::max<int64_t>(1, clusters);
  const int64_t full = tiles / clusters, rem = tiles % clusters;
  TileCost t;
  t.waves = (double)full + (rem == 0 ? 0.0 : (can_split && 2 * rem <= clusters ? 0.8 : 1.0));
  t.single_wave = tiles <= clusters;
  t.cta_group = cg;
  const double w = bn / 256.0;
  double per_kb;
  if (cg == 2) {
    per_kb = w + 0.22 * (256 - bn) / 128.0;
    t.fixed = 15.0 - 1.9 * (bn - 128) / 128.0;
  } else {
    per_kb = ka == 1 ? 1.15 * w : w + 0.18 * (256 - bn) / 128.0;
    t.fixed = 11.0 - 0.4 * (bn - 128) / 128.0;
  }
  t.main_loop = (double)k_blocks * per_kb;
  t.epilogue = (double)(bn / gb300::kEpiChunk) * (2.5 + 0.08 * epi_kb);
  return t;
}

// Whether the automatic choice offers two epilogue warps per lane quarter: the
// tiles fit in one wave (each CTA's epilogue runs after its only main loop,
// with nothing to hide it), or the epilogue is at least as long as the main
// loop.
bool two_epilogue_warps_pay(const TileCost& t) {
  return t.single_wave || t.epilogue >= t.main_loop;
}

double plan_cost(const TileCost& t, int epw) {
  const double main_loop = epw == 2 ? 1.015 * t.main_loop : t.main_loop;
  const double epilogue = epw == 2 ? 0.55 * t.epilogue : t.epilogue;
  const double fixed = epw == 2 ? 0.9 * t.fixed : t.fixed;
  const double pair_single = t.single_wave && t.cta_group == 2 ? 4.0 : 0.0;
  return t.waves * (std::max(main_loop, epilogue) + fixed) + pair_single;
}

// Whether the automatic choice splits k-blocks across clusters (stream-K) for
// a single partial wave of `tiles` tiles on `units` clusters.  Never: on GB300
// the 2048^3 bf16 GEMM with fp32 C/D ran 26.2-26.7 us with stream-K on all 152
// SMs (128 x 256 tiles or 256 x 256 pairs) against 20.5-20.9 us without, in
// alternating runs; each cluster issues 16 % fewer k-blocks, but its MMA
// issuer's cycles per stage rose from ~710 to ~1020 (ring statistics), and
// copies that skipped the partial stores and reads (timing only) still took
// 21.2 us at ~930 cycles per stage: without stream-K every CTA works on the
// same k-block at the same time, so each A/B line is fetched for many CTAs at
// once, and the staggered k offsets of stream-K lose that.  A single wave of
// 152 tiles (2432 x 2048 x 2048) runs in the same ~21 us as 128, so the 24
// idle SMs are not what the single wave loses.  Forced (stream_k = 2) it
// runs, with its parity tests.
bool stream_k_pays(int64_t tiles, int64_t k_blocks, int64_t units) {
  (void)tiles; (void)k_blocks; (void)units;
  return false;
}

// Whether the last wave of a variant may run as half-width items: clusters of
// one CTA group (groups of a larger cluster share operands), half tiles that
// are whole epilogue chunks, and B staged in whole 128-byte atoms at half
// width.
bool can_split_tail(const gemm_problem_t& p, int cg, int bn, int mc, int nc) {
  if (mc != 1 || nc != 1) return false;
  if ((bn / 2) % gb300::kEpiChunk != 0) return false;
  const int atom = 128 / dtype_bytes(p.dtypes.ab);
  return p.layoutB == GEMM_K_MAJOR || (bn / cg / 2) % atom == 0;
}

// Resident clusters of `csize` CTAs: the device's measured occupancy when
// known (clusters_by_size[csize]), else SMs / csize.
int64_t resident_clusters(int sm_count, const int* clusters_by_size, int csize) {
  if (clusters_by_size && csize <= 8 && clusters_by_size[csize] > 0)
    return clusters_by_size[csize];
  return std::max(1, sm_count / csize);
}

gemm_status_t plan(const gemm_problem_t* pp, int sm_count, int smem_optin,
                   const gemm_config_t* forced, gemm_config_t* out,
                   const int* clusters_by_size = nullptr, bool stream_k_ok = true) {
  gemm_status_t st = validate(pp);
  if (st != GEMM_OK) return st;
  if (!out || sm_count <= 0 || smem_optin <= 0) return GEMM_ERR_INVALID_ARG;
  const gemm_problem_t& p = *pp;
  const int ab_bytes = dtype_bytes(p.dtypes.ab);

  const int fcg = forced ? forced->cta_group : 0;
  const int fbn = forced ? forced->tile_n : 0;
  const int fmc = forced ? forced->cluster_m : 0;
  const int fnc = forced ? forced->cluster_n : 0;
  const int fepw = forced ? forced->epi_warps : 0;
  int cg = 0, bn = 0, mc = 0, nc = 0, epw = 0;
  double best = 1e300;
  // KB an epilogue chunk (128 x 32 elements of each tensor) moves per CTA.
  const double epi_kb =
      128.0 * gb300::kEpiChunk *
      ((reads_c(p) ? dtype_bytes(p.dtypes.c) : 0) + (reads_x(p) ? dtype_bytes(p.dtypes.x) : 0) +
       dtype_bytes(p.dtypes.d) + (p.Y ? dtype_bytes(p.dtypes.y) : 0)) / 1024.0;
  // Widest tiles first: among equal costs the wider (fewer-tile) one wins.
  // The automatic choice takes widths of 128 and more (the range the cost
  // model's constants were measured on); 64 and 96 run when forced.
  for (int a : {2, 1})
    for (int b = 256; b >= 64; b -= 32)
      for (int m : {1, 2})
        for (int n : {1, 2}) {
          if ((fcg && a != fcg) || (fbn && b != fbn)) continue;
          if (!fbn && b < 128) continue;
          // The library for multi-GPU processes has no multicast kernels.
          if (!GB300_MULTICAST && (m > 1 || n > 1)) continue;
          // Automatic choice: no operand-sharing clusters (see plan_cost); a
          // forced cluster shape fixes both extents (0 counts as 1).
          if (fmc || fnc) {
            if (m != std::max(fmc, 1) || n != std::max(fnc, 1)) continue;
          } else if (m != 1 || n != 1) {
            continue;
          }
          if (!variant_supports(p, a, b, m, n)) continue;
          const int ka = gb300::k_atoms(a, b);
          const int64_t tiles = cdiv(std::max<int64_t>(p.M, 1), 128 * a * m) *
                                cdiv(std::max<int64_t>(p.N, 1), (int64_t)b * n) *
                                std::max<int64_t>(p.L, 1);
          const int64_t units = resident_clusters(sm_count, clusters_by_size, a * m * n);
          const TileCost tc = tile_cost(tiles, cdiv(p.K, 128 / ab_bytes), a, ka, b, units, epi_kb,
                                        can_split_tail(p, a, b, m, n) &&
                                            !(forced && forced->tail_split == 1));
          // Epilogue warps per lane quarter: forced, or 1 and (where it pays,
          // for clusters of one CTA group) 2.
          for (int e : {1, 2}) {
            if (fepw ? e != fepw
                     : e == 2 && (m != 1 || n != 1 || !two_epilogue_warps_pay(tc)))
              continue;
            const double c = plan_cost(tc, e);
            if (c < best - 1e-9) { best = c; cg = a; bn = b; mc = m; nc = n; epw = e; }
          }
        }
  if (!cg) return GEMM_ERR_UNSUPPORTED_CONFIG;
  if (gemm_tmem_columns(128, bn) > (int)gb300::kAccStride) return GEMM_ERR_UNSUPPORTED_CONFIG;
  const int ka = gb300::k_atoms(cg, bn);
  const int csize = cg * mc * nc;

  // Epilogue slots: a C/D region and an X/Y region of 128 x 32 elements each,
  // sized for the wider of the two types that share it.
  const int slot = epi_slot_bytes(p);
  auto max_stages_for = [&](int slots) {
    int n = 0;
    while (n < kMaxStages && total_smem(cg, bn, ka, n + 1, slots, slot) <= smem_optin) ++n;
    return n;
  };
  // The deepest A/B ring that still leaves two epilogue slots, then every
  // further slot that fits: more slots let C/X loads run further ahead, which
  // keeps the epilogue ahead of fast main loops (8-bit inputs, short K).  (A
  // CTA's last tile takes the C/X its lookahead has not reached from the
  // drained ring, so single-wave problems need no extra slots.)
  const int max_stages = max_stages_for(2);
  const int stages = forced && forced->stages ? forced->stages : max_stages;
  const int64_t tiles_m = cdiv(std::max<int64_t>(p.M, 1), 128 * cg * mc);
  const int64_t tiles_n = cdiv(std::max<int64_t>(p.N, 1), (int64_t)bn * nc);
  const int64_t tiles = tiles_m * tiles_n * std::max<int64_t>(p.L, 1);
  const int64_t units = resident_clusters(sm_count, clusters_by_size, csize);
  if (stages < 2 || stages > max_stages) return GEMM_ERR_UNSUPPORTED_CONFIG;
  int slots = 2;
  while (slots < kMaxEpiSlots && total_smem(cg, bn, ka, stages, slots + 1, slot) <= smem_optin)
    ++slots;
  if (forced && forced->epi_slots) {
    slots = forced->epi_slots;
    if (slots < 2 || slots > kMaxEpiSlots ||
        total_smem(cg, bn, ka, stages, slots, slot) > smem_optin)
      return GEMM_ERR_UNSUPPORTED_CONFIG;
  }

  // Strips of 12 CTA-group tile rows: with the serpentine strip order and the
  // K direction alternating per wave, 8192^3 reads 1.206 GB from DRAM per
  // launch at 12 (1.235 GB at 8, 1.514 GB at 4, 1.307 GB at 16) and runs 0.5-0.8 %
  // faster than at 8; other shapes measured the same at 8 and 12 (re-checked on
  // the current kernel, 3 x 3000 launches each: 12 734.5-735.7 us, 8 736.4-737.8,
  // 10 737-740, 14 738-740, 16 738-741, 6 744-745).  A cluster
  // tile stacks cluster_m group tiles, so the strip counts 12 / cluster_m of
  // them (B shared along M, 8192^3: 1.29 GB read at 6 against 1.58 GB at 12).
  int group_m = forced && forced->group_m ? forced->group_m : std::max(1, 12 / mc);
  group_m = (int)std::max<int64_t>(1, std::min<int64_t>(group_m, tiles_m));

  gemm_config_t c{};
  c.cta_group = cg;
  c.tile_n = bn;
  c.stages = stages;
  c.group_m = group_m;
  c.tile_m = 128 * cg;
  c.cluster_m = mc;
  c.cluster_n = nc;
  c.epi_warps = epw;
  if (c.epi_warps == 2 && csize != cg) return GEMM_ERR_UNSUPPORTED_CONFIG;
  c.l2_hints = forced && (forced->l2_hints & 0x100) ? (forced->l2_hints & 0x3F) : kDefaultL2Hints;
  c.epi_wait_ns = forced && forced->epi_wait_ns > 0 ? forced->epi_wait_ns - 1 : kDefaultEpiWaitNs;
  c.inject_stall = forced && forced->inject_stall ? 1 : 0;
  c.tile_k = 128 / ab_bytes * ka;
  c.acc_stages = gb300::kAccStages;
  c.ring_bytes = ring_bytes(cg, bn, ka, stages);
  c.epi_slots = slots;
  c.epi_slot_bytes = slot;
  // At least half the opt-in limit: one CTA per SM, so no two CTAs ever
  // contend for the 512 tensor-memory columns each allocates.
  c.smem_bytes = std::max(total_smem(cg, bn, ka, stages, slots, slot), smem_optin / 2 + 1024);
  c.tiles = tiles;
  // Stream-K: when the tiles fill less than one wave of clusters, every
  // resident cluster takes an equal contiguous share of all the tiles'
  // k-blocks (fp32 accumulators, clusters of one CTA group, at least one
  // k-block per cluster); a tile's earlier k-blocks come back to its owner as
  // fp32 partial sums, added in cluster order.
  const int64_t k_blocks = cdiv(p.K, (int64_t)c.tile_k);
  const int fsk = forced ? forced->stream_k : 0;
  const bool sk_possible = stream_k_ok && mc == 1 && nc == 1 && p.dtypes.acc != GEMM_F16 &&
                           p.K > 0 && tiles < units && tiles * k_blocks >= units &&
                           bn / gb300::kEpiChunk >= 2 && units * cg <= sm_count;
  const bool sk = sk_possible && (fsk == 2 || (fsk == 0 && stream_k_pays(tiles, k_blocks, units)));
  c.stream_k = sk ? (int)units : 0;
  int64_t split = 0;
  if (!sk && can_split_tail(p, cg, bn, mc, nc) && !(forced && forced->tail_split == 1)) {
    const int64_t rem = tiles % units;
    if (rem > 0 && 2 * rem <= units) split = rem;
  }
  c.tail_split = (int)split;
  c.grid_ctas = (int)((sk ? units : std::min<int64_t>(tiles + split, units)) * csize);
  *out = c;
  return GEMM_OK;
}

CUtensorMapDataType tma_type(int dt) {
  switch (dt) {
    case GEMM_F16: return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    case GEMM_BF16: return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    case GEMM_TF32: return CU_TENSOR_MAP_DATA_TYPE_FLOAT32;   // raw fp32 words
    default: return CU_TENSOR_MAP_DATA_TYPE_UINT8;   // fp8: bytes, never converted
  }
}

// Operand tensor map.  K-major: dims {K, rows, L}, box {one 128-byte atom of
// K, box_rows}.  MN-major: dims {rows, K, L}, box {128 bytes of rows, tile_k}.
// Out-of-range elements of a box are filled with zeros.
bool encode_operand(EncodeTiledFn enc, CUtensorMap* map, const void* ptr, int dt, int64_t rows,
                    int64_t K, int64_t L, int64_t ld, bool mn_major, int box_rows, int tile_k) {
  const int64_t es = dtype_bytes(dt);
  cuuint64_t dims[3], strides[2];
  cuuint32_t box[3], estr[3] = {1, 1, 1};
  if (!mn_major) {
    dims[0] = (cuuint64_t)K; dims[1] = (cuuint64_t)rows; dims[2] = (cuuint64_t)L;
    strides[0] = (cuuint64_t)(ld * es);
    strides[1] = (cuuint64_t)(ld * es * rows);
    box[0] = (cuuint32_t)(128 / es); box[1] = (cuuint32_t)box_rows; box[2] = 1;
  } else {
    dims[0] = (cuuint64_t)rows; dims[1] = (cuuint64_t)K; dims[2] = (cuuint64_t)L;
    strides[0] = (cuuint64_t)(ld * es);
    strides[1] = (cuuint64_t)(ld * es * K);
    box[0] = (cuuint32_t)(128 / es); box[1] = (cuuint32_t)tile_k; box[2] = 1;
  }
  CUresult r = enc(map, tma_type(dt), 3, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Epilogue tensor map over a packed M x N x L tensor, box = 32 rows x 32
// columns (one epilogue warp's rows of one chunk).  Row-major: dims {N, M, L},
// 128-byte (fp32) or 64-byte (16-bit) rows swizzled to match the epilogue's
// shared-memory reads.  Column-major: dims {M, N, L}, unswizzled.
bool encode_epi(EncodeTiledFn enc, CUtensorMap* map, const void* ptr, int dt, int64_t M,
                int64_t N, int64_t L, bool m_major) {
  const int64_t es = dtype_bytes(dt);
  cuuint64_t dims[3], strides[2];
  cuuint32_t box[3], estr[3] = {1, 1, 1};
  CUtensorMapSwizzle sw;
  CUtensorMapDataType ty = dt == GEMM_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : tma_type(dt);
  if (!m_major) {
    dims[0] = (cuuint64_t)N; dims[1] = (cuuint64_t)M; dims[2] = (cuuint64_t)L;
    strides[0] = (cuuint64_t)(N * es);
    strides[1] = (cuuint64_t)(N * es * M);
    box[0] = gb300::kEpiChunk; box[1] = gb300::kSubRows; box[2] = 1;
    sw = es == 4 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  } else {
    dims[0] = (cuuint64_t)M; dims[1] = (cuuint64_t)N; dims[2] = (cuuint64_t)L;
    strides[0] = (cuuint64_t)(M * es);
    strides[1] = (cuuint64_t)(M * es * N);
    box[0] = gb300::kSubRows; box[1] = gb300::kEpiChunk; box[2] = 1;
    sw = CU_TENSOR_MAP_SWIZZLE_NONE;
  }
  CUresult r = enc(map, ty, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

uint32_t make_idesc(int a_type, int b_type_, bool acc_f16, int cg, int bn, bool a_mn, bool b_mn) {
  // kind::f16 / kind::tf32: format 0 = fp16, 1 = bf16, 2 = tf32.
  // kind::f8f6f4: 0 = e4m3, 1 = e5m2.
  auto fmt = [](int t) {
    return t == GEMM_TF32 ? 2u : (t == GEMM_BF16 || t == GEMM_E5M2) ? 1u : 0u;
  };
  uint32_t d = 0;
  d |= (acc_f16 ? 0u : 1u) << 4;                  // accumulator (D) format: 0 fp16, 1 fp32
  d |= fmt(a_type) << 7;                          // A format
  d |= fmt(b_type_) << 10;                        // B format
  d |= (a_mn ? 1u : 0u) << 15;                    // A MN-major
  d |= (b_mn ? 1u : 0u) << 16;                    // B MN-major
  d |= (uint32_t)(bn >> 3) << 17;                 // N >> 3
  d |= (uint32_t)((128 * cg) >> 4) << 24;         // M >> 4
  return d;
}

// Plan the launch of problem `p` on handle `h` (which the caller holds
// locked) and fill `ent`: configuration, kernel, grid, tensor maps and kernel
// parameters (the status word and timeout are set at each launch).
gemm_status_t prepare_launch(gemm_handle* h, const gemm_problem_t& p, LaunchEntry& ent) {
  const int64_t M = p.M, N = p.N, K = p.K, L = p.L;
  const void *A = p.A, *B = p.B, *C = p.C, *X = p.X;
  void *D = p.D, *Y = p.Y;
  const int64_t lda = p.lda, ldb = p.ldb;
  const gemm_layout_t layoutA = p.layoutA, layoutB = p.layoutB;
  const float alpha = p.alpha, beta = p.beta, x_factor = p.x_factor;
  const gemm_dtypes_t* dtypes = &p.dtypes;
  gemm_config_t cfg{};
  const gemm_status_t st = plan(&p, h->sm_count, h->smem_optin, h->forced ? &h->forced_cfg : nullptr, &cfg,
            h->clusters_by_size, h->sk_partials != nullptr && h->sk_flags != nullptr);
  if (st != GEMM_OK) return st;

  const int ab_bytes = dtype_bytes(dtypes->ab);
  const int csize = cfg.cta_group * cfg.cluster_m * cfg.cluster_n;
  const int ka = gb300::k_atoms(cfg.cta_group, cfg.tile_n);
  const int sk = cfg.stream_k > 0 ? 1 : 0;
  const void* kern = gb300::kernel_for(ab_bytes, cfg.cta_group, ka, cfg.cluster_m,
                                       cfg.cluster_n, cfg.epi_warps, sk);
  if (!kern) return GEMM_ERR_UNSUPPORTED_CONFIG;
  VariantState& vs = h->variants[ab_bytes == 2 ? 0 : ab_bytes == 1 ? 1 : 2][cfg.cta_group - 1]
                                [ka - 1][cfg.cluster_m - 1][cfg.cluster_n - 1]
                                [cfg.epi_warps - 1][sk];

  cudaLaunchConfig_t lc{};
  cudaLaunchAttribute attr[1];
  lc.blockDim = dim3(gb300::threads_for(cfg.epi_warps));
  lc.dynamicSmemBytes = (size_t)cfg.smem_bytes;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;

  // The attribute is raised once to the device's opt-in limit, so that every
  // prepared launch of this kernel (cached ones included) may use any size.
  if (!vs.smem_attr_set) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             h->smem_optin) != cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_CUDA;
    }
    vs.smem_attr_set = true;
  }
  if (vs.occ_smem != cfg.smem_bytes) {
    int nclusters = 0;
    lc.gridDim = dim3((unsigned)(csize * h->sm_count));
    if (cudaOccupancyMaxActiveClusters(&nclusters, kern, &lc) != cudaSuccess || nclusters <= 0) {
      cudaGetLastError();
      return GEMM_ERR_CUDA;
    }
    vs.occ_smem = cfg.smem_bytes;
    vs.max_clusters = nclusters;
  }
  int64_t clusters = std::min<int64_t>(cfg.tiles + cfg.tail_split, vs.max_clusters);
  if (cfg.stream_k > 0) {
    // Stream-K runs one item pair on every cluster the kernel can keep
    // resident; the k-block ranges are cut for exactly that many clusters.
    const int64_t k_blocks = cdiv(K, (int64_t)cfg.tile_k);
    clusters = std::min<int64_t>(cfg.stream_k, vs.max_clusters);
    if (clusters <= cfg.tiles || cfg.tiles * k_blocks < clusters) {
      clusters = std::min<int64_t>(cfg.tiles, vs.max_clusters);   // not worth it here: off
      cfg.stream_k = 0;
    } else {
      cfg.stream_k = (int)clusters;
    }
  }
  cfg.grid_ctas = (int)(clusters * csize);

  const bool a_mn = layoutA == GEMM_MN_MAJOR, b_mn = layoutB == GEMM_MN_MAJOR;
  CUtensorMap tmA, tmB;
  std::memset(&tmA, 0, sizeof(tmA));
  std::memset(&tmB, 0, sizeof(tmB));
  if (K > 0) {
    // Each CTA loads 128 / cluster_n A rows and tile_n / cta_group / cluster_m
    // B rows per K atom (the rest of its slices arrive from the CTAs that
    // share them).
    if (!encode_operand(h->encode, &tmA, A, dtypes->ab, M, K, L, lda, a_mn, 128 / cfg.cluster_n,
                        cfg.tile_k) ||
        !encode_operand(h->encode, &tmB, B, dtypes->ab, N, K, L, ldb, b_mn,
                        cfg.tile_n / cfg.cta_group / cfg.cluster_m, cfg.tile_k))
      return GEMM_ERR_CUDA;
  }

  const bool cd_m = dtypes->cdxy_major == GEMM_MN_MAJOR;
  CUtensorMap tmC, tmX, tmD, tmY;
  std::memset(&tmC, 0, sizeof(tmC));
  std::memset(&tmX, 0, sizeof(tmX));
  std::memset(&tmY, 0, sizeof(tmY));
  if (!encode_epi(h->encode, &tmD, D, dtypes->d, M, N, L, cd_m) ||
      (reads_c(p) && !encode_epi(h->encode, &tmC, C, dtypes->c, M, N, L, cd_m)) ||
      (reads_x(p) && !encode_epi(h->encode, &tmX, X, dtypes->x, M, N, L, cd_m)) ||
      (Y && !encode_epi(h->encode, &tmY, Y, dtypes->y, M, N, L, cd_m)))
    return GEMM_ERR_CUDA;

  KernelParams kp{};
  kp.M = (int)M; kp.N = (int)N; kp.K = (int)K; kp.L = (int)L;
  kp.bn = cfg.tile_n;
  kp.tiles_m = (int)cdiv(M, (int64_t)cfg.tile_m * cfg.cluster_m);
  kp.tiles_n = (int)cdiv(N, (int64_t)cfg.tile_n * cfg.cluster_n);
  kp.num_tiles = (int)cfg.tiles;
  kp.k_blocks = (int)cdiv(K, cfg.tile_k);
  kp.group_m = cfg.group_m;
  kp.stages = cfg.stages;
  kp.a_mn_major = a_mn;
  kp.b_mn_major = b_mn;
  const bool acc_f16 = dtypes->acc == GEMM_F16;
  kp.idesc = make_idesc(dtypes->ab, b_type(*dtypes), acc_f16, cfg.cta_group, cfg.tile_n, a_mn,
                        b_mn);
  kp.idesc_half = make_idesc(dtypes->ab, b_type(*dtypes), acc_f16, cfg.cta_group, cfg.tile_n / 2,
                             a_mn, b_mn);
  kp.split_start = (int)(cfg.tiles - cfg.tail_split);
  kp.num_items = (int)(cfg.tiles + cfg.tail_split);
  if (cfg.stream_k > 0) {
    // every resident cluster takes an equal share of all k-blocks, as up to
    // two items (the head of one tile, the tail of the previous one)
    kp.sk_units = cfg.stream_k;
    kp.sk_iters = cfg.tiles * (long long)kp.k_blocks;
    kp.num_items = 2 * cfg.stream_k;
    kp.sk_partials = h->sk_partials;
    kp.sk_flags = h->sk_flags;
  }
  kp.l2_hints = (uint32_t)cfg.l2_hints;
  kp.epi_wait_ns = (uint32_t)cfg.epi_wait_ns;
  kp.inject_stall = cfg.inject_stall;
  // fp16 accumulators keep increasing K: their rounding points are defined on
  // running sums from k = 0.
  kp.k_alternate = acc_f16 || cfg.stream_k > 0 ? 0 : 1;
  kp.status = h->d_status;
  kp.timeout_ns = h->timeout_ns;
  kp.epi.c_dt = dtypes->c;
  kp.epi.d_dt = dtypes->d;
  kp.epi.x_dt = dtypes->x;
  kp.epi.y_dt = dtypes->y;
  kp.epi.cd_m_major = cd_m;
  kp.epi.read_c = reads_c(p);
  kp.epi.read_x = reads_x(p);
  kp.epi.write_y = Y != nullptr;
  kp.epi.alpha = alpha;
  kp.epi.beta = beta;
  kp.epi.x_factor = x_factor;
  kp.epi.relu = dtypes->epilogue == GEMM_EPI_RELU;
  kp.epi.acc_f16 = acc_f16;
  kp.epi.slots = cfg.epi_slots;
  {
    const int sub = 128 * gb300::kEpiChunk;
    int cd = dtype_bytes(dtypes->d);
    if (reads_c(p)) cd = std::max(cd, dtype_bytes(dtypes->c));
    kp.epi.cd_bytes = (uint32_t)(sub * cd);
    kp.epi.xy_bytes = (uint32_t)(cfg.epi_slot_bytes - sub * cd);
  }

  ent.cfg = cfg;
  ent.kern = kern;
  ent.cluster_ctas = csize;
  ent.maps[0] = tmA; ent.maps[1] = tmB; ent.maps[2] = tmC;
  ent.maps[3] = tmX; ent.maps[4] = tmD; ent.maps[5] = tmY;
  ent.kp = kp;
  return GEMM_OK;
}

// Status of a non-zero device status word: a failed bounds check of the
// debug build (0xD0......) or a watchdog timeout (0xE0......).
gemm_status_t status_of_word(uint32_t word) {
  if (word == 0) return GEMM_OK;
  return (word >> 24) == 0xD0u ? GEMM_ERR_DEVICE_CHECK : GEMM_ERR_DEVICE_TIMEOUT;
}

// Resident clusters of 1, 2, 4 and 8 CTAs at one CTA per SM (every
// configuration uses more than half of the shared memory), from the occupancy
// calculator on a representative kernel; `device` must be current.  The
// kernel's shared-memory attribute is process-wide: it is raised to the
// opt-in limit, as every prepared launch raises it, and never lowered, since
// another handle may have launches prepared with more than the size queried
// here.  Counts the calculator does not give stay 0 (the planner then
// assumes SMs / cluster size).
void query_cluster_occupancy(int device, int sms, int optin, int (&clusters)[9]) {
  (void)device;
  const void* kern = gb300::kernel_for(2, 2, 2, 1, 1);
  const int smem = optin / 2 + 1024;
  if (kern && cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, optin) ==
                  cudaSuccess) {
    for (int cs : {1, 2, 4, 8}) {
      cudaLaunchConfig_t lc{};
      cudaLaunchAttribute attr[1];
      lc.gridDim = dim3((unsigned)(cs * sms));
      lc.blockDim = dim3(gb300::kThreads);
      lc.dynamicSmemBytes = (size_t)smem;
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = (unsigned)cs;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      lc.attrs = attr;
      lc.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &lc) == cudaSuccess) clusters[cs] = n;
    }
  }
  cudaGetLastError();
}

}  // namespace

// ====================================================================== C ABI

GEMM_API const char* gemm_status_string(gemm_status_t s) {
  switch (s) {
    case GEMM_OK: return "GEMM_OK";
    case GEMM_ERR_INVALID_ARG: return "GEMM_ERR_INVALID_ARG";
    case GEMM_ERR_UNSUPPORTED_DTYPE: return "GEMM_ERR_UNSUPPORTED_DTYPE";
    case GEMM_ERR_MISALIGNED: return "GEMM_ERR_MISALIGNED";
    case GEMM_ERR_UNSUPPORTED_ARCH: return "GEMM_ERR_UNSUPPORTED_ARCH";
    case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA";
    case GEMM_ERR_DEVICE_TIMEOUT: return "GEMM_ERR_DEVICE_TIMEOUT";
    case GEMM_ERR_UNSUPPORTED_CONFIG: return "GEMM_ERR_UNSUPPORTED_CONFIG";
    case GEMM_ERR_DEVICE_CHECK: return "GEMM_ERR_DEVICE_CHECK";
  }
  return "GEMM_ERR_UNKNOWN";
}

GEMM_API int gemm_tmem_columns(int tile_m, int tile_n) {
  if (tile_m <= 0 || tile_n <= 0 || tile_m > 256 || tile_n > 256) return 0;
  if (tile_m % 64 != 0 || tile_n % 8 != 0) return 0;
  const int blocks = (tile_m % 128 == 0) ? tile_m / 128 : tile_m / 64;
  return blocks * tile_n;
}

GEMM_API gemm_status_t gemm_check(const gemm_problem_t* p) { return validate(p); }

GEMM_API gemm_status_t gemm_plan(const gemm_problem_t* p, int sm_count, int smem_optin,
                                 const gemm_config_t* forced, gemm_config_t* out) {
  return plan(p, sm_count, smem_optin, forced, out);
}

GEMM_API gemm_status_t gemm_create(gemm_handle_t* out, int device) {
  if (!out) return GEMM_ERR_INVALID_ARG;
  *out = nullptr;
  int count = 0;
  if (cudaGetDeviceCount(&count) != cudaSuccess) { cudaGetLastError(); return GEMM_ERR_CUDA; }
  if (device < 0 || device >= count) return GEMM_ERR_INVALID_ARG;
  int major = 0, minor = 0, sms = 0, optin = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) !=
          cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  if (major != 10 || minor != 3) return GEMM_ERR_UNSUPPORTED_ARCH;

  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }

  int prev = 0;
  cudaGetDevice(&prev);
  if (cudaSetDevice(device) != cudaSuccess) { cudaGetLastError(); return GEMM_ERR_CUDA; }
  uint32_t* status = nullptr;
  cudaError_t e = cudaMalloc(&status, sizeof(uint32_t));
  if (e == cudaSuccess) e = cudaMemset(status, 0, sizeof(uint32_t));
  cudaSetDevice(prev);
  if (e != cudaSuccess) {
    if (status) cudaFree(status);
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  // Resident clusters of 1, 2, 4 and 8 CTAs at one CTA per SM.
  int clusters[9] = {0, 0, 0, 0, 0, 0, 0, 0, 0};
  if (cudaSetDevice(device) == cudaSuccess) query_cluster_occupancy(device, sms, optin, clusters);
  cudaGetLastError();
  cudaSetDevice(prev);
  gemm_handle* h = new gemm_handle();
  for (int i = 0; i < 9; ++i) h->clusters_by_size[i] = clusters[i];
  h->device = device;
  h->sm_count = sms;
  h->smem_optin = optin;
  h->encode = reinterpret_cast<EncodeTiledFn>(fn);
  h->d_status = status;
  if constexpr (gb300::kRingStats) {
    // one counter block per CTA of the largest grid (one CTA per SM)
    const size_t bytes = (size_t)sms * gb300::kStatWords * sizeof(unsigned long long);
    if (cudaSetDevice(device) != cudaSuccess || cudaMalloc(&h->d_stats, bytes) != cudaSuccess ||
        cudaMemset(h->d_stats, 0, bytes) != cudaSuccess) {
      cudaGetLastError();
      cudaSetDevice(prev);
      cudaFree(h->d_stats);
      cudaFree(status);
      delete h;
      return GEMM_ERR_CUDA;
    }
    cudaSetDevice(prev);
  }
  // Stream-K workspace (20 MB on 152 SMs), allocated once here so that no
  // launch allocates; without it the planner never chooses stream-K.
  if (cudaSetDevice(device) == cudaSuccess) {
    const size_t pbytes = (size_t)sms * 128 * 256 * sizeof(float);
    if (cudaMalloc(&h->sk_partials, pbytes) != cudaSuccess ||
        cudaMalloc(&h->sk_flags, (size_t)sms * sizeof(uint32_t)) != cudaSuccess ||
        cudaMemset(h->sk_flags, 0, (size_t)sms * sizeof(uint32_t)) != cudaSuccess) {
      cudaGetLastError();
      if (h->sk_partials) cudaFree(h->sk_partials);
      if (h->sk_flags) cudaFree(h->sk_flags);
      h->sk_partials = nullptr;
      h->sk_flags = nullptr;
    }
  }
  cudaSetDevice(prev);
  *out = h;
  return GEMM_OK;
}

GEMM_API gemm_status_t gemm_destroy(gemm_handle_t h) {
  if (!h) return GEMM_OK;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(h->device);
  cudaFree(h->d_status);
  if (h->ws) cudaFree(h->ws);
  if (h->d_stats) cudaFree(h->d_stats);
  if (h->sk_partials) cudaFree(h->sk_partials);
  if (h->sk_flags) cudaFree(h->sk_flags);
  cudaSetDevice(prev);
  delete h;
  return GEMM_OK;
}

GEMM_API gemm_status_t gemm_set_config(gemm_handle_t h, const gemm_config_t* cfg) {
  if (!h) return GEMM_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> g(h->mu);
  if (!cfg) {
    h->forced = false;
    ++h->config_gen;
    return GEMM_OK;
  }
  if ((cfg->cta_group && cfg->cta_group != 1 && cfg->cta_group != 2) ||
      (cfg->tile_n && !valid_tile_n(cfg->tile_n)) || cfg->stages < 0 ||
      (cfg->cluster_m && cfg->cluster_m != 1 && cfg->cluster_m != 2) ||
      (cfg->cluster_n && cfg->cluster_n != 1 && cfg->cluster_n != 2) ||
      cfg->epi_slots < 0 || cfg->epi_slots > kMaxEpiSlots || cfg->epi_wait_ns < 0 ||
      cfg->tail_split < 0 || cfg->tail_split > 1 || cfg->epi_warps < 0 || cfg->epi_warps > 2 ||
      cfg->stream_k < 0 || cfg->stream_k > 2 ||
      cfg->epi_wait_ns > 1000001 ||
      cfg->stages > kMaxStages || cfg->group_m < 0)
    return GEMM_ERR_INVALID_ARG;
  h->forced = true;
  h->forced_cfg = *cfg;
  ++h->config_gen;
  return GEMM_OK;
}

GEMM_API gemm_status_t gemm_last_config(gemm_handle_t h, gemm_config_t* out) {
  if (!h || !out) return GEMM_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> g(h->mu);
  *out = h->last;
  return GEMM_OK;
}

GEMM_API gemm_status_t gemm_set_timeout_ns(gemm_handle_t h, uint64_t ns) {
  if (!h) return GEMM_ERR_INVALID_ARG;
  h->timeout_ns = ns ? ns : kDefaultTimeoutNs;
  return GEMM_OK;
}

GEMM_API gemm_status_t gemm_run(gemm_handle_t h, int64_t M, int64_t N, int64_t K, int64_t L,
                                const void* A, int64_t lda, gemm_layout_t layoutA, const void* B,
                                int64_t ldb, gemm_layout_t layoutB, const void* C, const void* X,
                                void* D, void* Y, float alpha, float beta, float x_factor,
                                const gemm_dtypes_t* dtypes, struct CUstream_st* stream) {
  NvtxRange range("gemm_run");
  if (!h || !dtypes) return GEMM_ERR_INVALID_ARG;
  gemm_problem_t p{M, N, K, L, A, lda, layoutA, B, ldb, layoutB, C, X, D, Y,
                   alpha, beta, x_factor, *dtypes};
  gemm_status_t st = validate(&p);
  if (st != GEMM_OK) return st;
  if (M == 0 || N == 0 || L == 0) return GEMM_OK;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess || cur != h->device) {
    cudaGetLastError();
    return GEMM_ERR_INVALID_ARG;
  }

  std::lock_guard<std::mutex> guard(h->mu);
  LaunchKey key;
  std::memset(&key, 0, sizeof(key));           // padding included: keys compare bytewise
  key.problem.M = M; key.problem.N = N; key.problem.K = K; key.problem.L = L;
  key.problem.A = A; key.problem.lda = lda; key.problem.layoutA = layoutA;
  key.problem.B = B; key.problem.ldb = ldb; key.problem.layoutB = layoutB;
  key.problem.C = C; key.problem.X = X; key.problem.D = D; key.problem.Y = Y;
  key.problem.alpha = alpha; key.problem.beta = beta; key.problem.x_factor = x_factor;
  key.problem.dtypes.ab = dtypes->ab; key.problem.dtypes.c = dtypes->c;
  key.problem.dtypes.d = dtypes->d; key.problem.dtypes.x = dtypes->x;
  key.problem.dtypes.y = dtypes->y; key.problem.dtypes.cdxy_major = dtypes->cdxy_major;
  key.problem.dtypes.b = dtypes->b; key.problem.dtypes.epilogue = dtypes->epilogue;
  key.problem.dtypes.acc = dtypes->acc;
  key.config_gen = h->config_gen;
  LaunchEntry* ent = nullptr;
  for (LaunchEntry& c : h->cache)
    if (c.valid && std::memcmp(&c.key, &key, sizeof(key)) == 0) { ent = &c; break; }
  if (!ent) {
    LaunchEntry& slot = h->cache[h->cache_next];
    slot.valid = false;
    NvtxRange prep("gemm_run:plan_and_encode");
    st = prepare_launch(h, p, slot);
    if (st != GEMM_OK) return st;
    slot.key = key;
    slot.valid = true;
    h->cache_next = (h->cache_next + 1) % kLaunchCacheEntries;
    ent = &slot;
  }

  cudaLaunchConfig_t lc{};
  cudaLaunchAttribute attr[2];
  lc.gridDim = dim3((unsigned)ent->cfg.grid_ctas);
  lc.blockDim = dim3(gb300::threads_for(ent->cfg.epi_warps));
  lc.dynamicSmemBytes = (size_t)ent->cfg.smem_bytes;
  lc.stream = reinterpret_cast<cudaStream_t>(stream);
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)ent->cluster_ctas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // Programmatic dependent launch: this grid may be scheduled while the
  // previous kernel of the stream finishes; the kernel waits for that kernel
  // (griddepcontrol.wait) before it touches global memory.
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 2;
  ent->kp.status = h->d_status;
  ent->kp.timeout_ns = h->timeout_ns;
  ent->kp.stats = h->d_stats;
  void* args[7] = {&ent->maps[0], &ent->maps[1], &ent->maps[2], &ent->maps[3], &ent->maps[4],
                   &ent->maps[5], &ent->kp};
  if (cudaLaunchKernelExC(&lc, ent->kern, args) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  h->last = ent->cfg;
  return GEMM_OK;
}

GEMM_API gemm_status_t gemm_run_host(gemm_handle_t h, int64_t M, int64_t N, int64_t K,
                                     int64_t L, const void* A, int64_t lda,
                                     gemm_layout_t layoutA, const void* B, int64_t ldb,
                                     gemm_layout_t layoutB, const void* C, const void* X,
                                     void* D, void* Y, float alpha, float beta,
                                     float x_factor, const gemm_dtypes_t* dtypes,
                                     struct CUstream_st* stream) {
  NvtxRange range("gemm_run_host");
  if (!h || !dtypes) return GEMM_ERR_INVALID_ARG;
  gemm_problem_t p{M, N, K, L, A, lda, layoutA, B, ldb, layoutB, C, X, D, Y,
                   alpha, beta, x_factor, *dtypes};
  gemm_status_t st = validate(&p);
  if (st != GEMM_OK) return st;
  if (M == 0 || N == 0 || L == 0) return GEMM_OK;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess || cur != h->device) {
    cudaGetLastError();
    return GEMM_ERR_INVALID_ARG;
  }
  // Element spans, first to last element: an operand with R rows of K (or K
  // rows of R) per batch ends ld - (extent of its contiguous dimension)
  // elements before a whole number of rows.
  const size_t es = (size_t)dtype_bytes(dtypes->ab);
  auto span = [](int64_t rows, int64_t ld, int64_t inner) {
    return rows > 0 ? (size_t)((rows - 1) * ld + inner) : (size_t)0;
  };
  const bool a_mn = layoutA == GEMM_MN_MAJOR, b_mn = layoutB == GEMM_MN_MAJOR;
  const size_t bytes_a = K > 0 ? es * (a_mn ? span(L * K, lda, M) : span(L * M, lda, K)) : 0;
  const size_t bytes_b = K > 0 ? es * (b_mn ? span(L * K, ldb, N) : span(L * N, ldb, K)) : 0;
  const size_t mnl = (size_t)M * (size_t)N * (size_t)L;
  const size_t bytes_c = reads_c(p) ? mnl * dtype_bytes(dtypes->c) : 0;
  const size_t bytes_x = reads_x(p) ? mnl * dtype_bytes(dtypes->x) : 0;
  const size_t bytes_d = mnl * dtype_bytes(dtypes->d);
  const size_t bytes_y = Y ? mnl * dtype_bytes(dtypes->y) : 0;
  auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
  const size_t off_b = up(bytes_a), off_c = off_b + up(bytes_b), off_x = off_c + up(bytes_c);
  const size_t off_d = off_x + up(bytes_x), off_y = off_d + up(bytes_d);
  const size_t need = off_y + up(bytes_y);
  uint8_t* ws;
  {
    std::lock_guard<std::mutex> g(h->ws_mu);
    if (h->ws_bytes < need) {
      // Earlier calls may still be reading or writing the old workspace:
      // let the device drain before it is released (growth is rare).
      if (h->ws && cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
      }
      if (h->ws) cudaFree(h->ws);
      h->ws = nullptr;
      h->ws_bytes = 0;
      if (cudaMalloc(&h->ws, need) != cudaSuccess) {
        cudaGetLastError();
        h->ws = nullptr;
        return GEMM_ERR_CUDA;
      }
      h->ws_bytes = need;
    }
    ws = static_cast<uint8_t*>(h->ws);
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  auto h2d = [&](size_t off, const void* src, size_t n) {
    return n == 0 || cudaMemcpyAsync(ws + off, src, n, cudaMemcpyHostToDevice, s) == cudaSuccess;
  };
  if (!h2d(0, A, bytes_a) || !h2d(off_b, B, bytes_b) || !h2d(off_c, C, bytes_c) ||
      !h2d(off_x, X, bytes_x)) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  st = gemm_run(h, M, N, K, L, K > 0 ? ws : nullptr, lda, layoutA, K > 0 ? ws + off_b : nullptr,
                ldb, layoutB, bytes_c ? ws + off_c : nullptr, bytes_x ? ws + off_x : nullptr,
                ws + off_d, Y ? ws + off_y : nullptr, alpha, beta, x_factor, dtypes, stream);
  if (st != GEMM_OK) return st;
  if (cudaMemcpyAsync(D, ws + off_d, bytes_d, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      (Y && cudaMemcpyAsync(Y, ws + off_y, bytes_y, cudaMemcpyDeviceToHost, s) != cudaSuccess)) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  return GEMM_OK;
}

GEMM_API gemm_status_t gemm_ring_stats(gemm_handle_t h, struct CUstream_st* stream,
                                       uint64_t* out, int max_ctas, int* n_ctas) {
  if (!h || !out || !n_ctas || max_ctas < 0) return GEMM_ERR_INVALID_ARG;
  *n_ctas = 0;
  if (!gb300::kRingStats || !h->d_stats) return GEMM_ERR_UNSUPPORTED_CONFIG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int n = std::min(h->last.grid_ctas, std::min(max_ctas, h->sm_count));
  if (cudaStreamSynchronize(s) != cudaSuccess ||
      (n > 0 && cudaMemcpy(out, h->d_stats, (size_t)n * gb300::kStatWords * sizeof(uint64_t),
                           cudaMemcpyDeviceToHost) != cudaSuccess)) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  *n_ctas = n;
  return GEMM_OK;
}

GEMM_API gemm_status_t gemm_sync_status(gemm_handle_t h, struct CUstream_st* stream,
                                        uint32_t* detail) {
  if (!h) return GEMM_ERR_INVALID_ARG;
  if (detail) *detail = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) { cudaGetLastError(); return GEMM_ERR_CUDA; }
  uint32_t word = 0;
  if (cudaMemcpyAsync(&word, h->d_status, sizeof(word), cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  if (detail) *detail = word;
  if (word != 0) {
    cudaMemsetAsync(h->d_status, 0, sizeof(uint32_t), s);
    // A launch that ended early may leave stream-K flags raised.
    if (h->sk_flags) cudaMemsetAsync(h->sk_flags, 0, (size_t)h->sm_count * sizeof(uint32_t), s);
    cudaStreamSynchronize(s);
    return status_of_word(word);
  }
  return GEMM_OK;
}

// ====================================================================== no-allocation entry point
//
// gemm_run_noalloc: the same GEMM for callers that must not allocate device
// memory.  The only device memory the kernel needs beyond the caller's
// tensors is its 4-byte watchdog status word, which gemm_create obtains with
// cudaMalloc; here it lives in a file-scope __device__ array instead, and the
// per-device state a handle would hold lives in static host storage.

// Scratch of gemm_run_noalloc: 64 words (256 bytes) on every GPU that loads
// this library, kept until the process exits.  A call uses one word (the
// watchdog status), whatever the problem size.
static constexpr int kNoallocScratchWords = 64;
static __device__ __align__(256) uint32_t g_noalloc_scratch[kNoallocScratchWords];

namespace {

constexpr int kNoallocWordsPerCall = 1;
constexpr int kNoallocMaxDevices = 64;

struct NoallocSlot {
  std::mutex mu;
  bool ready = false;
  gemm_handle handle;   // static storage; its d_status points at the scratch
};
NoallocSlot g_noalloc_slots[kNoallocMaxDevices];

// One-time set-up for `device` (which must be current): device checks, the
// tensor-map encoder, resident-cluster counts, and the device address of the
// scratch array.  Nothing is allocated.
gemm_status_t noalloc_setup(gemm_handle& h, int device) {
  int major = 0, minor = 0, sms = 0, optin = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) !=
          cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  if (major != 10 || minor != 3) return GEMM_ERR_UNSUPPORTED_ARCH;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  // The array's name is only a host-side stand-in: the kernel needs the
  // device address, which the runtime resolves for the current device.
  void* scratch = nullptr;
  if (cudaGetSymbolAddress(&scratch, g_noalloc_scratch) != cudaSuccess || !scratch) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  int clusters[9] = {0, 0, 0, 0, 0, 0, 0, 0, 0};
  query_cluster_occupancy(device, sms, optin, clusters);
  for (int i = 0; i < 9; ++i) h.clusters_by_size[i] = clusters[i];
  h.device = device;
  h.sm_count = sms;
  h.smem_optin = optin;
  h.encode = reinterpret_cast<EncodeTiledFn>(fn);
  h.d_status = static_cast<uint32_t*>(scratch);
  return GEMM_OK;
}

}  // namespace

GEMM_API gemm_status_t gemm_run_noalloc(int64_t M, int64_t N, int64_t K, int64_t L,
                                        const void* A, int64_t lda, gemm_layout_t layoutA,
                                        const void* B, int64_t ldb, gemm_layout_t layoutB,
                                        const void* C, const void* X, void* D, void* Y,
                                        float alpha, float beta, float x_factor,
                                        const gemm_dtypes_t* dtypes, struct CUstream_st* stream,
                                        uint32_t* watchdog_out) {
  NvtxRange range("gemm_run_noalloc");
  if (watchdog_out) *watchdog_out = 0;
  // Scratch a call needs against what the array holds (a constant one word).
  if (kNoallocWordsPerCall > kNoallocScratchWords) return GEMM_ERR_INVALID_ARG;
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess) { cudaGetLastError(); return GEMM_ERR_CUDA; }
  if (device < 0 || device >= kNoallocMaxDevices) return GEMM_ERR_INVALID_ARG;
  NoallocSlot& slot = g_noalloc_slots[device];
  {
    std::lock_guard<std::mutex> g(slot.mu);
    if (!slot.ready) {
      const gemm_status_t st = noalloc_setup(slot.handle, device);
      if (st != GEMM_OK) return st;
      slot.ready = true;
    }
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // The status word must read zero when the kernel starts: the array keeps
  // whatever the previous call left in it.
  if (cudaMemsetAsync(slot.handle.d_status, 0, sizeof(uint32_t) * kNoallocWordsPerCall, s) !=
      cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  const gemm_status_t st = gemm_run(&slot.handle, M, N, K, L, A, lda, layoutA, B, ldb, layoutB,
                                    C, X, D, Y, alpha, beta, x_factor, dtypes, stream);
  if (st != GEMM_OK || !watchdog_out) return st;
  // Read back on the caller's stream only (a plain cudaMemcpy would also wait
  // on every other blocking stream of the device).
  uint32_t word = 0;
  if (cudaMemcpyAsync(&word, slot.handle.d_status, sizeof(word), cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  *watchdog_out = word;
  return status_of_word(word);
}
