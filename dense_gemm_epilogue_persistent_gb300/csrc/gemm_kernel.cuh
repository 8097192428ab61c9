// Persistent, warp-specialised batched GEMM with a fused epilogue for sm_103a.
//
//   Y = A*B,   D = alpha*(A*B) + beta*C + x_factor*X
//   (fp32 accumulation, or fp16 for fp16/fp8 inputs; fp32 epilogue; optional relu
//   of alpha*(A*B) + beta*C before X is added)
//
// What the kernel computes and its warp roles follow "custom_epilogue_dense_gemm.py"
// (CuTeDSL Blackwell example), module docstring "This GEMM works as follows" (DMA
// warp; MMA warp; EPILOGUE warps that tcgen05.ld the accumulator, TMA-load C and X
// through shared memory, compute Y and D, and TMA-store D and Y; persistent tile
// scheduling) and the 2-SM tcgen05 scheme of "04_mma_tma_2sm_sm100.cu" (CuTe
// Blackwell tutorial 04, "Step 2: The Mainloop": the leader CTA issues the pair's
// MMA; tensor-memory allocation and MMA-completion arrivals reach both CTAs).  The
// thread roles (128 epilogue threads + one MMA warp + one TMA warp = 192 threads,
// one CTA per SM, the whole 512-column tensor memory split into accumulator stages)
// follow the cuBLASDx "API Card: Blackwell Pipeline (tcgen05)", host-side and
// "Depth and shared memory" bullets.
//
// Block = 6 warps (10 with EPW = 2):
//   warp 0      TMA producer: one lane streams A and B k-blocks into a ring of
//               `stages` shared-memory slots, each guarded by full/empty mbarriers.
//   warp 1      tensor-memory allocator + MMA issuer: one lane of the leader CTA
//               issues tcgen05.mma into one of two accumulator stages in tensor
//               memory, frees ring slots with tcgen05.commit, and hands finished
//               accumulators to the epilogue with another commit.
//   warps 2..   epilogue: warp w owns TMEM lanes 32*(w%4)..+31 (= 32 tile rows)
//               and runs its own pipeline over them, in 32-column chunks through
//               its share of the `slots` shared-memory slots: its lane 0
//               TMA-loads the C and X sub-tiles ahead (across tile boundaries, so
//               the next tile's C/X arrive during its main loop); each lane
//               requests its accumulator columns, reads its C/X row while they
//               load, computes in fp32 and writes D and Y back into the sub-slot,
//               and lane 0 TMA-stores them.  With EPW = 2 two warps own each
//               lane quarter and take its chunks alternately, so the per-chunk
//               latency chain (accumulator load, shared-memory traffic, store
//               issue) of one warp overlaps the other's.
// Every cluster walks the same static persistent tile sequence
// t = cluster_id, cluster_id + num_clusters, ...; with two accumulator stages the
// epilogue of tile i overlaps the main loop of tile i+1.  Tiles are ordered in
// strips of group_m tile rows, odd strips walking N backwards, and odd waves of
// tiles walk K downwards (fp32 accumulators), so each wave starts on the operand
// blocks the previous one read last, while they are still in L2.  The kernel touches
// global memory only after griddepcontrol.wait, so a launch with programmatic
// stream serialization overlaps its prologue with the previous grid's tail.
//
// Clusters: CG*MC*NC CTAs = MC x NC CTA groups (pairs when CG = 2), MC stacked
// along M and NC side by side along N.  Groups in one column of the cluster
// compute vertically adjacent tiles with the same B columns, so each CTA
// loads only 1/MC of its B slice and TMA-multicasts it to the matching CTA of
// every group in that column; groups in one row share A rows the same way
// (1/NC of the A slice each, multicast along the row).  This is the multicast
// pattern of "04_mma_tma_2sm_sm100.cu", "TMA Setup": B multicast along cluster
// M, A along cluster N.  A ring slot may then be refilled only after every
// group's MMA has drained it, so MMA completion is multicast to all CTAs of
// the cluster.  The multicast loads themselves live in ptx_multicast.cuh,
// which only the units instantiating such clusters include.
//
// The tile width BN (a multiple of 32 up to 256) is a launch parameter; the
// two accumulator stages sit 256 tensor-memory columns apart whatever BN is.
//
// Every barrier wait is bounded (watchdog): on expiry the kernel records a code
// in a device status word, raises a CTA-wide abort flag, lets in-flight copies
// drain, frees its tensor memory and returns.  Epilogue decisions that follow a
// wait are made uniform across the 128 epilogue threads with bar.red.and, so no
// thread is ever left alone at a named barrier.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace gb300 {

enum : int { DT_F32 = 0, DT_F16 = 1, DT_BF16 = 2, DT_E4M3 = 3 };

struct EpiParams {
  int c_dt, d_dt, x_dt, y_dt;
  int cd_m_major;            // 0: (l*M + m)*N + n   1: (l*N + n)*M + m
  int read_c, read_x, write_y;
  float alpha, beta, x_factor;
  int relu;                  // D = max(alpha*acc + beta*C, 0) + x_factor*X
  int acc_f16;               // accumulator is fp16: one per 32-bit TMEM column, low half
  int slots;                 // epilogue shared-memory slots (>= 2)
  uint32_t cd_bytes;         // bytes of a slot's C/D region
  uint32_t xy_bytes;         // bytes of a slot's X/Y region (0: neither X nor Y)
};

struct KernelParams {
  int M, N, K, L;
  int bn;                    // tile width of one CTA group (multiple of 32, <= 256)
  int tiles_m, tiles_n;      // cluster tiles per batch along M (128*CG*MC rows) and N (BN*NC)
  int num_tiles;             // tiles_m * tiles_n * L
  int k_blocks;              // ceil(K / tile_k)
  int group_m;               // rasterisation strip height (tiles)
  int stages;                // A/B ring depth
  int a_mn_major, b_mn_major;
  uint32_t idesc;            // tcgen05 instruction descriptor
  int split_start;           // tiles from here on run as two half-width items (num_tiles: none)
  int num_items;             // split_start + 2 * (num_tiles - split_start)
  uint32_t idesc_half;       // instruction descriptor of a half-width item (N / 2)
  uint32_t epi_wait_ns;      // suspend-time hint of the epilogue's accumulator wait (0: none)
  int inject_stall;          // test only: the MMA warp first waits on a barrier nobody arrives at
  int k_alternate;           // odd waves of tiles walk K from the last k-block down
  uint32_t l2_hints;         // L2 eviction priority (0 normal, 1 last, 2 first):
                             //   bits 0-1 A/B loads, 2-3 C/X loads, 4-5 D/Y stores
  uint32_t* status;          // device status word (watchdog)
  unsigned long long timeout_ns;
  unsigned long long* stats; // ring statistics (statistics build only; else unused)
  // Stream-K (tiles fewer than resident clusters): sk_units clusters split the
  // sk_iters = num_tiles * k_blocks k-blocks of all tiles into equal contiguous
  // ranges; a tile's k-blocks held by several clusters are summed in fp32
  // through sk_partials (one 128 x bn slot per CTA) and sk_flags.  0: off.
  int sk_units;
  long long sk_iters;
  float* sk_partials;
  uint32_t* sk_flags;
  EpiParams epi;
};

// Ring statistics: a separate build of the library (GB300_RING_STATS=1) in
// which each CTA's producer, MMA issuer and epilogue store thread count the
// clock cycles they spend waiting on each barrier and in their loops, so the
// ring's stall picture can be read per role.  The product build compiles none
// of it.  Per CTA kStatWords counters, in the order of the enum.
#ifndef GB300_RING_STATS
#define GB300_RING_STATS 0
#endif
constexpr bool kRingStats = GB300_RING_STATS != 0;
enum : int {
  kStatMmaFull = 0,     // MMA issuer: cycles waiting for a stage to land
  kStatMmaAcc,          //   ... waiting for a free accumulator stage
  kStatMmaLoop,         //   ... in its whole loop
  kStatMmaStages,       //   stages issued
  kStatProdEmpty,       // producer: cycles waiting for a stage to drain
  kStatProdLoop,        //   ... in its whole loop
  kStatEpiTfull,        // epilogue store thread: cycles waiting for an accumulator
  kStatEpiCfull,        //   ... waiting for C/X to land
  kStatEpiLoop,         //   ... in its whole loop
  kStatEpiChunks,       //   chunks the CTA processed (all epilogue warps of a lane quarter)
  kStatEpiRead,         //   ... from C/X landing to C/X read and accumulator columns in registers
  kStatEpiMath,         //   ... computing D and Y and writing them to shared memory
  kStatEpiIssue,        //   ... issuing the stores (and the next loads, with their wait)
  kStatEpiOwnChunks,    //   chunks the recording warp processed (the three above are its own)
  kStatWords = 16
};

__device__ __forceinline__ long long stat_clock() {
  if constexpr (kRingStats) return clock64();
  else return 0;
}

// Threads of a CTA: the TMA warp, the MMA warp and four (or eight, with two
// epilogue warps per tensor-memory lane quarter) epilogue warps.
constexpr int threads_for(int epi_warps_per_quarter) { return 64 + 128 * epi_warps_per_quarter; }
constexpr int kThreads = threads_for(1);
constexpr int kAccStages = 2;
constexpr uint32_t kTmemCols = 512;
constexpr int kEpiChunk = 32;          // columns per epilogue chunk
constexpr int kEpiLeader = 64;         // epilogue thread that records the ring statistics
constexpr int kSubRows = 32;           // rows of one epilogue warp's sub-tiles
constexpr int kMaxChunks = 8;          // 32-column epilogue chunks of the widest tile
constexpr int kMaxEpiWarps = 8;        // epilogue warps of the largest CTA

constexpr uint32_t kAccStride = 256;   // tensor-memory columns between accumulator stages

template <int CG, int AB_BYTES, int KA, int MC, int NC>
struct Geometry {
  static constexpr int BM = 128;                 // A rows staged per CTA
  static constexpr int ATOM_K = 128 / AB_BYTES;  // K of one 128-byte swizzle row
  static constexpr int BK = ATOM_K * KA;         // K per ring stage (KA 128-byte K atoms)
  static constexpr int A_ATOM = BM * 128;        // bytes of one K-major A atom (128 rows)
  static constexpr int A_STAGE = A_ATOM * KA;    // bytes
  static constexpr int UMMA_K = 32 / AB_BYTES;   // K per tcgen05.mma (32 bytes: 8 tf32,
                                                 // 16 fp16/bf16, 32 fp8)
  static constexpr int K_STEPS = BK / UMMA_K;    // instructions per stage
  static constexpr int STEPS_PER_ATOM = ATOM_K / UMMA_K;   // 4
  static constexpr int ATOM_MN = 128 / AB_BYTES; // MN extent of one MN-major swizzle atom
  static constexpr int ATOM_BYTES = BK * 128;    // bytes of one MN-major atom column
  static constexpr int GROUPS = MC * NC;         // CTA groups per cluster
  static constexpr int CLUSTER = CG * GROUPS;    // CTAs per cluster
  static constexpr int CM = BM * CG * MC;        // output rows per cluster tile
  static constexpr int A_PART = BM / NC;         // A rows each CTA loads (and multicasts)
  static_assert(KA == 1 || KA == 2, "k atoms per stage");
  static_assert(CLUSTER <= 8, "portable cluster size");
  static_assert(kAccStages * kAccStride <= kTmemCols, "accumulators must fit tensor memory");
};

// The B-side sizes that follow from the runtime tile width.
struct TileN {
  int bn;        // output columns of one CTA group's tile
  int bn_cta;    // B rows staged per CTA (bn / CG)
  int bn_part;   // B rows each CTA loads (and multicasts): bn_cta / MC
  int b_atom;    // bytes of one K-major B atom (bn_cta rows of 128 bytes)
  int b_stage;   // bytes of B per ring stage
  int chunks;    // 32-column epilogue chunks per whole tile
};

// Watchdog codes: 0xE0RRBBBB, RR = role, BBBB = low 16 bits of blockIdx.x.
enum : uint32_t {
  kWaitProducer = 1, kWaitMmaFull = 2, kWaitMmaAcc = 3, kWaitEpilogue = 4, kWaitEpiLoad = 5,
  kWaitInjected = 6, kWaitPartial = 7
};

struct Watch {
  volatile uint32_t* abort;
  uint32_t* status;
  unsigned long long timeout_ns;
};

// Debug build (GB300_DEBUG=1, a separate library): before use, every TMA
// copy's shared-memory range and inner coordinate (16-byte aligned, stores not
// below zero), every tensor-memory column range the MMA writes or the
// epilogue reads, and every MMA operand address are checked.  A failed check
// records 0xD0CCBBBB (CC the check, BBBB the low 16 bits of the block) in the
// status word, raises the abort flag and skips the access, so the launch ends
// through the watchdog's drain path; nothing traps.  The product build
// compiles none of it.
#ifndef GB300_DEBUG
#define GB300_DEBUG 0
#endif
constexpr bool kDebug = GB300_DEBUG != 0;
enum : uint32_t {
  kChkLoadA = 1, kChkLoadB = 2, kChkMmaTmem = 3, kChkMmaSmem = 4, kChkEpiTmem = 5,
  kChkEpiSmem = 6, kChkEpiLoad = 7, kChkEpiStore = 8
};

__device__ __forceinline__ bool dbg_check(bool cond, uint32_t check, const Watch& w) {
  if constexpr (!kDebug) {
    (void)cond; (void)check; (void)w;
    return true;
  } else {
    if (cond) return true;
    *w.abort = 1u;
    atomicCAS(w.status, 0u, 0xD0000000u | (check << 16) | (blockIdx.x & 0xFFFFu));
    return false;
  }
}

// [lo, lo + bytes) lies inside [begin, end).
__device__ __forceinline__ bool in_range(uint32_t lo, uint32_t bytes, uint32_t begin,
                                         uint32_t end) {
  return lo >= begin && lo + bytes <= end;
}

// Bounded wait for the phase with parity `parity`.  A non-zero `hint_ns` lets
// the hardware suspend the thread up to that long per probe (for long waits
// whose spinning would take issue slots from the TMA and MMA warps).
// kLocal: a barrier only this CTA's own TMA loads complete (CTA-scope acquire).
template <bool kLocal = false>
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const Watch& w,
                                           uint32_t role, uint32_t hint_ns = 0) {
  auto probe = [&]() {
    if constexpr (kLocal) return mbar_try_wait_cta(bar, parity);
    else return hint_ns ? mbar_try_wait_hint(bar, parity, hint_ns) : mbar_try_wait(bar, parity);
  };
  if (kLocal ? mbar_try_wait_cta(bar, parity) : mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (probe()) return true;
    if (*w.abort) return false;
    if (globaltimer_ns() - t0 > w.timeout_ns) {
      *w.abort = 1u;
      atomicCAS(w.status, 0u, 0xE0000000u | (role << 16) | (blockIdx.x & 0xFFFFu));
      return false;
    }
  }
}

// Linear tile id -> (m tile, n tile, batch).  Tiles are walked in strips of
// `group_m` M-tiles so that concurrently resident tiles share A and B rows in L2.
__device__ __forceinline__ void tile_coords(int t, const KernelParams& p, int& tm, int& tn,
                                            int& tl) {
  const int per_batch = p.tiles_m * p.tiles_n;
  tl = t / per_batch;
  const int r = t - tl * per_batch;
  const int span = p.group_m * p.tiles_n;
  const int g = r / span;
  const int first_m = g * p.group_m;
  const int gm = min(p.tiles_m - first_m, p.group_m);
  const int rr = r - g * span;
  tm = first_m + rr % gm;
  tn = rr / gm;
  if (g & 1) tn = p.tiles_n - 1 - tn;   // odd strips walk N backwards (serpentine)
}

// Work item -> tile and half.  Items below split_start are whole tiles; the
// rest are the two half-width (tile_n / 2) halves of the last tiles, so that
// the final, partial wave of tiles runs as a wave of half tiles.  half = -1
// for a whole tile, else 0 or 1.
__device__ __forceinline__ int item_tile(int it, const KernelParams& p, int& half) {
  if (it < p.split_start) {
    half = -1;
    return it;
  }
  const int r = it - p.split_start;
  half = r & 1;
  return p.split_start + (r >> 1);
}

// One work item of a cluster: k-blocks [kb0, kb1) of tile `tile` (half as in
// item_tile).  owner: the item ends at the tile's last k-block, so its
// epilogue writes the tile; otherwise (stream-K only) it publishes a partial
// sum.  empty: no work (stream-K only: a cluster whose range is one segment
// has nothing at its second item position).  Without stream-K, K = 0 gives
// items of no k-block whose epilogue still writes D = beta C + x_factor X.
struct Work {
  int tile, half, kb0, kb1;
  bool owner, empty;
};

// Stream-K: the cluster whose range holds k-block i of the flattened
// (tile, k-block) space, ranges [u T / U, (u + 1) T / U).
__device__ __forceinline__ int sk_unit_of(long long i, const KernelParams& p) {
  return (int)(((i + 1) * p.sk_units - 1) / p.sk_iters);
}

// Item `it` of the static walk (it = cluster + n * clusters).  Without stream-K
// every item is a whole tile (or half tile) over all k-blocks.  With stream-K
// each cluster has two item positions: a range that crosses a tile boundary is
// the tail of tile t0 (which it owns) and the head of tile t0 + 1 (a partial
// for that tile's owner); the head comes first, so that its partial is
// published while the owned tail is computed, and no cluster ever waits for a
// partial that is computed after a wait of its own.
template <bool kSK>
__device__ __forceinline__ Work work_item(int it, const KernelParams& p, int num_clusters) {
  Work w;
  if (!kSK || !p.sk_units) {
    w.tile = item_tile(it, p, w.half);
    w.kb0 = 0;
    w.kb1 = p.k_blocks;
    w.owner = true;
    w.empty = false;
    return w;
  }
  w.half = -1;
  const int u = it % num_clusters, pos = it / num_clusters;
  const long long T = p.sk_iters, U = p.sk_units, kb = p.k_blocks;
  const long long b = u * T / U, e = (u + 1) * T / U;
  const long long t0 = b / kb, t1 = (e - 1) / kb;
  w.tile = 0;
  w.kb0 = w.kb1 = 0;
  w.owner = false;
  w.empty = true;
  if (u >= U || pos > 1 || b >= e) return w;     // (the grid has exactly U clusters)
  w.empty = false;
  if (t0 == t1) {
    if (pos != 0) {
      w.empty = true;
      return w;
    }
    w.tile = (int)t0;
    w.kb0 = (int)(b - t0 * kb);
    w.kb1 = (int)(e - t0 * kb);
    w.owner = e == (t0 + 1) * kb;
  } else if (pos == 0) {                  // head of tile t1: a partial
    w.tile = (int)t1;
    w.kb1 = (int)(e - t1 * kb);
  } else {                                // tail of tile t0: owned
    w.tile = (int)t0;
    w.kb0 = (int)(b - t0 * kb);
    w.kb1 = (int)kb;
    w.owner = true;
  }
  return w;
}

// ------------------------------------------------------------------ epilogue smem

// Two fp32 values -> one 32-bit word of two 16-bit values (first in the low
// half), rounded to nearest even.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ float2 unpack_f16x2(uint32_t w) {
  return __half22float2(*reinterpret_cast<const __half2*>(&w));
}
__device__ __forceinline__ float2 unpack_bf16x2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// Epilogue sub-tiles hold one warp's 32 rows x 32 columns of one tensor, as TMA
// lays them out:
//   row-major tensors: [row][32 columns], 128-byte rows (fp32, 128-byte swizzle:
//     16-byte chunk j of row r sits at chunk j ^ (r & 7)) or 64-byte rows (16-bit,
//     64-byte swizzle: chunk j ^ ((r >> 1) & 3));
//   column-major tensors: [column][32 rows], unswizzled.
// Lane r touches only row r; the swizzles make each 8-row group of a warp hit
// distinct banks.  The type and layout branches are uniform and sit outside the
// element loops, and 16-bit values convert two at a time.
// Calls f(i, value) for the 32 values of row r, in pieces as they are loaded,
// so that a caller folding them into another array keeps only a few of them
// in registers at a time.
template <bool BF16, typename F>
__device__ __forceinline__ void smem_row_each_16(const uint8_t* sub, int m_major, int r, F&& f) {
  auto unpack = [](uint32_t w) { return BF16 ? unpack_bf16x2(w) : unpack_f16x2(w); };
  if (!m_major) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 q = *reinterpret_cast<const uint4*>(sub + r * 64 + ((j ^ ((r >> 1) & 3)) << 4));
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 v = unpack(w[k]);
        f(8 * j + 2 * k, v.x);
        f(8 * j + 2 * k + 1, v.y);
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t lo = *reinterpret_cast<const uint16_t*>(sub + (2 * i * kSubRows + r) * 2);
      const uint32_t hi = *reinterpret_cast<const uint16_t*>(sub + ((2 * i + 1) * kSubRows + r) * 2);
      const float2 v = unpack(lo | (hi << 16));
      f(2 * i, v.x);
      f(2 * i + 1, v.y);
    }
  }
}

// Calls f(i, value) for the 32 values of row r, in pieces as they are loaded,
// so that a caller folding them into another array keeps only a few of them
// in registers at a time.
template <typename F>
__device__ __forceinline__ void smem_row_each(const uint8_t* sub, int dt, int m_major, int r,
                                              F&& f) {
  if (dt == DT_BF16) {
    smem_row_each_16<true>(sub, m_major, r, f);
  } else if (dt != DT_F32) {
    smem_row_each_16<false>(sub, m_major, r, f);
  } else if (!m_major) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float4 q = *reinterpret_cast<const float4*>(sub + r * 128 + ((j ^ (r & 7)) << 4));
      f(4 * j, q.x);
      f(4 * j + 1, q.y);
      f(4 * j + 2, q.z);
      f(4 * j + 3, q.w);
    }
  } else {
#pragma unroll
    for (int c = 0; c < kEpiChunk; ++c)
      f(c, *reinterpret_cast<const float*>(sub + (c * kSubRows + r) * 4));
  }
}

__device__ __forceinline__ void smem_read_row(const uint8_t* sub, int dt, int m_major, int r,
                                              float (&v)[kEpiChunk]) {
  smem_row_each(sub, dt, m_major, r, [&](int i, float x) { v[i] = x; });
}

__device__ __forceinline__ void smem_write_row(uint8_t* sub, int dt, int m_major, int r,
                                               const float (&v)[kEpiChunk]) {
  if (dt == DT_F32) {
    if (!m_major) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        *reinterpret_cast<float4*>(sub + r * 128 + ((j ^ (r & 7)) << 4)) =
            make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    } else {
#pragma unroll
      for (int c = 0; c < kEpiChunk; ++c) *reinterpret_cast<float*>(sub + (c * kSubRows + r) * 4) = v[c];
    }
    return;
  }
  uint32_t w[16];
  if (dt == DT_BF16) {
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = pack_f16x2(v[2 * i], v[2 * i + 1]);
  }
  if (!m_major) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      *reinterpret_cast<uint4*>(sub + r * 64 + ((j ^ ((r >> 1) & 3)) << 4)) =
          make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      *reinterpret_cast<uint16_t*>(sub + (2 * i * kSubRows + r) * 2) = (uint16_t)(w[i] & 0xFFFFu);
      *reinterpret_cast<uint16_t*>(sub + ((2 * i + 1) * kSubRows + r) * 2) = (uint16_t)(w[i] >> 16);
    }
  }
}

// Bytes of one warp's sub-tile of a tensor of type dt.
__device__ __forceinline__ uint32_t sub_bytes(int dt) {
  return (uint32_t)(kSubRows * kEpiChunk) * (dt == DT_F32 ? 4u : 2u);
}

// ------------------------------------------------------------------ the kernel

template <int CG, int AB_BYTES, int KA, int MC, int NC, int EPW, int SK>
__global__ void __launch_bounds__(threads_for(EPW), 1)
persistent_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmC,
                       const __grid_constant__ CUtensorMap tmX,
                       const __grid_constant__ CUtensorMap tmD,
                       const __grid_constant__ CUtensorMap tmY,
                       const __grid_constant__ KernelParams p) {
  using G = Geometry<CG, AB_BYTES, KA, MC, NC>;
  constexpr int KIND = (AB_BYTES == 1) ? 1 : (AB_BYTES == 4 ? 2 : 0);
  constexpr bool MULTI = G::CLUSTER > 1;
  const int BN = p.bn;
  TileN tn_geo;
  tn_geo.bn = BN;
  tn_geo.bn_cta = BN / CG;
  tn_geo.bn_part = tn_geo.bn_cta / MC;
  tn_geo.b_atom = tn_geo.bn_cta * 128;
  tn_geo.b_stage = tn_geo.b_atom * KA;
  tn_geo.chunks = BN / kEpiChunk;
  const TileN& T = tn_geo;
  // Stream-K items (a separate instantiation, so that the other kernels carry
  // none of its code).
  constexpr bool kSK = SK != 0;

  // The next GEMM of the stream may start its prologue on SMs this grid leaves
  // idle; it touches global memory only after its own dependency wait below.
  grid_launch_dependents();

  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the swizzle atoms (identical in both CTAs of a pair:
  // same kernel, same layout).
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t crank = MULTI ? cluster_ctarank() : 0u;
  const uint32_t rank = crank % CG;               // CTA within its pair
  const uint32_t grp = crank / CG;                // group within the cluster: gn * MC + gm
  const uint32_t gm = grp % MC;                   // the group's row in the cluster (along M)
  const uint32_t gn = grp / MC;                   // ... and column (along N)
  const uint32_t pair_leader = grp * CG;          // cluster rank of the pair's leader
  const int cluster_id = blockIdx.x / G::CLUSTER;
  const int num_clusters = gridDim.x / G::CLUSTER;
  // CTAs receiving this CTA's B part: the same peer position in every group of
  // its cluster column; its A part: the same position in every group of its row.
  uint16_t b_mask = 0, a_mask = 0;
#pragma unroll
  for (int g = 0; g < MC; ++g) b_mask |= (uint16_t)(1u << ((gn * MC + g) * CG + rank));
#pragma unroll
  for (int g = 0; g < NC; ++g) a_mask |= (uint16_t)(1u << ((g * MC + gm) * CG + rank));
  const uint16_t all_mask = (uint16_t)((1u << G::CLUSTER) - 1u);
  const uint16_t pair_mask = (uint16_t)(((1u << CG) - 1u) << pair_leader);
  const int S = p.stages;
  const EpiParams& e = p.epi;
  const int E = e.slots;
  const uint32_t slot_bytes = e.cd_bytes + e.xy_bytes;

  // [B ring][A ring][epilogue slots][full x S][empty x S][tfull x 2][tempty x 2]
  // [cfull x 4E (per epilogue warp and slot)][tmem address][abort flag][never]
  // [rfull x 8 x 8 (per epilogue warp and chunk)][pdone][pread]  ("never": a
  // barrier nothing arrives at, waited on only when a stall is injected to
  // test the watchdog)
  const uint32_t b_ring = base;
  const uint32_t a_ring = b_ring + S * T.b_stage;
  const uint32_t epi0 = a_ring + S * G::A_STAGE;
  const uint32_t bars = epi0 + E * slot_bytes;
  const uint32_t full0 = bars, empty0 = bars + 8u * S;
  const uint32_t tfull0 = bars + 16u * S, tempty0 = tfull0 + 16u;
  const uint32_t cfull0 = tempty0 + 16u;
  const uint32_t holder = cfull0 + 8u * 4u * E;     // a cfull barrier per warp and slot
  volatile uint32_t* const holder_ptr = reinterpret_cast<volatile uint32_t*>(gbase + (holder - base));
  volatile uint32_t* const abort_ptr = holder_ptr + 1;
  const uint32_t never_bar = holder + 8u;
  // a ring-batch barrier per epilogue warp and chunk of a tile
  const uint32_t rfull0 = never_bar + 8u;
  // stream-K: every epilogue warp has stored its partial rows (pdone) / read
  // the partials it adds (pread)
  const uint32_t pdone = rfull0 + 8u * (uint32_t)(kMaxEpiWarps * kMaxChunks);
  const uint32_t pread = pdone + 8u;
  const uint32_t ring_bytes = (uint32_t)S * ((uint32_t)G::A_STAGE + (uint32_t)T.b_stage);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8u * s, 1);
      mbar_init(empty0 + 8u * s, G::GROUPS);   // one MMA commit per group
    }
    for (int a = 0; a < kAccStages; ++a) {
      mbar_init(tfull0 + 8u * a, 1);
      mbar_init(tempty0 + 8u * a, 4 * EPW * CG);   // every epilogue warp of the CTA (pair)
    }
    for (int s = 0; s < 4 * E; ++s) mbar_init(cfull0 + 8u * s, 1);
    mbar_init(never_bar, 1);
    for (int q = 0; q < kMaxEpiWarps * kMaxChunks; ++q) mbar_init(rfull0 + 8u * q, 1);
    if constexpr (kSK) {
      mbar_init(pdone, 4 * EPW);
      mbar_init(pread, 4 * EPW);
    }
    *abort_ptr = 0u;
    fence_barrier_init();
    if (p.k_blocks > 0) {                    // A and B are encoded only when K > 0
      prefetch_tensormap(&tmA);
      prefetch_tensormap(&tmB);
    }
    prefetch_tensormap(&tmD);
    if (p.epi.write_y) prefetch_tensormap(&tmY);
    if (p.epi.read_c) prefetch_tensormap(&tmC);
    if (p.epi.read_x) prefetch_tensormap(&tmX);
  }
  if (warp == 1) {
    tmem_alloc<CG>(holder, kTmemCols);
    tmem_relinquish<CG>();
  }
  tc_fence_before_sync();
  __syncthreads();
  if constexpr (MULTI) cluster_sync_all();
  tc_fence_after_sync();
  const uint32_t tmem_base = *holder_ptr;
  // Everything above touched only this CTA's shared and tensor memory and the
  // kernel parameters.  From here on global memory is read and written: wait
  // for the previous grid of the stream (programmatic dependent launch).
  grid_dependency_wait();

  const Watch w{abort_ptr, p.status, p.timeout_ns};

  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      const uint64_t pol = make_l2_policy(p.l2_hints & 3u);
      const uint32_t tx_bytes = (uint32_t)(CG * (G::A_STAGE + T.b_stage));
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      long long st_empty = 0;
      const long long st_t0 = stat_clock();
      for (int it = cluster_id; ok && it < p.num_items; it += num_clusters) {
        const Work wk = work_item<kSK>(it, p, num_clusters);
        if (wk.empty) continue;
        const int half = wk.half;
        int tm, tn, tl;
        tile_coords(wk.tile, p, tm, tn, tl);
        // A half-width item covers columns [half * BN/2, +BN/2) of its tile: its
        // CTAs load full B boxes from that origin and the MMA reads their first
        // half.  m0: this CTA's 128 A rows; n0: the first of its B rows, plus
        // the offset of the part it loads for its cluster column.
        const int item_n = half < 0 ? BN : BN / 2;
        const int m0 = tm * G::CM + (int)gm * (G::BM * CG) + (int)rank * G::BM;
        const int n0 = tn * (BN * NC) + (int)gn * BN + (half > 0 ? BN / 2 : 0) +
                       (int)rank * (item_n / CG) + (int)gm * (item_n / CG / MC);
        // Alternate waves walk K in opposite directions, so the k-blocks one
        // wave reads last are the first the next wave reads, while they are
        // still in L2.  The MMA side only counts stages, so the order is the
        // producer's alone.
        const bool k_down = p.k_alternate && ((it / num_clusters) & 1);
        for (int kb = wk.kb0; kb < wk.kb1; ++kb) {
          const long long t_w = stat_clock();
          if (!wait_phase(empty0 + 8u * s, ph ^ 1u, w, kWaitProducer)) { ok = false; break; }
          if constexpr (kRingStats) st_empty += clock64() - t_w;
          const uint32_t fb = full0 + 8u * s;
          if (rank == 0) mbar_arrive_expect_tx(fb, tx_bytes);
          const uint32_t fb_target = (CG == 2) ? map_to_rank(fb, pair_leader) : fb;
          const int k0 = (k_down ? p.k_blocks - 1 - kb : kb) * G::BK;
          const uint32_t sa = a_ring + s * G::A_STAGE;
          const uint32_t sb = b_ring + s * T.b_stage;
          // (debug build: the box's bytes inside this stage, the inner
          // coordinate a whole 16 bytes)
          auto issue_a = [&](uint32_t dst, int c0, int c1, uint32_t bytes) {
            if (!dbg_check(in_range(dst, bytes, sa, sa + G::A_STAGE) &&
                               ((long long)c0 * AB_BYTES) % 16 == 0 && c1 >= 0,
                           kChkLoadA, w)) { ok = false; return; }
            OperandLoad<CG, (NC > 1)>::load(dst, &tmA, fb_target, c0, c1, tl, a_mask, pol);
          };
          auto issue_b = [&](uint32_t dst, int c0, int c1, uint32_t bytes) {
            if (!dbg_check(in_range(dst, bytes, sb, sb + (uint32_t)T.b_stage) &&
                               ((long long)c0 * AB_BYTES) % 16 == 0 && c1 >= 0,
                           kChkLoadB, w)) { ok = false; return; }
            OperandLoad<CG, (MC > 1)>::load(dst, &tmB, fb_target, c0, c1, tl, b_mask, pol);
          };
          if (!p.a_mn_major) {
            // boxes {ATOM_K, A_PART}: this CTA's part of its cluster row's A rows
#pragma unroll
            for (int a = 0; a < KA; ++a)
              issue_a(sa + a * G::A_ATOM + gn * G::A_PART * 128, k0 + a * G::ATOM_K,
                      m0 + (int)gn * G::A_PART, G::A_PART * 128);
          } else {
            // boxes {ATOM_MN, BK}: this CTA's share of the A rows' MN atoms
            constexpr int PER = G::BM / G::ATOM_MN / NC;
#pragma unroll
            for (int j = 0; j < PER; ++j) {
              const int aj = (int)gn * PER + j;
              issue_a(sa + aj * G::ATOM_BYTES, m0 + aj * G::ATOM_MN, k0, G::ATOM_BYTES);
            }
          }
          if (!p.b_mn_major) {
            // boxes {ATOM_K, bn_part}
#pragma unroll
            for (int a = 0; a < KA; ++a)
              issue_b(sb + a * T.b_atom + gm * T.bn_part * 128, k0 + a * G::ATOM_K, n0,
                      (uint32_t)T.bn_part * 128u);
          } else {
            const int atoms = T.bn_part / G::ATOM_MN;          // boxes {ATOM_MN, BK}
            for (int j = 0; j < atoms; ++j)
              issue_b(sb + ((int)gm * atoms + j) * G::ATOM_BYTES, n0 + j * G::ATOM_MN, k0,
                      G::ATOM_BYTES);
          }
          if (kDebug && !ok) break;
          if (++s == S) { s = 0; ph ^= 1u; }
        }
      }
      if constexpr (kRingStats) if (p.stats) {
        unsigned long long* const o = p.stats + (size_t)blockIdx.x * kStatWords;
        o[kStatProdEmpty] = st_empty;
        o[kStatProdLoop] = clock64() - st_t0;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (rank == 0 && lane == 0) {
      int s = 0, acc = 0;
      uint32_t ph = 0, aph = 0;
      long long st_full = 0, st_acc = 0, st_stages = 0;
      const long long st_t0 = stat_clock();
      bool ok = !p.inject_stall || wait_phase(never_bar, 0u, w, kWaitInjected);
      for (int it = cluster_id; ok && it < p.num_items; it += num_clusters) {
        const Work wk = work_item<kSK>(it, p, num_clusters);
        if (wk.empty) continue;
        const long long t_a = stat_clock();
        if (!wait_phase(tempty0 + 8u * acc, aph ^ 1u, w, kWaitMmaAcc)) break;
        if constexpr (kRingStats) st_acc += clock64() - t_a;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + (uint32_t)acc * kAccStride;
        const uint32_t idesc = wk.half < 0 ? p.idesc : p.idesc_half;
        // (debug build: the item's accumulator columns inside its stage)
        if (!dbg_check((uint32_t)(wk.half < 0 ? BN : BN / 2) <= kAccStride &&
                           (uint32_t)acc * kAccStride + kAccStride <= kTmemCols,
                       kChkMmaTmem, w))
          break;
        for (int kb = wk.kb0; kb < wk.kb1; ++kb) {
          const long long t_f = stat_clock();
          if (!wait_phase(full0 + 8u * s, ph, w, kWaitMmaFull)) { ok = false; break; }
          if constexpr (kRingStats) { st_full += clock64() - t_f; ++st_stages; }
          tc_fence_after_sync();
          const uint32_t sa = a_ring + s * G::A_STAGE;
          const uint32_t sb = b_ring + s * T.b_stage;
#pragma unroll
          for (int k = 0; k < G::K_STEPS; ++k) {
            // K-major: atoms of rows x 128 bytes, 8-row groups 1024 bytes
            // apart; step k selects atom k / STEPS_PER_ATOM and moves 32 bytes
            // along its swizzled rows.  MN-major: K rows of 128 bytes, 8-row
            // groups 1024 apart, MN atoms ATOM_BYTES apart; step k moves
            // UMMA_K rows.
            const int ka = k / G::STEPS_PER_ATOM, kk = k % G::STEPS_PER_ATOM;
            const uint64_t ad = p.a_mn_major
                ? smem_desc_sw128(sa + k * G::UMMA_K * 128, G::ATOM_BYTES, 1024)
                : smem_desc_sw128(sa + ka * G::A_ATOM + kk * 32, 16, 1024);
            const uint64_t bd = p.b_mn_major
                ? smem_desc_sw128(sb + k * G::UMMA_K * 128, G::ATOM_BYTES, 1024)
                : smem_desc_sw128(sb + ka * T.b_atom + kk * 32, 16, 1024);
            // (debug build: both operands' start addresses inside the stage)
            if (kDebug && !dbg_check(
                    in_range(p.a_mn_major ? sa + k * G::UMMA_K * 128 : sa + ka * G::A_ATOM + kk * 32,
                             32, sa, sa + G::A_STAGE) &&
                        in_range(p.b_mn_major ? sb + k * G::UMMA_K * 128
                                              : sb + ka * T.b_atom + kk * 32,
                                 32, sb, sb + (uint32_t)T.b_stage),
                    kChkMmaSmem, w)) {
              ok = false;
              break;
            }
            const bool accumulate = kSK ? (kb != wk.kb0 || k != 0) : (kb | k) != 0;
            umma<CG, KIND>(d_tmem, ad, bd, idesc, accumulate ? 1u : 0u);
          }
          if (kDebug && !ok) break;
          umma_commit<CG, MULTI>(empty0 + 8u * s, all_mask);   // slot drained: tell every loader
          if (++s == S) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        umma_commit<CG, (CG == 2)>(tfull0 + 8u * acc, pair_mask);   // accumulator ready
        if (++acc == kAccStages) { acc = 0; aph ^= 1u; }
      }
      if constexpr (kRingStats) if (p.stats) {
        unsigned long long* const o = p.stats + (size_t)blockIdx.x * kStatWords;
        o[kStatMmaFull] = st_full;
        o[kStatMmaAcc] = st_acc;
        o[kStatMmaLoop] = clock64() - st_t0;
        o[kStatMmaStages] = st_stages;
      }
    }
    if constexpr (kRingStats) {
      if (p.stats && rank != 0 && lane == 0) {   // the pair's other CTA issues no MMAs
        unsigned long long* const o = p.stats + (size_t)blockIdx.x * kStatWords;
        o[kStatMmaFull] = o[kStatMmaAcc] = o[kStatMmaLoop] = o[kStatMmaStages] = 0ull;
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- epilogue
    // Each epilogue warp runs its own pipeline over the 32 tile rows whose
    // accumulator lanes it may read, through its own ring of shared-memory
    // sub-slots (32 rows x 32 columns of C/D and of X/Y): lane 0 TMA-loads the
    // C/X sub-tiles ahead (across tile boundaries), every lane reads its row,
    // computes D and Y and writes them back in place, and lane 0 TMA-stores
    // them.  With EPW = 2 two warps share each lane quarter and take its
    // chunks alternately (stream 0 the even, stream 1 the odd ones), each
    // with half the sub-slots.  The warps never wait on one another; they
    // meet only in the accumulator stage's release count.
    const int q = warp & 3;                 // TMEM lane quarter this warp may read
    const int ew = warp - 2;                // epilogue warp index, 0 .. 4 * EPW - 1
    const int strm = ew >> 2;               // which of the quarter's EPW chunk streams
    const bool lead = lane == 0;
    const bool loads = e.read_c || e.read_x;
    const uint32_t load_tx = (e.read_c ? sub_bytes(e.c_dt) : 0u) + (e.read_x ? sub_bytes(e.x_dt) : 0u);
    const uint32_t sub = slot_bytes / 4;               // one warp's share of a slot
    const uint32_t cd_sub = e.cd_bytes / 4;            // ... of which C/D
    // sub-slots of this warp: all E with one warp per quarter, else E / 2
    const int Ew = EPW == 1 ? E : max(1, E / EPW);
    const uint32_t ring0 = epi0 + (uint32_t)(ew * Ew) * sub;
    const uint32_t bar0 = cfull0 + 8u * (uint32_t)(ew * Ew);
    const uint64_t pol_in = make_l2_policy((p.l2_hints >> 2) & 3u);
    const uint64_t pol_out = make_l2_policy((p.l2_hints >> 4) & 3u);

    // Lane 0 walks this warp's stream of chunks (of BN / 32 per whole tile,
    // half that per half-width item, in item order: the chunks j = strm,
    // strm + EPW, ...) with a cursor that issues the TMA loads of its rows'
    // C/X into the warp's sub-slots.  The cursor computes an item's
    // coordinates once, when it enters the item.  TMA coordinates are
    // (column, row, batch) for row-major C/D/X/Y and (row, column, batch) for
    // column-major ones.
    struct Cursor { int it, j, nch, row0, col0, tl; };
    auto cursor_enter = [&](Cursor& cc) {
      for (; cc.it < p.num_items; cc.it += num_clusters) {
        const Work wk = work_item<kSK>(cc.it, p, num_clusters);
        if (wk.empty || !wk.owner) continue;   // no C/X: nothing, or a stream-K partial
        const int half = wk.half;
        cc.nch = half < 0 ? T.chunks : T.chunks / 2;
        if (strm >= cc.nch) continue;       // no chunk of this item in this stream
        int tm, tn;
        tile_coords(wk.tile, p, tm, tn, cc.tl);
        cc.j = strm;
        cc.row0 = tm * G::CM + (int)gm * (G::BM * CG) + (int)rank * G::BM + q * kSubRows;
        cc.col0 = tn * (BN * NC) + (int)gn * BN + (half > 0 ? BN / 2 : 0);
        return;
      }
    };
    auto cursor_next = [&](Cursor& cc) {
      if (cc.it < p.num_items && (cc.j += EPW) >= cc.nch) {
        cc.it += num_clusters;
        cursor_enter(cc);
      }
    };
    auto cursor_xy = [&](const Cursor& cc, int& x0, int& x1) {
      const int col = cc.col0 + cc.j * kEpiChunk;
      x0 = e.cd_m_major ? cc.row0 : col;
      x1 = e.cd_m_major ? col : cc.row0;
    };
    // (debug build: a C/X load's sub-slot inside the slots or the drained
    // ring, its inner coordinate a whole 16 bytes of both types)
    const uint32_t slots_end = epi0 + (uint32_t)E * slot_bytes;
    auto inner_ok = [&](int x, int dt) { return ((long long)x * (dt == DT_F32 ? 4 : 2)) % 16 == 0; };
    auto load_ok = [&](uint32_t dst, int x0) {
      const bool in_slots = in_range(dst, sub, ring0, ring0 + (uint32_t)Ew * sub) &&
                            dst + sub <= slots_end;
      const bool in_ring = in_range(dst, sub, b_ring, b_ring + ring_bytes);
      return (in_slots || in_ring) && (!e.read_c || inner_ok(x0, e.c_dt)) &&
             (!e.read_x || inner_ok(x0, e.x_dt));
    };
    Cursor ld{cluster_id, 0, 0, 0, 0, 0};
    int ld_slot = 0;
    auto issue_loads = [&]() {              // lane 0 only
      if (ld.it < p.num_items) {
        int x0, x1;
        cursor_xy(ld, x0, x1);
        const uint32_t slot = ring0 + (uint32_t)ld_slot * sub;
        const uint32_t bar = bar0 + 8u * (uint32_t)ld_slot;
        if (dbg_check(load_ok(slot, x0), kChkEpiLoad, w)) {
          mbar_arrive_expect_tx(bar, load_tx);
          if (e.read_c) tma_load_3d(slot, &tmC, bar, x0, x1, ld.tl, pol_in);
          if (e.read_x) tma_load_3d(slot + cd_sub, &tmX, bar, x0, x1, ld.tl, pol_in);
        }
      }
      if (++ld_slot == Ew) ld_slot = 0;
      cursor_next(ld);
    };

    // Loads run Ew - 1 chunks ahead (one sub-slot: the next chunk's load is
    // issued once the current chunk's store has read the sub-slot).
    if (lead && loads) {
      cursor_enter(ld);
      for (int c = 0; c < max(1, Ew - 1); ++c) issue_loads();
    }
    __syncwarp();

    int acc = 0;
    uint32_t aph = 0;
    int gc = 0;                             // chunk counter of this warp's stream
    int slot_idx = 0;                       // gc % Ew
    uint32_t slot_ph = 0;                   // (gc / Ew) & 1: phase of the slot's cfull barrier
    bool ok = true;
    long long st_tfull = 0, st_cfull = 0, st_read = 0, st_math = 0, st_issue = 0;
    long long st_chunks = 0;
    const long long st_t0 = stat_clock();
    for (int it = cluster_id; ok && it < p.num_items; it += num_clusters) {
      const Work wk = work_item<kSK>(it, p, num_clusters);
      if (wk.empty) continue;
      const int half = wk.half;
      int tm, tn, tl;
      tile_coords(wk.tile, p, tm, tn, tl);
      const int nchunks = half < 0 ? T.chunks : T.chunks / 2;
      const int ncol0 = tn * (BN * NC) + (int)gn * BN + (half > 0 ? BN / 2 : 0);
      const long long t_t = stat_clock();
      const bool ready = wait_phase(tfull0 + 8u * acc, aph, w, kWaitEpilogue, p.epi_wait_ns);
      if constexpr (kRingStats) st_tfull += clock64() - t_t;
      ok = __all_sync(0xFFFFFFFFu, ready);
      if (!ok) break;
      tc_fence_after_sync();
      if constexpr (kRingStats) st_chunks += nchunks;
      // The accumulator stage is handed back to the MMA warp after this
      // warp's last chunk of the item; a warp with no chunk in the item does
      // so at once.
      auto release_acc = [&]() {
        tc_fence_before_sync();
        __syncwarp();
        if (lead) {
          if constexpr (CG == 1) mbar_arrive(tempty0 + 8u * acc);
          else mbar_arrive_cluster(map_to_rank(tempty0 + 8u * acc, pair_leader));
        }
      };
      if (strm >= nchunks) {                // (never with stream-K: whole tiles, >= 2 chunks)
        release_acc();
        if (++acc == kAccStages) { acc = 0; aph ^= 1u; }
        continue;
      }
      const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)acc * kAccStride;
      // Stream-K partial sums: this CTA's slot of 128 x BN fp32 values, laid
      // out [chunk][16-byte piece][row] so that a warp's 32 rows of one piece
      // are 512 contiguous bytes.
      auto partial_rows = [&](int slot_cluster) {
        return reinterpret_cast<float4*>(p.sk_partials) +
               (size_t)(slot_cluster * CG + (int)rank) * (size_t)(BN * 32) + q * kSubRows + lane;
      };
      if (kSK && !wk.owner) {
        // ---- stream-K: the head of a tile another cluster owns.  Its
        // accumulator goes to this CTA's partial slot; once every epilogue
        // warp's stores are ordered, one thread publishes the slot's flag.
        float4* const dst = partial_rows(cluster_id);
        for (int j = strm; j < nchunks; j += EPW) {
          uint32_t raw[32];
          tmem_load_32cols(tbase + 32u * j, raw);
          tmem_wait_ld(raw);
          if (j + EPW >= nchunks) release_acc();
#pragma unroll
          for (int pc = 0; pc < 8; ++pc)
            __stcg(dst + (size_t)(j * 8 + pc) * 128,
                   make_float4(__uint_as_float(raw[4 * pc]), __uint_as_float(raw[4 * pc + 1]),
                               __uint_as_float(raw[4 * pc + 2]), __uint_as_float(raw[4 * pc + 3])));
        }
        fence_acq_rel_gpu();
        __syncwarp();
        if (lead) mbar_arrive(pdone);
        if (ew == 0) {
          const bool all = wait_phase<true>(pdone, 0u, w, kWaitPartial);
          if (lead && all) st_release_gpu(p.sk_flags + cluster_id * CG + (int)rank, 1u);
          ok = __all_sync(0xFFFFFFFFu, all);
        }
        if (++acc == kAccStages) { acc = 0; aph ^= 1u; }
        continue;
      }
      // This CTA's last item: once its accumulator is ready the operand ring
      // has been drained for good (no main loop follows), so the C/X chunks
      // the lookahead has not loaded yet all go into the ring at once, and
      // the rest of the epilogue waits on one load latency, not one per
      // chunk.  batch0: first chunk of the item taken from the ring (nchunks:
      // none).
      // Only lane 0 keeps the cursor; it decides and tells the warp.
      int batch0 = nchunks;
      if (loads && (it + num_clusters >= p.num_items || (kSK && p.sk_units))) {   // (stream-K: owned items come last)
        const int nb = ld.it == it ? (nchunks - ld.j + EPW - 1) / EPW : 0;   // this warp's
        if (lead && nb > 0 && (uint32_t)nb * (4u * EPW) * sub <= ring_bytes) {
          batch0 = ld.j;
          for (int c = 0; c < nb; ++c) {
            int x0, x1;
            cursor_xy(ld, x0, x1);
            const uint32_t dst = b_ring + (uint32_t)(c * 4 * EPW + ew) * sub;
            const uint32_t rb = rfull0 + 8u * (uint32_t)(ew * kMaxChunks + c);
            if (!dbg_check(load_ok(dst, x0), kChkEpiLoad, w)) break;
            mbar_arrive_expect_tx(rb, load_tx);
            if (e.read_c) tma_load_3d(dst, &tmC, rb, x0, x1, ld.tl, pol_in);
            if (e.read_x) tma_load_3d(dst + cd_sub, &tmX, rb, x0, x1, ld.tl, pol_in);
            cursor_next(ld);
          }
          ld.it = p.num_items;               // the cursor has nothing left to load
        }
        batch0 = __shfl_sync(0xFFFFFFFFu, batch0, 0);
      }
      // Stream-K owner: the clusters sk_first .. cluster_id - 1 hold the tile's
      // earlier k-blocks; wait until each has published its partial (after the C/X loads
      // above are under way).
      int sk_first = cluster_id;
      if (kSK && p.sk_units) {
        sk_first = sk_unit_of((long long)wk.tile * p.k_blocks, p);
        bool got = true;
        for (int c = sk_first; got && c < cluster_id; ++c) {
          const uint32_t* f = p.sk_flags + c * CG + (int)rank;
          const uint64_t t0 = globaltimer_ns();
          while (ld_acquire_gpu(f) == 0u) {
            if (*w.abort) { got = false; break; }
            if (globaltimer_ns() - t0 > w.timeout_ns) {
              *w.abort = 1u;
              atomicCAS(w.status, 0u, 0xE0000000u | (kWaitPartial << 16) | (blockIdx.x & 0xFFFFu));
              got = false;
              break;
            }
          }
        }
        ok = __all_sync(0xFFFFFFFFu, got);
        if (!ok) break;
      }
      const int row0 = tm * G::CM + (int)gm * (G::BM * CG) + (int)rank * G::BM + q * kSubRows;
#pragma unroll 1
      for (int j = strm; j < nchunks; j += EPW, ++gc) {
        // The accumulator columns are requested first: their latency overlaps
        // the wait for C/X and the shared-memory reads below.
        uint32_t raw_acc[32];
        // (debug build: the chunk's 32 columns inside the item's accumulator)
        if (dbg_check(32 * (j + 1) <= (half < 0 ? BN : BN / 2) &&
                          (uint32_t)acc * kAccStride + 32u * (j + 1) <= kTmemCols,
                      kChkEpiTmem, w))
          tmem_load_32cols(tbase + 32u * j, raw_acc);
        else
          for (int i = 0; i < 32; ++i) raw_acc[i] = 0u;
        const bool from_ring = j >= batch0;
        const int bc = (j - batch0) / EPW;  // index in this warp's ring batch
        const uint32_t s_addr = from_ring ? b_ring + (uint32_t)(bc * 4 * EPW + ew) * sub
                                          : ring0 + (uint32_t)slot_idx * sub;
        uint8_t* const slot = gbase + (s_addr - base);
        float cv[kEpiChunk], xv[kEpiChunk];
        bool got = dbg_check(from_ring ? in_range(s_addr, sub, b_ring, b_ring + ring_bytes)
                                       : in_range(s_addr, sub, ring0, ring0 + (uint32_t)Ew * sub) &&
                                             s_addr + sub <= slots_end,
                             kChkEpiSmem, w);
        const long long t_c = stat_clock();
        if (loads && got)
          got = from_ring ? wait_phase<true>(rfull0 + 8u * (uint32_t)(ew * kMaxChunks + bc), 0u, w,
                                             kWaitEpiLoad)
                          : wait_phase<true>(bar0 + 8u * slot_idx, slot_ph, w, kWaitEpiLoad);
        long long t_r = 0;
        if constexpr (kRingStats) { t_r = clock64(); st_cfull += t_r - t_c; }
        got = __all_sync(0xFFFFFFFFu, got);
        if constexpr (EPW == 1) {
          // One warp per lane quarter: the C/X rows are read while the
          // accumulator load is in flight.
          if (got && e.read_c) {
            smem_read_row(slot, e.c_dt, e.cd_m_major, lane, cv);
          } else {
#pragma unroll
            for (int i = 0; i < kEpiChunk; ++i) cv[i] = 0.f;
          }
          if (got && e.read_x) smem_read_row(slot + cd_sub, e.x_dt, e.cd_m_major, lane, xv);
        }
        __syncwarp();                       // the .aligned wait needs the whole warp
        tmem_wait_ld(raw_acc);
        // Normalise the accumulator to fp32 bit patterns once per chunk (uniform
        // branches), so the per-element epilogue below is the same for every case.
        if (p.k_blocks == 0) {
#pragma unroll
          for (int i = 0; i < 32; ++i) raw_acc[i] = 0u;     // K = 0: nothing was accumulated
        } else if (e.acc_f16) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            raw_acc[i] = __float_as_uint(__half2float(__ushort_as_half((uint16_t)raw_acc[i])));
        }
        // Stream-K owner: add the earlier k-blocks' partial sums, in the
        // order of the clusters that hold them (fp32 accumulators only).
        for (int c = sk_first; kSK && c < cluster_id; ++c) {
          const float4* const src = partial_rows(c) + (size_t)j * 8 * 128;
#pragma unroll
          for (int pc = 0; pc < 8; ++pc) {
            const float4 v = __ldcg(src + pc * 128);
            raw_acc[4 * pc] = __float_as_uint(__uint_as_float(raw_acc[4 * pc]) + v.x);
            raw_acc[4 * pc + 1] = __float_as_uint(__uint_as_float(raw_acc[4 * pc + 1]) + v.y);
            raw_acc[4 * pc + 2] = __float_as_uint(__uint_as_float(raw_acc[4 * pc + 2]) + v.z);
            raw_acc[4 * pc + 3] = __float_as_uint(__uint_as_float(raw_acc[4 * pc + 3]) + v.w);
          }
        }
        if (j + EPW >= nchunks) release_acc();   // this warp's last chunk of the stage
        ok = got;
        if (!ok) break;
        long long t_m = 0;
        if constexpr (kRingStats) { t_m = clock64(); st_read += t_m - t_r; }
        // No store still reads the sub-slot D and Y go into (with C/X loads,
        // the load that filled it was issued after that), and every lane has
        // read its C/X row before any lane overwrites the sub-slot (a narrower
        // D packs rows differently from a wider C).
        if (lead && !loads) {
          if (Ew >= 2) bulk_wait_group_read<1>();
          else bulk_wait_group_read<0>();
        }
        __syncwarp();
        // D from the accumulator, C (zero when not read) and X; the branches
        // are uniform and outside the element loops.
        float dv[kEpiChunk];
        const float al = e.alpha, be = e.beta, xf = e.x_factor;
        if constexpr (EPW == 2) {
          // Two warps per lane quarter (a 168-register budget): C and X are
          // folded into D as their pieces are read, after the accumulator
          // load, so no whole C or X row is held; the same operations in the
          // same order as below, so both forms give the same bits.
          auto fold_c = [&](bool first) {   // first: dv = be * c, else dv = fma(be, c, dv)
            if (e.read_c) {
              if (first)
                smem_row_each(slot, e.c_dt, e.cd_m_major, lane,
                              [&](int i, float c) { dv[i] = be * c; });
              else
                smem_row_each(slot, e.c_dt, e.cd_m_major, lane,
                              [&](int i, float c) { dv[i] = fmaf(be, c, dv[i]); });
            } else {
#pragma unroll
              for (int i = 0; i < kEpiChunk; ++i) dv[i] = first ? be * 0.f : fmaf(be, 0.f, dv[i]);
            }
          };
          if (e.read_x && !e.relu) {
            // fmaf(al, acc, fmaf(be, c, xf * x))
            smem_row_each(slot + cd_sub, e.x_dt, e.cd_m_major, lane,
                          [&](int i, float x) { dv[i] = xf * x; });
            fold_c(false);
#pragma unroll
            for (int i = 0; i < kEpiChunk; ++i)
              dv[i] = fmaf(al, __uint_as_float(raw_acc[i]), dv[i]);
          } else {
            // fmaf(al, acc, be * c), then relu, then fmaf(xf, x, .)
            fold_c(true);
#pragma unroll
            for (int i = 0; i < kEpiChunk; ++i)
              dv[i] = fmaf(al, __uint_as_float(raw_acc[i]), dv[i]);
            if (e.relu) {
#pragma unroll
              for (int i = 0; i < kEpiChunk; ++i) dv[i] = fmaxf(dv[i], 0.f);
            }
            if (e.read_x)
              smem_row_each(slot + cd_sub, e.x_dt, e.cd_m_major, lane,
                            [&](int i, float x) { dv[i] = fmaf(xf, x, dv[i]); });
          }
          __syncwarp();                     // every lane has read its C/X row
        } else if (e.read_x) {
          if (e.relu) {
#pragma unroll
            for (int i = 0; i < kEpiChunk; ++i)
              dv[i] = fmaf(xf, xv[i], fmaxf(fmaf(al, __uint_as_float(raw_acc[i]), be * cv[i]), 0.f));
          } else {
#pragma unroll
            for (int i = 0; i < kEpiChunk; ++i)
              dv[i] = fmaf(al, __uint_as_float(raw_acc[i]), fmaf(be, cv[i], xf * xv[i]));
          }
        } else {
          if (e.relu) {
#pragma unroll
            for (int i = 0; i < kEpiChunk; ++i)
              dv[i] = fmaxf(fmaf(al, __uint_as_float(raw_acc[i]), be * cv[i]), 0.f);
          } else {
#pragma unroll
            for (int i = 0; i < kEpiChunk; ++i)
              dv[i] = fmaf(al, __uint_as_float(raw_acc[i]), be * cv[i]);
          }
        }
        smem_write_row(slot, e.d_dt, e.cd_m_major, lane, dv);
        if (e.write_y) {
          float yv[kEpiChunk];
#pragma unroll
          for (int i = 0; i < kEpiChunk; ++i) yv[i] = __uint_as_float(raw_acc[i]);
          smem_write_row(slot + cd_sub, e.y_dt, e.cd_m_major, lane, yv);
        }
        fence_proxy_async_smem();
        __syncwarp();
        long long t_i = 0;
        if constexpr (kRingStats) { t_i = clock64(); st_math += t_i - t_m; }
        if (lead) {
          const int col0 = ncol0 + j * kEpiChunk;
          const int x0 = e.cd_m_major ? row0 : col0, x1 = e.cd_m_major ? col0 : row0;
          // (debug build: a store starts at non-negative coordinates, its inner
          // one a whole 16 bytes of both output types)
          if (dbg_check(x0 >= 0 && x1 >= 0 && inner_ok(x0, e.d_dt) &&
                            (!e.write_y || inner_ok(x0, e.y_dt)),
                        kChkEpiStore, w)) {
            tma_store_3d(&tmD, s_addr, x0, x1, tl, pol_out);
            if (e.write_y) tma_store_3d(&tmY, s_addr + cd_sub, x0, x1, tl, pol_out);
          }
          bulk_commit_group();
          if (loads) {
            // C/X of chunk gc+Ew-1 go into the sub-slot of chunk gc-1, once its
            // store (the one before the store just issued) has read it (with
            // one sub-slot: chunk gc+1 into chunk gc's, once its store has);
            // with nothing left to load (the drained-ring batch has the rest)
            // no store is waited for.
            if (ld.it < p.num_items) {
              if (Ew >= 2) bulk_wait_group_read<1>();
              else bulk_wait_group_read<0>();
            }
            issue_loads();
          }
        }
        if (++slot_idx == Ew) { slot_idx = 0; slot_ph ^= 1u; }
        __syncwarp();
        if constexpr (kRingStats) st_issue += clock64() - t_i;
      }
      if (kSK && p.sk_units && sk_first < cluster_id && ok) {
        // Every epilogue warp has read the partials: clear their flags for
        // the next launch (which reads nothing before this grid completes).
        __syncwarp();
        if (lead) mbar_arrive(pread);
        if (ew == 0) {
          const bool all = wait_phase<true>(pread, 0u, w, kWaitPartial);
          if (lead && all)
            for (int c = sk_first; c < cluster_id; ++c) p.sk_flags[c * CG + (int)rank] = 0u;
          ok = __all_sync(0xFFFFFFFFu, all);
        }
      }
      if (++acc == kAccStages) { acc = 0; aph ^= 1u; }
    }
    // The stores must have read their shared memory before the CTA exits; their
    // writes to global memory complete with the grid.
    if (lead) bulk_wait_group_read<0>();
    if constexpr (kRingStats) {
      if (threadIdx.x == kEpiLeader && p.stats) {
        unsigned long long* const o = p.stats + (size_t)blockIdx.x * kStatWords;
        o[kStatEpiTfull] = st_tfull;
        o[kStatEpiCfull] = st_cfull;
        o[kStatEpiLoop] = clock64() - st_t0;
        o[kStatEpiChunks] = st_chunks;
        o[kStatEpiOwnChunks] = gc;
        o[kStatEpiRead] = st_read;
        o[kStatEpiMath] = st_math;
        o[kStatEpiIssue] = st_issue;
      }
    }
    __syncwarp();
  }

  // ------------------------------------------------------------ teardown
  __syncthreads();
  if (*abort_ptr) {
    // A wait gave up: let copies and MMAs already issued drain before the
    // shared and tensor memory they target are released.
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 2000000ull) {
    }
  }
  __syncwarp();
  if constexpr (MULTI) cluster_sync_all();    // other CTAs may still use our smem/TMEM
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc<CG>(tmem_base, kTmemCols);
  }
}

}  // namespace gb300
