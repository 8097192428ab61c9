// Persistent, warp-specialised batched GEMM with a fused epilogue for sm_103a.
//
//   Y = A*B,   D = alpha*(A*B) + beta*C + x_factor*X     (fp32 accumulate + epilogue)
//
// What the kernel computes and its warp roles follow "custom_epilogue_dense_gemm.py"
// (CuTeDSL Blackwell example), module docstring "This GEMM works as follows" (DMA
// warp, MMA warp, EPILOGUE warps; persistent tile scheduling) and the 2-SM tcgen05
// scheme of "04_mma_tma_2sm_sm100.cu" (CuTe Blackwell tutorial 04, "Step 2: The
// Mainloop" -- the leader CTA issues the pair's MMA; tensor-memory allocation and
// MMA-completion arrivals reach both CTAs).  The thread roles (128 epilogue threads +
// one MMA warp + one TMA warp = 192 threads, one CTA per SM, the whole 512-column
// tensor memory split into accumulator stages) follow the cuBLASDx "API Card:
// Blackwell Pipeline (tcgen05)", host-side and "Depth and shared memory" bullets.
//
// Block = 6 warps:
//   warp 0      TMA producer: one lane streams A and B k-blocks into a ring of
//               `stages` shared-memory slots, each guarded by full/empty mbarriers.
//   warp 1      tensor-memory allocator + MMA issuer: one lane of the leader CTA
//               issues tcgen05.mma into one of two accumulator stages in tensor
//               memory, frees ring slots with tcgen05.commit, and hands finished
//               accumulators to the epilogue with another commit.
//   warps 2..5  epilogue: tcgen05.ld the accumulator (warp w owns TMEM lanes
//               32*(w%4)..+31 = tile rows), release the accumulator stage, read C
//               and X, compute in fp32, convert and store D and Y.
// Every CTA (pair) walks the same static persistent tile sequence
// t = cluster_id, cluster_id + num_clusters, ...; with two accumulator stages the
// epilogue of tile i overlaps the main loop of tile i+1.
//
// Every barrier wait is bounded (watchdog): on expiry the kernel records a code
// in a device status word, raises a CTA-wide abort flag, lets in-flight copies
// drain, frees its tensor memory and returns.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace gb300 {

enum : int { DT_F32 = 0, DT_F16 = 1, DT_BF16 = 2, DT_E4M3 = 3 };

struct EpiParams {
  const void* C;
  const void* X;
  void* D;
  void* Y;
  int c_dt, d_dt, x_dt, y_dt;
  int cd_m_major;            // 0: (l*M + m)*N + n   1: (l*N + n)*M + m
  int read_c, read_x, write_y;
  float alpha, beta, x_factor;
};

struct KernelParams {
  int M, N, K, L;
  int tiles_m, tiles_n;      // tiles per batch along M (of 128*cta_group rows) and N
  int num_tiles;             // tiles_m * tiles_n * L
  int k_blocks;              // ceil(K / tile_k)
  int group_m;               // rasterisation strip height (tiles)
  int stages;                // ring depth
  int a_mn_major, b_mn_major;
  uint32_t idesc;            // tcgen05 instruction descriptor
  uint32_t* status;          // device status word (watchdog)
  unsigned long long timeout_ns;
  EpiParams epi;
};

constexpr int kThreads = 192;
constexpr int kAccStages = 2;
constexpr uint32_t kTmemCols = 512;

template <int CG, int BN, int AB_BYTES>
struct Geometry {
  static constexpr int BM = 128;                 // A rows staged per CTA
  static constexpr int BK = 128 / AB_BYTES;      // K per ring stage: one 128-byte row
  static constexpr int BN_CTA = BN / CG;         // B rows staged per CTA
  static constexpr int A_STAGE = BM * 128;       // bytes
  static constexpr int B_STAGE = BN_CTA * 128;   // bytes
  static constexpr int UMMA_K = 32 / AB_BYTES;   // K per tcgen05.mma (32 bytes)
  static constexpr int K_STEPS = BK / UMMA_K;    // instructions per stage
  static constexpr int ATOM_MN = 128 / AB_BYTES; // MN extent of one MN-major swizzle atom
  static constexpr int ATOM_BYTES = BK * 128;    // bytes of one MN-major atom column
  static_assert(BN % 32 == 0 && BN <= 256, "tile_n");
  static_assert(kAccStages * BN <= (int)kTmemCols, "accumulators must fit tensor memory");
};

// Watchdog codes: 0xE0RRBBBB, RR = role, BBBB = low 16 bits of blockIdx.x.
enum : uint32_t { kWaitProducer = 1, kWaitMmaFull = 2, kWaitMmaAcc = 3, kWaitEpilogue = 4 };

struct Watch {
  volatile uint32_t* abort;
  uint32_t* status;
  unsigned long long timeout_ns;
};

__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const Watch& w,
                                           uint32_t role) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
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
}

// ------------------------------------------------------------------ epilogue I/O

__device__ __forceinline__ float bits16_to_f32(uint32_t b, int dt) {
  return dt == DT_BF16 ? __uint_as_float(b << 16) : __half2float(__ushort_as_half((uint16_t)b));
}

__device__ __forceinline__ uint32_t f32_to_bits16(float v, int dt) {
  return dt == DT_BF16 ? (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v))
                       : (uint32_t)__half_as_ushort(__float2half_rn(v));
}

// Load 8 consecutive row elements starting at element `off` (16-byte aligned)
// of a row-major tensor; `valid` elements of the 8 exist (8 or 4).
__device__ __forceinline__ void load8(const void* base, int dt, int64_t off, int valid,
                                      float (&v)[8]) {
  if (dt == DT_F32) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + off);
    const float4 a = p[0];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    if (valid > 4) {
      const float4 b = p[1];
      v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
      v[4] = v[5] = v[6] = v[7] = 0.f;
    }
  } else {
    const uint4 q = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + off);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = bits16_to_f32(w[i] & 0xFFFFu, dt);
      v[2 * i + 1] = bits16_to_f32(w[i] >> 16, dt);
    }
  }
}

__device__ __forceinline__ void store8(void* base, int dt, int64_t off, int valid,
                                       const float (&v)[8]) {
  if (dt == DT_F32) {
    float4* p = reinterpret_cast<float4*>(static_cast<float*>(base) + off);
    p[0] = make_float4(v[0], v[1], v[2], v[3]);
    if (valid > 4) p[1] = make_float4(v[4], v[5], v[6], v[7]);
  } else {
    uint4 q;
    q.x = f32_to_bits16(v[0], dt) | (f32_to_bits16(v[1], dt) << 16);
    q.y = f32_to_bits16(v[2], dt) | (f32_to_bits16(v[3], dt) << 16);
    q.z = f32_to_bits16(v[4], dt) | (f32_to_bits16(v[5], dt) << 16);
    q.w = f32_to_bits16(v[6], dt) | (f32_to_bits16(v[7], dt) << 16);
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(base) + off) = q;
  }
}

__device__ __forceinline__ float load1(const void* base, int dt, int64_t off) {
  if (dt == DT_F32) return static_cast<const float*>(base)[off];
  return bits16_to_f32(static_cast<const uint16_t*>(base)[off], dt);
}

__device__ __forceinline__ void store1(void* base, int dt, int64_t off, float v) {
  if (dt == DT_F32)
    static_cast<float*>(base)[off] = v;
  else
    static_cast<uint16_t*>(base)[off] = (uint16_t)f32_to_bits16(v, dt);
}

__device__ __forceinline__ float epi_combine(const EpiParams& e, float acc, float c, float x) {
  // alpha*acc + beta*c + x_factor*x in fp32 (terms that are not read are 0).
  return fmaf(e.alpha, acc, fmaf(e.beta, c, e.x_factor * x));
}

// One thread's 32 consecutive columns [col0, col0+32) of output row `row`.
__device__ __forceinline__ void epilogue_row_chunk(const EpiParams& e, int M, int N, int row,
                                                   int col0, int l, const float (&acc)[32]) {
  if (row >= M) return;
  const int64_t batch = (int64_t)l * M * N;
  if (!e.cd_m_major) {
    const int64_t rowoff = batch + (int64_t)row * N;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const int c = col0 + 8 * g;
      if (c >= N) break;
      const int valid = min(8, N - c);
      float cv[8], xv[8], dv[8], yv[8];
      if (e.read_c) load8(e.C, e.c_dt, rowoff + c, valid, cv);
      else {
#pragma unroll
        for (int i = 0; i < 8; ++i) cv[i] = 0.f;
      }
      if (e.read_x) load8(e.X, e.x_dt, rowoff + c, valid, xv);
      else {
#pragma unroll
        for (int i = 0; i < 8; ++i) xv[i] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        yv[i] = acc[8 * g + i];
        dv[i] = epi_combine(e, yv[i], cv[i], xv[i]);
      }
      store8(e.D, e.d_dt, rowoff + c, valid, dv);
      if (e.write_y) store8(e.Y, e.y_dt, rowoff + c, valid, yv);
    }
  } else {
    // Column-major outputs: each store instruction of the warp covers 32
    // consecutive rows of one column.
#pragma unroll 4
    for (int j = 0; j < 32; ++j) {
      const int col = col0 + j;
      if (col >= N) break;
      const int64_t off = batch + (int64_t)col * M + row;
      const float c = e.read_c ? load1(e.C, e.c_dt, off) : 0.f;
      const float x = e.read_x ? load1(e.X, e.x_dt, off) : 0.f;
      store1(e.D, e.d_dt, off, epi_combine(e, acc[j], c, x));
      if (e.write_y) store1(e.Y, e.y_dt, off, acc[j]);
    }
  }
}

// ------------------------------------------------------------------ the kernel

template <int CG, int BN, int AB_BYTES>
__global__ void __launch_bounds__(kThreads, 1)
persistent_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ KernelParams p) {
  using G = Geometry<CG, BN, AB_BYTES>;
  constexpr int KIND = (AB_BYTES == 1) ? 1 : 0;

  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the 128-byte-swizzle atoms (identical in both CTAs
  // of a pair: same kernel, same layout).
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = (CG == 2) ? cluster_ctarank() : 0u;
  const int cluster_id = blockIdx.x / CG;
  const int num_clusters = gridDim.x / CG;
  const int S = p.stages;

  // Shared layout: [B ring][A ring][full x S][empty x S][tfull x 2][tempty x 2][tmem addr][abort]
  const uint32_t b_ring = base;
  const uint32_t a_ring = b_ring + S * G::B_STAGE;
  const uint32_t bars = a_ring + S * G::A_STAGE;
  const uint32_t full0 = bars, empty0 = bars + 8u * S;
  const uint32_t tfull0 = bars + 16u * S, tempty0 = tfull0 + 16u;
  const uint32_t holder = tempty0 + 16u;
  volatile uint32_t* const holder_ptr = reinterpret_cast<volatile uint32_t*>(gbase + (holder - base));
  volatile uint32_t* const abort_ptr = holder_ptr + 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8u * s, 1);
      mbar_init(empty0 + 8u * s, 1);
    }
    for (int a = 0; a < kAccStages; ++a) {
      mbar_init(tfull0 + 8u * a, 1);
      mbar_init(tempty0 + 8u * a, 4 * CG);   // every epilogue warp of the CTA (pair)
    }
    *abort_ptr = 0u;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc<CG>(holder, kTmemCols);
    tmem_relinquish<CG>();
  }
  tc_fence_before_sync();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync_all();
  tc_fence_after_sync();
  const uint32_t tmem_base = *holder_ptr;

  const Watch w{abort_ptr, p.status, p.timeout_ns};

  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      prefetch_tensormap(&tmA);
      prefetch_tensormap(&tmB);
      const uint32_t tx_bytes = (uint32_t)(CG * (G::A_STAGE + G::B_STAGE));
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int t = cluster_id; ok && t < p.num_tiles; t += num_clusters) {
        int tm, tn, tl;
        tile_coords(t, p, tm, tn, tl);
        const int m0 = tm * (G::BM * CG) + (int)rank * G::BM;
        const int n0 = tn * BN + (int)rank * G::BN_CTA;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!wait_phase(empty0 + 8u * s, ph ^ 1u, w, kWaitProducer)) { ok = false; break; }
          const uint32_t fb = full0 + 8u * s;
          if (rank == 0) mbar_arrive_expect_tx(fb, tx_bytes);
          const uint32_t fb_target = (CG == 2) ? map_to_rank(fb, 0) : fb;
          const int k0 = kb * G::BK;
          const uint32_t sa = a_ring + s * G::A_STAGE;
          const uint32_t sb = b_ring + s * G::B_STAGE;
          auto issue = [&](const CUtensorMap* map, uint32_t dst, int c0, int c1) {
            if constexpr (CG == 1) tma_load_3d(dst, map, fb_target, c0, c1, tl);
            else tma_load_3d_pair(dst, map, fb_target, c0, c1, tl);
          };
          if (!p.a_mn_major) {
            issue(&tmA, sa, k0, m0);                           // box {BK, 128}
          } else {
#pragma unroll
            for (int j = 0; j < G::BM / G::ATOM_MN; ++j)       // boxes {ATOM_MN, BK}
              issue(&tmA, sa + j * G::ATOM_BYTES, m0 + j * G::ATOM_MN, k0);
          }
          if (!p.b_mn_major) {
            issue(&tmB, sb, k0, n0);                           // box {BK, BN_CTA}
          } else {
#pragma unroll
            for (int j = 0; j < G::BN_CTA / G::ATOM_MN; ++j)
              issue(&tmB, sb + j * G::ATOM_BYTES, n0 + j * G::ATOM_MN, k0);
          }
          if (++s == S) { s = 0; ph ^= 1u; }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (rank == 0 && lane == 0) {
      int s = 0, acc = 0;
      uint32_t ph = 0, aph = 0;
      bool ok = true;
      for (int t = cluster_id; ok && t < p.num_tiles; t += num_clusters) {
        if (!wait_phase(tempty0 + 8u * acc, aph ^ 1u, w, kWaitMmaAcc)) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!wait_phase(full0 + 8u * s, ph, w, kWaitMmaFull)) { ok = false; break; }
          tc_fence_after_sync();
          const uint32_t sa = a_ring + s * G::A_STAGE;
          const uint32_t sb = b_ring + s * G::B_STAGE;
#pragma unroll
          for (int k = 0; k < G::K_STEPS; ++k) {
            // K-major: rows of 128 bytes, 8-row groups 1024 bytes apart; step k
            // moves 32 bytes along the swizzled row.  MN-major: K rows of 128
            // bytes, 8-row groups 1024 apart, MN atoms ATOM_BYTES apart; step k
            // moves UMMA_K rows.
            const uint64_t ad = p.a_mn_major
                ? smem_desc_sw128(sa + k * G::UMMA_K * 128, G::ATOM_BYTES, 1024)
                : smem_desc_sw128(sa + k * 32, 16, 1024);
            const uint64_t bd = p.b_mn_major
                ? smem_desc_sw128(sb + k * G::UMMA_K * 128, G::ATOM_BYTES, 1024)
                : smem_desc_sw128(sb + k * 32, 16, 1024);
            umma<CG, KIND>(d_tmem, ad, bd, p.idesc, (kb | k) != 0 ? 1u : 0u);
          }
          umma_commit<CG>(empty0 + 8u * s, (uint16_t)0x3);     // frees the slot in both CTAs
          if (++s == S) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        umma_commit<CG>(tfull0 + 8u * acc, (uint16_t)0x3);     // accumulator ready
        if (++acc == kAccStages) { acc = 0; aph ^= 1u; }
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;                 // TMEM lane quarter this warp may read
    int acc = 0;
    uint32_t aph = 0;
    for (int t = cluster_id; t < p.num_tiles; t += num_clusters) {
      int tm, tn, tl;
      tile_coords(t, p, tm, tn, tl);
      if (!wait_phase(tfull0 + 8u * acc, aph, w, kWaitEpilogue)) break;
      tc_fence_after_sync();
      const int row = tm * (G::BM * CG) + (int)rank * G::BM + q * 32 + lane;
      const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tmem_load_32cols(tbase + 32u * c, r);
        tmem_wait_ld();
        if (c == BN / 32 - 1) {
          // The whole stage has been read: hand it back to the MMA warp.
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) {
            if constexpr (CG == 1) mbar_arrive(tempty0 + 8u * acc);
            else mbar_arrive_cluster(map_to_rank(tempty0 + 8u * acc, 0));
          }
        }
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = p.k_blocks > 0 ? __uint_as_float(r[j]) : 0.f;
        epilogue_row_chunk(p.epi, p.M, p.N, row, tn * BN + 32 * c, tl, v);
      }
      if (++acc == kAccStages) { acc = 0; aph ^= 1u; }
    }
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
  if constexpr (CG == 2) cluster_sync_all();   // the peer may still use our smem/TMEM
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc<CG>(tmem_base, kTmemCols);
  }
}

}  // namespace gb300
