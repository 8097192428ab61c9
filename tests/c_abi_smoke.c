/* A plain C99 client of the library: only include/gemm_gb300.h and
 * libgemm_gb300.so, no CUDA headers or runtime of its own.
 *
 *   c_abi_smoke check   host-only calls (validation, planning, status names)
 *   c_abi_smoke run     one GEMM on host buffers through gemm_run_host: f16
 *                       integer inputs in [-2, 2], fp32 C and D, compared
 *                       exactly with integer arithmetic (every intermediate is
 *                       an integer below 2^24)
 * Exit status 0 on success. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "gemm_gb300.h"

/* IEEE binary16 bit patterns of the integers -2..2. */
static uint16_t f16_bits(int v) {
  static const uint16_t tab[5] = {0xC000u, 0xBC00u, 0x0000u, 0x3C00u, 0x4000u};
  return tab[v + 2];
}

static gemm_dtypes_t dtypes_f16_f32(void) {
  gemm_dtypes_t t;
  memset(&t, 0, sizeof t);
  t.ab = GEMM_F16;
  t.c = GEMM_F32;
  t.d = GEMM_F32;
  t.x = GEMM_F32;
  t.y = GEMM_F32;
  t.cdxy_major = GEMM_K_MAJOR;
  return t;
}

static int check(void) {
  gemm_problem_t p;
  gemm_config_t cfg;
  memset(&p, 0, sizeof p);
  p.M = 1000; p.N = 1024; p.K = 512; p.L = 2;
  p.A = (const void*)(uintptr_t)0x100000; p.lda = 512; p.layoutA = GEMM_K_MAJOR;
  p.B = (const void*)(uintptr_t)0x200000; p.ldb = 512; p.layoutB = GEMM_K_MAJOR;
  p.C = (const void*)(uintptr_t)0x300000; p.D = (void*)(uintptr_t)0x400000;
  p.alpha = 1.0f; p.beta = 1.0f; p.x_factor = 0.0f;
  p.dtypes = dtypes_f16_f32();
  if (gemm_check(&p) != GEMM_OK) { puts("check: valid problem rejected"); return 1; }
  if (gemm_plan(&p, 152, 232448, NULL, &cfg) != GEMM_OK || cfg.tiles <= 0) {
    puts("plan failed"); return 1;
  }
  printf("plan: %dx%d tiles, cta_group %d, %d stages, %d epilogue slots, %lld tiles\n",
         cfg.tile_m, cfg.tile_n, cfg.cta_group, cfg.stages, cfg.epi_slots, (long long)cfg.tiles);
  p.lda = 516;                                   /* 1032-byte rows: not 16-byte aligned */
  if (gemm_check(&p) != GEMM_ERR_MISALIGNED) { puts("check: misalignment missed"); return 1; }
  if (strcmp(gemm_status_string(GEMM_ERR_MISALIGNED), "GEMM_ERR_MISALIGNED") != 0) return 1;
  puts("check: OK");
  return 0;
}

static int run(void) {
  enum { M = 200, N = 136, K = 256, L = 2 };
  uint16_t* A = malloc(sizeof(uint16_t) * L * M * K);
  uint16_t* B = malloc(sizeof(uint16_t) * L * N * K);
  int* Ai = malloc(sizeof(int) * L * M * K);
  int* Bi = malloc(sizeof(int) * L * N * K);
  float* C = malloc(sizeof(float) * L * M * N);
  float* D = malloc(sizeof(float) * L * M * N);
  if (!A || !B || !Ai || !Bi || !C || !D) return 1;
  uint32_t seed = 12345u;
  for (int i = 0; i < L * M * K; ++i) {
    seed = seed * 1664525u + 1013904223u;
    Ai[i] = (int)((seed >> 16) % 5u) - 2;
    A[i] = f16_bits(Ai[i]);
  }
  for (int i = 0; i < L * N * K; ++i) {
    seed = seed * 1664525u + 1013904223u;
    Bi[i] = (int)((seed >> 16) % 5u) - 2;
    B[i] = f16_bits(Bi[i]);
  }
  for (int i = 0; i < L * M * N; ++i) {
    seed = seed * 1664525u + 1013904223u;
    C[i] = (float)((int)((seed >> 16) % 7u) - 3);
  }
  gemm_handle_t h = NULL;
  gemm_status_t st = gemm_create(&h, 0);
  if (st != GEMM_OK) { printf("create: %s\n", gemm_status_string(st)); return 1; }
  const gemm_dtypes_t dt = dtypes_f16_f32();
  st = gemm_run_host(h, M, N, K, L, A, K, GEMM_K_MAJOR, B, K, GEMM_K_MAJOR, C, NULL, D, NULL,
                     1.5f, -0.5f, 0.0f, &dt, NULL);
  uint32_t detail = 0;
  if (st == GEMM_OK) st = gemm_sync_status(h, NULL, &detail);
  if (st != GEMM_OK) { printf("run: %s %#x\n", gemm_status_string(st), detail); return 1; }
  long bad = 0;
  for (int l = 0; l < L; ++l)
    for (int m = 0; m < M; ++m)
      for (int n = 0; n < N; ++n) {
        long acc = 0;
        for (int k = 0; k < K; ++k)
          acc += (long)Ai[(l * M + m) * K + k] * Bi[(l * N + n) * K + k];
        const double want = 1.5 * (double)acc - 0.5 * (double)C[(l * M + m) * N + n];
        if ((double)D[(l * M + m) * N + n] != want) ++bad;
      }
  gemm_destroy(h);
  free(A); free(B); free(Ai); free(Bi); free(C); free(D);
  if (bad) { printf("run: %ld of %d entries differ\n", bad, L * M * N); return 1; }
  puts("run: OK (bit-exact)");
  return 0;
}

int main(int argc, char** argv) {
  if (argc > 1 && strcmp(argv[1], "run") == 0) return run();
  return check();
}
