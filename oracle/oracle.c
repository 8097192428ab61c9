/*
 * Plain fp64 CPU oracle for the batched GEMM with custom epilogue.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg use this file.  It shares no code, header or
 * table with the CUDA library and the library never calls it.
 *
 * What it computes (for every batch l < L, row m < M, column n < N):
 *
 *   acc(m,n,l) = sum_{k=0}^{K-1} A(m,k,l) * B(n,k,l)          (B is N x K)
 *   Y(m,n,l)   = acc(m,n,l)
 *   D(m,n,l)   = alpha * acc(m,n,l) + beta * C(m,n,l) + x_factor * X(m,n,l)
 *   relu variant: D = max(alpha * acc + beta * C, 0) + x_factor * X
 *
 * Sources:
 *   - "04_mma_tma_2sm_sm100.cu" (CUTLASS CuTe Blackwell tutorial 04), header
 *     comment: D = beta*C + alpha*A*B with A MxK K-major, B NxK K-major,
 *     C and D MxN N-major; epilogue "AXPBY RMEM -> RMEM" step.
 *   - "custom_epilogue_dense_gemm.py" (CuTeDSL Blackwell custom-epilogue
 *     example), module docstring: Y = A*B and D = (A*B)*alpha + C*beta +
 *     X*x_factor, A is MxKxL, B is NxKxL, C/D/X/Y are MxNxL and share one
 *     major order; the epilogue function itself adds a relu that the
 *     docstring omits -- this oracle follows the docstring (no relu).
 *
 * Arithmetic: every input is decoded exactly to double (fp16, bf16, fp32 and
 * OCP FP8 E4M3/E5M2 all embed exactly in binary64; A and B may differ in type), the dot product is summed in
 * double in increasing k, the epilogue is evaluated in double, and results
 * are rounded once, round-to-nearest-even, to the output format.  The sum
 * of |a*b| is returned too: it scales the comparison bound; so, on request,
 * does the sum of the running sums' magnitudes at fixed chunk boundaries
 * (the bound of a half-precision accumulator, see entry()).
 *
 * Layout conventions (element strides; ld = leading dimension):
 *   A K-major : A(m,k,l) at (l*M + m)*lda + k        (lda >= K)
 *   A M-major : A(m,k,l) at (l*K + k)*lda + m        (lda >= M)
 *   B K-major : B(n,k,l) at (l*N + n)*ldb + k        (ldb >= K)
 *   B N-major : B(n,k,l) at (l*K + k)*ldb + n        (ldb >= N)
 *   C/X N-major: (l*M + m)*N + n;  M-major: (l*N + n)*M + m
 * Outputs are written in logical order [l][m][n].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Type codes of this oracle (its own numbering). */
/* OR_TF32: fp32 storage holding values representable in tf32; decoded like fp32. */
enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2, OR_E4M3 = 3, OR_E5M2 = 4, OR_TF32 = 5 };

/* ---------------------------------------------------------------- decoders */

/* IEEE 754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
static double decode_f16(uint32_t h) {
  int s = (h >> 15) & 1, e = (h >> 10) & 0x1F, f = h & 0x3FF;
  double v;
  if (e == 0)
    v = ldexp((double)f, -24);               /* subnormal: f * 2^-24 */
  else if (e == 31)
    v = f ? NAN : INFINITY;
  else
    v = ldexp(1.0 + f / 1024.0, e - 15);
  return s ? -v : v;
}

/* bfloat16: the upper half of binary32: 1 sign, 8 exponent (bias 127), 7 fraction. */
static double decode_bf16(uint32_t h) {
  int s = (h >> 15) & 1, e = (h >> 7) & 0xFF, f = h & 0x7F;
  double v;
  if (e == 0)
    v = ldexp((double)f, -133);              /* subnormal: f * 2^-133 */
  else if (e == 255)
    v = f ? NAN : INFINITY;
  else
    v = ldexp(1.0 + f / 128.0, e - 127);
  return s ? -v : v;
}

/* OCP 8-bit floating point, E4M3 variant: 1 sign, 4 exponent (bias 7),
 * 3 mantissa bits; no infinities; S.1111.111 is NaN; max normal 448. */
static double decode_e4m3(uint32_t b) {
  int s = (b >> 7) & 1, e = (b >> 3) & 0xF, f = b & 0x7;
  double v;
  if (e == 0)
    v = ldexp((double)f, -9);                /* subnormal: f/8 * 2^(1-7) */
  else if (e == 15 && f == 7)
    v = NAN;
  else
    v = ldexp(1.0 + f / 8.0, e - 7);
  return s ? -v : v;
}

/* OCP 8-bit floating point, E5M2 variant: 1 sign, 5 exponent (bias 15),
 * 2 mantissa bits; IEEE-like: exponent 31 is infinity (mantissa 0) or NaN;
 * subnormals m/4 * 2^(1-15). */
static double decode_e5m2(uint32_t b) {
  int s = (b >> 7) & 1, e = (b >> 2) & 0x1F, f = b & 0x3;
  double v;
  if (e == 0)
    v = ldexp((double)f, -16);               /* subnormal: f/4 * 2^-14 */
  else if (e == 31)
    v = f ? NAN : INFINITY;
  else
    v = ldexp(1.0 + f / 4.0, e - 15);
  return s ? -v : v;
}

static double decode_f32(uint32_t w) {
  float f;
  memcpy(&f, &w, 4);
  return (double)f;
}

static int elem_bytes(int dt) {
  switch (dt) {
    case OR_F32: return 4;
    case OR_TF32: return 4;
    case OR_F16: return 2;
    case OR_BF16: return 2;
    case OR_E4M3: return 1;
    case OR_E5M2: return 1;
  }
  return 0;
}

/* Decoded value of every 16-bit and 8-bit code, filled once from the
 * decoders above (a cache of the same function, nothing more). */
static double tab_f16[65536], tab_bf16[65536], tab_e4m3[256], tab_e5m2[256];
static int tabs_ready = 0;

static void build_tables(void) {
#ifdef _OPENMP
#pragma omp critical(oracle_tables)
#endif
  {
    if (!tabs_ready) {
      for (uint32_t c = 0; c < 65536; ++c) {
        tab_f16[c] = decode_f16(c);
        tab_bf16[c] = decode_bf16(c);
      }
      for (uint32_t c = 0; c < 256; ++c) {
        tab_e4m3[c] = decode_e4m3(c);
        tab_e5m2[c] = decode_e5m2(c);
      }
      tabs_ready = 1;
    }
  }
}

/* Decode element `idx` of a buffer of type `dt`. */
static double load_elem(const void* p, int dt, int64_t idx) {
  switch (dt) {
    case OR_F32:
    case OR_TF32: { uint32_t w; memcpy(&w, (const char*)p + 4 * idx, 4); return decode_f32(w); }
    case OR_F16: return tab_f16[((const uint16_t*)p)[idx]];
    case OR_BF16: return tab_bf16[((const uint16_t*)p)[idx]];
    case OR_E4M3: return tab_e4m3[((const uint8_t*)p)[idx]];
    case OR_E5M2: return tab_e5m2[((const uint8_t*)p)[idx]];
  }
  return NAN;
}

double oracle_decode(int dt, uint32_t code) {
  switch (dt) {
    case OR_F32:
    case OR_TF32: return decode_f32(code);
    case OR_F16: return decode_f16(code & 0xFFFF);
    case OR_BF16: return decode_bf16(code & 0xFFFF);
    case OR_E4M3: return decode_e4m3(code & 0xFF);
    case OR_E5M2: return decode_e5m2(code & 0xFF);
  }
  return NAN;
}

/* ---------------------------------------------------------------- rounding */

/* Round x to the nearest value with `mant` explicit fraction bits, minimum
 * normal exponent `emin`, round-half-to-even (nearbyint in the default
 * rounding mode).  Overflow handling is left to the caller. */
static double round_to_format(double x, int mant, int emin) {
  if (x == 0.0 || isnan(x) || isinf(x)) return x;
  int E;
  frexp(fabs(x), &E);              /* |x| = f * 2^E, f in [0.5, 1) */
  int e = E - 1;                   /* |x| in [2^e, 2^(e+1)) */
  if (e < emin) e = emin;          /* subnormal range: fixed quantum */
  double q = ldexp(1.0, e - mant); /* spacing of the format at |x| */
  return nearbyint(x / q) * q;     /* x/q is exact (power-of-two scale) */
}

static uint16_t encode_f16(double x) {
  uint16_t s = signbit(x) ? 0x8000 : 0;
  if (isnan(x)) return 0x7E00;
  double r = round_to_format(x, 10, -14);
  double a = fabs(r);
  if (a >= 65536.0) return s | 0x7C00; /* 2^16: past the largest finite (65504) */
  if (a == 0.0) return s;
  if (a < ldexp(1.0, -14)) return s | (uint16_t)(a / ldexp(1.0, -24));
  int E;
  double f = frexp(a, &E);         /* a = f*2^E, f in [0.5,1) */
  int e = E - 1;
  uint16_t frac = (uint16_t)((2.0 * f - 1.0) * 1024.0);
  return s | (uint16_t)((e + 15) << 10) | frac;
}

static uint16_t encode_bf16(double x) {
  uint16_t s = signbit(x) ? 0x8000 : 0;
  if (isnan(x)) return 0x7FC0;
  double r = round_to_format(x, 7, -126);
  double a = fabs(r);
  if (a >= ldexp(1.0, 128)) return s | 0x7F80;
  if (a == 0.0) return s;
  if (a < ldexp(1.0, -126)) return s | (uint16_t)(a / ldexp(1.0, -133));
  int E;
  double f = frexp(a, &E);
  int e = E - 1;
  uint16_t frac = (uint16_t)((2.0 * f - 1.0) * 128.0);
  return s | (uint16_t)((e + 127) << 7) | frac;
}

/* Round n doubles once, RNE, into the storage format `dt` (F32/F16/BF16). */
void oracle_round(int dt, const double* in, int64_t n, void* out) {
  for (int64_t i = 0; i < n; ++i) {
    switch (dt) {
      case OR_F32: { float f = (float)in[i]; memcpy((char*)out + 4 * i, &f, 4); break; }
      case OR_F16: ((uint16_t*)out)[i] = encode_f16(in[i]); break;
      case OR_BF16: ((uint16_t*)out)[i] = encode_bf16(in[i]); break;
    }
  }
}

/* ---------------------------------------------------------------- the GEMM */

typedef struct {
  int64_t M, N, K, L;
  const void* A; int64_t lda; int a_mn_major;
  const void* B; int64_t ldb; int b_mn_major;
  const void* C; const void* X;
  int a_dt, b_dt, c_dt, x_dt, cd_m_major;
  double alpha, beta, xf;
  int use_c, use_x, relu;
  int64_t acc_chunk;  /* > 0: also report sum_j |partial sum after chunk j| (see entry) */
} oracle_problem;

static int64_t a_index(const oracle_problem* p, int64_t m, int64_t k, int64_t l) {
  return p->a_mn_major ? (l * p->K + k) * p->lda + m : (l * p->M + m) * p->lda + k;
}
static int64_t b_index(const oracle_problem* p, int64_t n, int64_t k, int64_t l) {
  return p->b_mn_major ? (l * p->K + k) * p->ldb + n : (l * p->N + n) * p->ldb + k;
}
static int64_t cd_index(const oracle_problem* p, int64_t m, int64_t n, int64_t l) {
  return p->cd_m_major ? (l * p->N + n) * p->M + m : (l * p->M + m) * p->N + n;
}

/* One output entry, straight from the definition.
 *
 * With acc_chunk = c > 0 it also returns, in *pp, the sum over the chunk
 * boundaries k = c, 2c, ... and k = K (the last, possibly shorter, chunk) of
 * the magnitude of the exact running sum |sum_{k' < k} a*b|.  A half-precision
 * accumulator is rounded once per tensor-core instruction, i.e. at these
 * boundaries (the cuBLASDx Blackwell page: a `half` accumulator for `half`
 * and fp8 inputs, one instruction consuming 16 K of 16-bit or 32 K of 8-bit
 * inputs), and each such rounding errs by at most half an fp16 ulp of the
 * running sum: this sum scales that part of the comparison bound.  It is not
 * part of the result. */
static void entry(const oracle_problem* p, int64_t m, int64_t n, int64_t l,
                  const double* arow, double* d, double* y, double* s, double* pp) {
  double acc = 0.0, sabs = 0.0, pabs = 0.0;
  for (int64_t k = 0; k < p->K; ++k) {
    double a = arow ? arow[k] : load_elem(p->A, p->a_dt, a_index(p, m, k, l));
    double b = load_elem(p->B, p->b_dt, b_index(p, n, k, l));
    acc += a * b;
    sabs += fabs(a * b);
    if (p->acc_chunk > 0 && ((k + 1) % p->acc_chunk == 0 || k + 1 == p->K)) pabs += fabs(acc);
  }
  double dv = p->alpha * acc;
  if (p->use_c) dv += p->beta * load_elem(p->C, p->c_dt, cd_index(p, m, n, l));
  /* relu variant ("custom_epilogue_dense_gemm.py", epilogue() function):
   * the rectifier applies to alpha*acc + beta*C, before X is added. */
  if (p->relu && dv < 0.0) dv = 0.0;
  if (p->use_x) dv += p->xf * load_elem(p->X, p->x_dt, cd_index(p, m, n, l));
  *d = dv;
  *y = acc;
  if (s) *s = sabs;
  if (pp) *pp = pabs;
}

static void fill_problem(oracle_problem* p, int64_t M, int64_t N, int64_t K, int64_t L,
                         const void* A, int64_t lda, int a_mn, const void* B, int64_t ldb,
                         int b_mn, const void* C, const void* X, int a_dt, int b_dt, int c_dt,
                         int x_dt, int cd_m_major, double alpha, double beta, double xf,
                         int use_c, int use_x, int relu, int64_t acc_chunk) {
  p->M = M; p->N = N; p->K = K; p->L = L;
  p->A = A; p->lda = lda; p->a_mn_major = a_mn;
  p->B = B; p->ldb = ldb; p->b_mn_major = b_mn;
  p->C = C; p->X = X;
  p->a_dt = a_dt; p->b_dt = b_dt; p->c_dt = c_dt; p->x_dt = x_dt; p->cd_m_major = cd_m_major;
  p->alpha = alpha; p->beta = beta; p->xf = xf;
  p->use_c = use_c && C != NULL;
  p->use_x = use_x && X != NULL;
  p->relu = relu;
  p->acc_chunk = acc_chunk;
}

/* Rows [m0, m1) of every batch, all columns.  D, Y, S, P are [L][m1-m0][N]
 * (S and P may be NULL; P is filled when acc_chunk > 0).  Returns 0, or -1
 * on a bad argument. */
int oracle_gemm_rows(int64_t M, int64_t N, int64_t K, int64_t L,
                     const void* A, int64_t lda, int a_mn, const void* B, int64_t ldb, int b_mn,
                     const void* C, const void* X, int a_dt, int b_dt, int c_dt, int x_dt,
                     int cd_m_major, double alpha, double beta, double xf, int use_c, int use_x,
                     int relu, int64_t acc_chunk, int64_t m0, int64_t m1, double* D, double* Y,
                     double* S, double* P, int nthreads) {
  if (M < 0 || N < 0 || K < 0 || L < 0 || m0 < 0 || m1 > M || m0 > m1) return -1;
  if (acc_chunk < 0) return -1;
  if (elem_bytes(a_dt) == 0 || elem_bytes(b_dt) == 0) return -1;
  build_tables();
  oracle_problem p;
  fill_problem(&p, M, N, K, L, A, lda, a_mn, B, ldb, b_mn, C, X, a_dt, b_dt, c_dt, x_dt,
               cd_m_major, alpha, beta, xf, use_c, use_x, relu, acc_chunk);
  int64_t rows = m1 - m0;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel
#endif
  {
    double* arow = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
    for (int64_t lm = 0; lm < L * rows; ++lm) {
      int64_t l = lm / rows, m = m0 + lm % rows;
      for (int64_t k = 0; k < K; ++k) arow[k] = load_elem(A, a_dt, a_index(&p, m, k, l));
      for (int64_t n = 0; n < N; ++n) {
        int64_t o = (l * rows + (m - m0)) * N + n;
        entry(&p, m, n, l, arow, &D[o], &Y[o], S ? &S[o] : NULL,
              P && acc_chunk > 0 ? &P[o] : NULL);
      }
    }
    free(arow);
  }
  return 0;
}

/* Selected entries (ms[i], ns[i], ls[i]), i < count. */
int oracle_gemm_entries(int64_t M, int64_t N, int64_t K, int64_t L,
                        const void* A, int64_t lda, int a_mn, const void* B, int64_t ldb, int b_mn,
                        const void* C, const void* X, int a_dt, int b_dt, int c_dt, int x_dt,
                        int cd_m_major, double alpha, double beta, double xf, int use_c, int use_x,
                        int relu, int64_t acc_chunk, const int64_t* ms, const int64_t* ns,
                        const int64_t* ls, int64_t count, double* D, double* Y, double* S,
                        double* P, int nthreads) {
  if (elem_bytes(a_dt) == 0 || elem_bytes(b_dt) == 0) return -1;
  if (acc_chunk < 0) return -1;
  for (int64_t i = 0; i < count; ++i)
    if (ms[i] < 0 || ms[i] >= M || ns[i] < 0 || ns[i] >= N || ls[i] < 0 || ls[i] >= L) return -1;
  build_tables();
  oracle_problem p;
  fill_problem(&p, M, N, K, L, A, lda, a_mn, B, ldb, b_mn, C, X, a_dt, b_dt, c_dt, x_dt,
               cd_m_major, alpha, beta, xf, use_c, use_x, relu, acc_chunk);
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16)
#endif
  for (int64_t i = 0; i < count; ++i)
    entry(&p, ms[i], ns[i], ls[i], NULL, &D[i], &Y[i], S ? &S[i] : NULL,
          P && acc_chunk > 0 ? &P[i] : NULL);
  return 0;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
