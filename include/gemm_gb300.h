/*
 * gemm_gb300.h -- C ABI of the GB300 (sm_103a) persistent batched GEMM with a
 * fused custom epilogue.
 *
 * Operation (for every batch l < L, row m < M, column n < N):
 *
 *     acc       = sum_k A(m,k,l) * B(n,k,l)        fp32 accumulation
 *     Y(m,n,l)  = acc                              (optional output)
 *     D(m,n,l)  = alpha*acc + beta*C(m,n,l) + x_factor*X(m,n,l)   (fp32 epilogue)
 *
 * Sources: "custom_epilogue_dense_gemm.py" (CuTeDSL Blackwell example), module
 * docstring "Y = A * B", "D = (A * B) * alpha + C * beta + X * x_factor", its
 * "Tensor dimensions" list (A is MxKxL, B is NxKxL, C/D/X/Y are MxNxL and share
 * one major order) and its "Constraints" list (A and B share one type; the
 * contiguous dimension of every tensor is 16-byte aligned);
 * "04_mma_tma_2sm_sm100.cu" (CuTe Blackwell tutorial 04), header comment
 * "D (f32) = beta * C (F32) + alpha * A (F16) * B (F16)".
 *
 * Memory: every tensor pointer is a DEVICE pointer on the handle's device,
 * owned by the caller; the library never allocates, frees or retains them.
 *
 * Layouts (element strides; ld = leading dimension in elements):
 *   A, GEMM_K_MAJOR : A(m,k,l) at (l*M + m)*lda + k      (lda >= K)
 *   A, GEMM_MN_MAJOR: A(m,k,l) at (l*K + k)*lda + m      (lda >= M)
 *   B, GEMM_K_MAJOR : B(n,k,l) at (l*N + n)*ldb + k      (ldb >= K)
 *   B, GEMM_MN_MAJOR: B(n,k,l) at (l*K + k)*ldb + n      (ldb >= N)
 *   C/D/X/Y are packed; dtypes->cdxy_major selects
 *     GEMM_K_MAJOR (row-major, "N-major"): (l*M + m)*N + n
 *     GEMM_MN_MAJOR (column-major, "M-major"): (l*N + n)*M + m
 *
 * Errors: validation happens on the host before anything is enqueued and is
 * reported synchronously by the return code.  gemm_run never synchronises;
 * a device-side watchdog (a bounded wait on every pipeline barrier) records a
 * timeout in a status word that gemm_sync_status reads.
 */
#ifndef GEMM_GB300_H
#define GEMM_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* the CUDA runtime's cudaStream_t is `struct CUstream_st*` */

typedef struct gemm_handle* gemm_handle_t;

typedef enum {
  GEMM_OK = 0,
  GEMM_ERR_INVALID_ARG = 1,        /* bad shape, NULL where required, bad enum, bad ld */
  GEMM_ERR_UNSUPPORTED_DTYPE = 2,  /* type combination not implemented */
  GEMM_ERR_MISALIGNED = 3,         /* pointer or leading dimension not 16-byte aligned */
  GEMM_ERR_UNSUPPORTED_ARCH = 4,   /* device is not compute capability 10.3 */
  GEMM_ERR_CUDA = 5,               /* a CUDA runtime/driver call failed */
  GEMM_ERR_DEVICE_TIMEOUT = 6,     /* a kernel pipeline wait exceeded its limit */
  GEMM_ERR_UNSUPPORTED_CONFIG = 7, /* a forced kernel configuration cannot run this problem */
  GEMM_ERR_DEVICE_CHECK = 8        /* debug library only: a device-side bounds check failed */
} gemm_status_t;

/* GEMM_TF32: fp32 storage read by the tensor core at tf32 precision (sign,
 * exponent and the upper 10 fraction bits; A and B must be K-major).  Any fp32
 * bit pattern is accepted.  Values that are tf32 values (low 13 fraction bits
 * zero) are exact inputs and the result meets the fp32-input bound; for other
 * values each operand is off by less than 2^-10 relative, each product by
 * less than 2^-9 + 2^-20, and the accumulator bound grows by that term:
 * |acc - exact| <= (2^-9 + 2^-20 + 2^-10) * sum_k |a*b|. */
typedef enum {
  GEMM_F32 = 0, GEMM_F16 = 1, GEMM_BF16 = 2, GEMM_E4M3 = 3, GEMM_E5M2 = 4, GEMM_TF32 = 5
} gemm_dtype_t;

/* Epilogue variants ("custom_epilogue_dense_gemm.py": the docstring's linear
 * form, and the relu its epilogue() function applies before X is added). */
typedef enum {
  GEMM_EPI_LINEAR = 0,   /* D = alpha*acc + beta*C + x_factor*X */
  GEMM_EPI_RELU = 1      /* D = max(alpha*acc + beta*C, 0) + x_factor*X */
} gemm_epilogue_t;

typedef enum { GEMM_K_MAJOR = 0, GEMM_MN_MAJOR = 1 } gemm_layout_t;

/* Per-call descriptor of types and epilogue.
 *   ab: A's type, F16, BF16, E4M3, E5M2 or TF32 (and B's, unless b is set).
 *   c, x: F32, F16 or BF16 (inputs).  d, y: F32, F16 or BF16 (outputs).
 *   cdxy_major: the one major order of C, D, X and Y.
 *   b: B's type when it differs from A's -- only fp8 pairs (E4M3 x E5M2 in
 *      either order, which tcgen05 kind::f8f6f4 takes); 0 (GEMM_F32) = same as ab.
 *   epilogue: GEMM_EPI_LINEAR (0) or GEMM_EPI_RELU.
 *   acc: the tensor-core accumulator, GEMM_F32 (0, the default) or GEMM_F16.
 *      F16 is taken for F16, E4M3 and E5M2 inputs only (the cuBLASDx
 *      Blackwell page: half inputs with a half or float accumulator, fp8 with
 *      half or float, bfloat16 and tf32 with float); otherwise the call
 *      returns GEMM_ERR_UNSUPPORTED_DTYPE.  An F16 accumulator is rounded to
 *      fp16 once per tensor-core instruction (every 16 K of 16-bit inputs,
 *      32 K of 8-bit) and overflows to infinity past 65504; Y is that fp16
 *      value and the epilogue still runs in fp32. */
typedef struct {
  gemm_dtype_t ab, c, d, x, y;
  gemm_layout_t cdxy_major;
  gemm_dtype_t b;
  gemm_epilogue_t epilogue;
  gemm_dtype_t acc;
} gemm_dtypes_t;

/* Kernel configuration.  Chosen automatically per problem shape unless the
 * handle has one forced (gemm_set_config).
 *   cta_group   1: each CTA owns a 128 x tile_n output tile (tcgen05 cta_group::1)
 *               2: a CTA pair owns a 256 x tile_n tile (tcgen05 cta_group::2);
 *                  each CTA stages 128 rows of A and tile_n/2 rows of B.
 *   tile_n      output tile width of one CTA group: 64 to 256 in steps of 32
 *               (the custom-epilogue example's "Constraints": MMA tile N a
 *               multiple of 32 up to 256; 32 itself is not offered).
 *   stages      depth of the shared-memory A/B ring (0 = as deep as fits).
 *   group_m     tile rasterisation: tiles are walked in column strips
 *               group_m tiles high, odd strips from the last column back;
 *               odd waves of tiles also walk K from the last k-block down
 *               (fp32 accumulators), so each wave starts on the operand
 *               blocks the previous one read last (0 = automatic: 12).
 *   cluster_m   CTA groups per thread-block cluster stacked along M, sharing
 *               their B columns through TMA multicast: 1 or 2.
 *   cluster_n   (after tail_split) CTA groups per cluster side by side along N,
 *               sharing their A rows through TMA multicast: 1 or 2.  The
 *               cluster holds cta_group * cluster_m * cluster_n CTAs.  As an
 *               input, both 0 = automatic; either non-zero fixes the shape (0
 *               counting as 1).  Multicast clusters are built only into the
 *               single-GPU library (libgemm_gb300.so); the library for
 *               processes that drive several GPUs (libgemm_gb300_nomc.so)
 *               returns GEMM_ERR_UNSUPPORTED_CONFIG for them.
 *   epi_slots   (also an input) epilogue slots, 2..6 (0 = automatic).
 *   epi_warps   (after cluster_n; also an input) epilogue warps per 32-lane
 *               quarter of the tensor-memory accumulator: 1 (4 epilogue warps,
 *               192 threads a CTA) or 2 (8 warps, 320 threads; the two warps
 *               of a quarter take its 32-column chunks alternately, each with
 *               half the epilogue slots; clusters of one CTA group only).
 *               0 = automatic: 2 where the tiles fit in one wave or the
 *               epilogue takes at least as long as the main loop, else 1.
 *   stream_k    (after epi_warps) when the tiles fill less than one wave of
 *               resident clusters, every cluster takes an equal contiguous
 *               share of all the tiles' k-blocks; the owner of a tile (the
 *               cluster holding its last k-block) adds the fp32 partial sums of
 *               its earlier k-blocks, in cluster order, before its epilogue.
 *               fp32 accumulators and clusters of one CTA group only; the
 *               partials go through a workspace the handle allocates at
 *               creation (gemm_run_noalloc never uses it).  As an input:
 *               0 = automatic, 1 = never, 2 = wherever allowed.  As an output:
 *               the number of clusters sharing the k-blocks (0 = off).
 *   Fields marked "diagnostic" are for tuning and testing the kernel, not
 *   part of the GEMM contract; leave them 0.
 *   l2_hints    (diagnostic; also an input) L2 eviction priority of the TMA
 *               copies, 2 bits
 *               each (0 normal, 1 evict-last, 2 evict-first): bits 0-1 A/B
 *               loads, 2-3 C/X loads, 4-5 D/Y stores.  As an input it applies
 *               only with bit 8 set (0 = automatic).
 *   epi_wait_ns (diagnostic; also an input) suspend-time hint, in ns, of the epilogue's
 *               wait for a finished accumulator; as an input, value + 1
 *               (0 = automatic, 1 = no hint).
 *   tail_split  tiles of the last, partial wave run as two half-width (tile_n/2)
 *               items each, so that wave takes about half as long; reports how
 *               many tiles were split.  As an input: 0 = automatic (split when the
 *               partial wave fills at most half the clusters), 1 = never.
 *   inject_stall  (diagnostic input, tests of the watchdog only) non-zero: the MMA warp
 *               first waits on a barrier nothing ever arrives at, so every launch
 *               ends through the watchdog with GEMM_ERR_DEVICE_TIMEOUT (role 6 in
 *               the status word) after the configured timeout.
 * Filled in by gemm_plan / reported by gemm_last_config:
 *   tile_m      128 * cta_group (rows of one CTA group's tile).
 *   tile_k      K elements per ring stage: one or two 128-byte swizzle atoms (64
 *               or 128 K for 16-bit inputs, 128 or 256 for 8-bit); two unless the
 *               tile is a single CTA's and wider than 128.
 *   acc_stages  tensor-memory accumulator stages (2: double buffered).
 *   ring_bytes  ring bytes per CTA: stages*(A stage + B stage) + 8 bytes per
 *               mbarrier (2 per stage, 2 per accumulator stage) + 4 bytes of
 *               tensor-memory address.
 *   epi_slots   epilogue shared-memory slots: C/X sub-tiles (128 rows x 32
 *               columns) are TMA-loaded epi_slots-1 chunks ahead (with two
 *               epilogue warps per quarter each warp has epi_slots/2 of them and
 *               loads that many minus one of its own chunks ahead, at least
 *               one); D/Y are staged in the same slot and TMA-stored.
 *   epi_slot_bytes  bytes of one epilogue slot.
 *   smem_bytes  dynamic shared memory per CTA (ring + epilogue slots + their
 *               barriers + alignment slack).
 *   tiles       number of output tiles; grid_ctas: CTAs launched. */
typedef struct {
  int cta_group, tile_n, stages, group_m;
  int tile_m, tile_k, acc_stages;
  int ring_bytes, smem_bytes;
  int64_t tiles;
  int grid_ctas;
  int epi_slots, epi_slot_bytes;
  int cluster_m;
  int l2_hints;
  int epi_wait_ns;
  int inject_stall;
  int tail_split;
  int cluster_n;
  int epi_warps;
  int stream_k;
} gemm_config_t;

/* Every argument of one gemm_run call, for the host-only planning calls. */
typedef struct {
  int64_t M, N, K, L;
  const void* A; int64_t lda; gemm_layout_t layoutA;
  const void* B; int64_t ldb; gemm_layout_t layoutB;
  const void* C; const void* X; void* D; void* Y;
  float alpha, beta, x_factor;
  gemm_dtypes_t dtypes;
} gemm_problem_t;

/* Create a handle for CUDA device `device`.  Checks the device is compute
 * capability 10.3 (GEMM_ERR_UNSUPPORTED_ARCH otherwise), caches its SM count
 * and shared-memory limit, resolves cuTensorMapEncodeTiled through the runtime
 * and allocates a 4-byte device status word and the stream-K workspace (one
 * 128 x 256 fp32 partial slot and one flag per SM: 20 MB on 152 SMs; if that
 * allocation fails the handle works without stream-K).  No later call on the
 * handle allocates device memory except gemm_run_host (its staging buffers).
 * *out is NULL on failure. */
gemm_status_t gemm_create(gemm_handle_t* out, int device);

/* Release the handle, its status word and its host-call workspace.  NULL is
 * accepted (no-op).  Work already enqueued with this handle must be complete. */
gemm_status_t gemm_destroy(gemm_handle_t h);

/* Enqueue D = alpha*(A*B) + beta*C + x_factor*X (and Y = A*B) on `stream`.
 *
 * M, N, K, L >= 0.  M, N or L == 0: nothing to do, returns GEMM_OK.
 * K == 0: acc = 0, so D = beta*C + x_factor*X and Y = 0.
 * A, B: required when K > 0.  lda/ldb as in the layout table above, and
 *   lda*sizeof(ab), ldb*sizeof(ab) multiples of 16 bytes.
 * C: read only when beta != 0 (then required); otherwise may be NULL.
 * X: read only when X != NULL and x_factor != 0.
 * D: required.  Y: written when non-NULL.
 * Every non-NULL pointer 16-byte aligned; the packed leading dimension of
 *   C/D/X/Y (N for row-major, M for column-major) times the element size a
 *   multiple of 16 bytes.
 * Aliasing: D may equal C when they have the same type (each element of C is
 *   read before the same element of D is written); any other overlap between
 *   an output and any tensor is undefined.
 * Asynchronous: returns once the kernel is enqueued; never synchronises.
 * The calling thread's current device must be the handle's device. */
gemm_status_t gemm_run(gemm_handle_t h, int64_t M, int64_t N, int64_t K, int64_t L,
                       const void* A, int64_t lda, gemm_layout_t layoutA,
                       const void* B, int64_t ldb, gemm_layout_t layoutB,
                       const void* C, const void* X, void* D, void* Y,
                       float alpha, float beta, float x_factor,
                       const gemm_dtypes_t* dtypes, struct CUstream_st* stream);

/* The same GEMM on HOST buffers.  A, B, C, X are read from host memory and D,
 * Y written back to host memory through a device workspace the handle owns:
 * on `stream`, in order, the inputs are copied to the device (each tensor's
 * element span, from its first to its last element), the GEMM runs on the
 * copies, and D and Y are copied back.  Returns once all of it is enqueued.
 *
 * Arguments, layouts, validation and result are gemm_run's (alignment is
 * checked on the host pointers).  The host buffers must stay valid, inputs
 * unmodified and outputs unread, until `stream` has passed the call
 * (gemm_sync_status, or a stream synchronisation).  Page-locked (pinned) host
 * memory lets the copies run asynchronously and overlap other streams;
 * pageable memory works, with copies that synchronise with the host.
 *
 * The workspace grows to the largest call seen (cudaMalloc, which
 * synchronises the device) and is freed by gemm_destroy.  Calls on one handle
 * share it, so they must be ordered (one stream, or synchronised); to overlap
 * calls, use one handle per stream.  Copy failures return GEMM_ERR_CUDA. */
gemm_status_t gemm_run_host(gemm_handle_t h, int64_t M, int64_t N, int64_t K, int64_t L,
                            const void* A, int64_t lda, gemm_layout_t layoutA,
                            const void* B, int64_t ldb, gemm_layout_t layoutB,
                            const void* C, const void* X, void* D, void* Y,
                            float alpha, float beta, float x_factor,
                            const gemm_dtypes_t* dtypes, struct CUstream_st* stream);

/* Diagnostic, not part of the GEMM contract.  Ring statistics, for studying
 * the kernel's pipeline (no counterpart on the pages).  Only the statistics build of the library (libgemm_gb300_stats.so,
 * compiled with GB300_RING_STATS=1; the product library returns
 * GEMM_ERR_UNSUPPORTED_CONFIG) counts, in each CTA of the last launch, the
 * clock cycles its roles spend waiting on the pipeline's barriers.  The call
 * synchronises `stream`, then copies min(grid CTAs, max_ctas) blocks of
 * GEMM_RING_STAT_WORDS counters to `out` (CTA-major) and stores the count in
 * *n_ctas.  Counters, in order: MMA issuer waiting for a stage to land,
 * waiting for a free accumulator stage, its whole loop, stages issued (these
 * four are zero in the non-leader CTA of a pair); producer waiting for a
 * stage to drain, its whole loop; epilogue store thread waiting for a
 * finished accumulator, waiting for C/X to land, its whole loop, the CTA's
 * epilogue chunks, then three parts of the store thread's chunk loop: from
 * C/X landing to C/X and accumulator columns in registers, computing D and Y
 * into shared memory, issuing the stores and next loads (with their wait);
 * the chunks the store thread's warp processed (the CTA's chunks with one
 * epilogue warp per lane quarter, about half of them with two); two spare
 * words. */
#define GEMM_RING_STAT_WORDS 16
gemm_status_t gemm_ring_stats(gemm_handle_t h, struct CUstream_st* stream, uint64_t* out,
                              int max_ctas, int* n_ctas);

/* Synchronise `stream`, then read and clear the handle's device status word.
 * Returns GEMM_ERR_DEVICE_TIMEOUT if any kernel since the last call hit its
 * watchdog, GEMM_ERR_DEVICE_CHECK if (debug library, libgemm_gb300_debug.so,
 * built with GB300_DEBUG=1) a device-side bounds check failed -- a TMA box
 * outside its shared-memory slot, a TMA coordinate that is not 16-byte
 * aligned or a store starting below zero, a tensor-memory column range past
 * its accumulator stage; the access was skipped and the status word holds
 * 0xD0CCBBBB, CC the check -- GEMM_ERR_CUDA if the stream reported an error,
 * else GEMM_OK.
 * *detail (optional; may be NULL) receives the raw status word (0 when
 * clean): an extension of the two-argument call, carrying the watchdog's
 * record 0xE0RRBBBB (RR the waiting role: 1 producer, 2 MMA waiting for
 * operands, 3 MMA waiting for an accumulator, 4 epilogue waiting for an
 * accumulator, 5 epilogue waiting for C/X, 6 injected stall, 7 stream-K
 * partial sums; BBBB the low bits of the block).  After an error the call
 * also clears the handle's stream-K flags. */
gemm_status_t gemm_sync_status(gemm_handle_t h, struct CUstream_st* stream, uint32_t* detail);

/* Human-readable name of a status code (static storage). */
const char* gemm_status_string(gemm_status_t s);

/* Host-only validation of one call's arguments, exactly as gemm_run performs
 * it (no device access; pointers are checked for NULL and alignment only). */
gemm_status_t gemm_check(const gemm_problem_t* p);

/* Host-only kernel configuration for problem `p` on a device with `sm_count`
 * SMs and `smem_optin` bytes of opt-in shared memory per block.  `forced`
 * (may be NULL) fixes cta_group/tile_n/stages/group_m; zero fields are
 * chosen automatically.  Returns GEMM_ERR_UNSUPPORTED_CONFIG when a forced
 * configuration cannot run the problem. */
gemm_status_t gemm_plan(const gemm_problem_t* p, int sm_count, int smem_optin,
                        const gemm_config_t* forced, gemm_config_t* out);

/* Force a kernel configuration for later gemm_run calls on this handle
 * (NULL restores automatic selection).  Used by tests and tuning sweeps. */
gemm_status_t gemm_set_config(gemm_handle_t h, const gemm_config_t* cfg);

/* The configuration chosen by the most recent successful gemm_run. */
gemm_status_t gemm_last_config(gemm_handle_t h, gemm_config_t* out);

/* Tensor-memory columns one fp32 accumulator of tile_m x tile_n occupies:
 * tile_m/128 blocks when tile_m is a multiple of 128, else tile_m/64 blocks,
 * times tile_n columns (the fit rule of the cuBLASDx Blackwell pipeline card,
 * "Size" bullet: 512 columns per SM).  0 for an invalid tile. */
int gemm_tmem_columns(int tile_m, int tile_n);

/* Watchdog limit for every pipeline wait of later launches, in nanoseconds
 * (0 restores the default of 4 seconds). */
gemm_status_t gemm_set_timeout_ns(gemm_handle_t h, uint64_t ns);

/* gemm_run without allocating anything: for callers that must not call
 * cudaMalloc -- code paths under a framework's memory pool that owns all of
 * the device's memory, latency-critical loops where cudaMalloc's device-wide
 * synchronisation would stall other work, and environments that forbid
 * dynamic allocation after start-up.  (The pages have no counterpart: this
 * is a library-level addition.)
 *
 * Same arguments, layouts, validation and result as gemm_run, but without a
 * handle: it runs on the calling thread's current device.  The kernel's one
 * piece of scratch memory, its 4-byte watchdog status word, lives in a
 * file-scope device array of 64 words (256 bytes) that every GPU loading the
 * library holds until the process exits; a call needs one word whatever the
 * problem size, and a call needing more than the array holds would be
 * rejected with GEMM_ERR_INVALID_ARG.
 *
 * The first call on a device does a one-time set-up there (device checks,
 * tensor-map encoder, the array's device address); make that first call
 * before any stream capture.  Each call clears the status word on `stream`
 * before its launch.  Every call shares the array, so calls that overlap on
 * the GPU (different streams, no ordering between them) race on the status
 * word: one may clear or report the other's watchdog record.
 *
 * watchdog_out NULL: asynchronous, like gemm_run; a watchdog record of that
 * launch is then never reported (there is no handle to read it with, and the
 * next call clears the word before its own launch).  Non-NULL: the call
 * synchronises `stream` (only that stream), stores the status word there and
 * returns GEMM_ERR_DEVICE_TIMEOUT if it is non-zero; pass NULL while
 * `stream` is being captured into a graph, since a synchronisation would end
 * the capture. */
gemm_status_t gemm_run_noalloc(int64_t M, int64_t N, int64_t K, int64_t L,
                               const void* A, int64_t lda, gemm_layout_t layoutA,
                               const void* B, int64_t ldb, gemm_layout_t layoutB,
                               const void* C, const void* X, void* D, void* Y,
                               float alpha, float beta, float x_factor,
                               const gemm_dtypes_t* dtypes, struct CUstream_st* stream,
                               uint32_t* watchdog_out);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_GB300_H */
