/*
 * gb300_gemm.h -- C ABI of the FP32 GEMM library for one NVIDIA GB300
 * (sm_103a).  Shared library: libgb300gemm.so.
 *
 * The operation is the dense single-precision matrix multiply of the
 * tiled-matmul course page ("Project - tiled matrix multiply": row-major
 * float matrices, C = A * B, 2*M*N*K FLOP of work), generalised with the
 * alpha/beta scaling of the cuBLAS SGEMM call shown in that page's section
 * "Stage 3 - the reference ceiling: cuBLAS":
 *
 *     C <- alpha * A * B + beta * C
 *
 * Storage is row-major throughout:
 *     A(i,k) = A[i*lda + k]   (M x K, lda >= K)
 *     B(k,j) = B[k*ldb + j]   (K x N, ldb >= N)
 *     C(i,j) = C[i*ldc + j]   (M x N, ldc >= N)
 *
 * Conventions shared by every call:
 *   - All matrix pointers are DEVICE pointers (cudaMalloc'd or from a
 *     framework allocator) on the current CUDA device; the caller owns them.
 *   - Calls that take a stream only enqueue work on it and return; results
 *     are ready after the caller synchronises that stream.  Launch errors are
 *     returned; errors raised while kernels run surface at the caller's
 *     synchronisation, and bounded-wait timeouts inside the tensor-core
 *     kernel are reported by gemm_check_status().
 *   - The library never exits the process; every call returns a status code
 *     (GEMM_OK or a negative GEMM_ERR_*).  gemm_strerror() describes it.
 *   - C must not overlap A or B (as in BLAS); the result is undefined if it
 *     does.
 */
#ifndef GB300_GEMM_H
#define GB300_GEMM_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define GEMM_API __attribute__((visibility("default")))
#else
#define GEMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* 2: gemm_plan_t gained b_split_in_kernel (callers built against version 1
 * pass a smaller struct to gemm_f32_plan / gemm_f32_op_plan). */
#define GEMM_ABI_VERSION 2

/* ---- status codes ---------------------------------------------------- */
#define GEMM_OK 0
#define GEMM_ERR_INVALID_ARG (-1)        /* null pointer, negative size, ld too small, unknown mode */
#define GEMM_ERR_UNSUPPORTED (-2)        /* mode not available for this device or shape */
#define GEMM_ERR_CUDA (-3)               /* a CUDA runtime call or a launch failed */
#define GEMM_ERR_DEVICE_TIMEOUT (-4)     /* a kernel's bounded wait ran out (see gemm_check_status) */
#define GEMM_ERR_WORKSPACE_TOO_SMALL (-5)/* caller workspace smaller than the plan needs */
#define GEMM_ERR_NO_DEVICE (-6)          /* no CUDA device visible */

/* ---- modes -------------------------------------------------------------
 * AUTO picks per shape (gemm_f32_plan tells which).  FP32_SIMT runs on the
 * CUDA cores in IEEE FP32 FMA arithmetic.  TF32X3 runs on the tcgen05
 * tensor cores with each operand split into a TF32 high part and a TF32
 * low part, D = Ahi*Bhi + Ahi*Blo + Alo*Bhi, accumulated in FP32 (FP32
 * accuracy; not bitwise equal to FP32_SIMT).  TF32 is one TF32 MMA per
 * product (operands rounded to TF32, 11 significant bits; FP32
 * accumulation): about three times the 3xTF32 rate, TF32-accurate only
 * (error up to about 2^-10 of sum |A||B|).  Non-finite inputs: NaN
 * propagates in every mode; an Inf gives the IEEE +-Inf on the CUDA cores
 * but NaN in the TF32 modes (the split puts Inf against a zero part of the
 * other operand, and Inf * 0 = NaN).  The remaining modes are the
 * course page's ladder kernels ("Stage 0" naive with x -> row, "Stage 1"
 * coalesced with x -> column, "Stage 2" shared-memory tiles of 16 or 32),
 * kept for comparison. */
#define GEMM_MODE_AUTO 0
#define GEMM_MODE_FP32_SIMT 1
#define GEMM_MODE_TF32X3 2
#define GEMM_MODE_TF32 3
#define GEMM_MODE_NAIVE 10
#define GEMM_MODE_COALESCED 11
#define GEMM_MODE_TILED16 12
#define GEMM_MODE_TILED32 13

/* kernel identifiers reported by gemm_f32_plan */
#define GEMM_KERNEL_NONE 0          /* nothing to launch (M or N is 0) */
#define GEMM_KERNEL_SCALE 1         /* K == 0 (or a call with alpha == 0): C <- beta*C only */
#define GEMM_KERNEL_NAIVE 2
#define GEMM_KERNEL_COALESCED 3
#define GEMM_KERNEL_TILED 4
#define GEMM_KERNEL_SIMT 5          /* register-tiled CUDA-core SGEMM */
#define GEMM_KERNEL_TC_TF32X3 6     /* tcgen05 3xTF32 */
#define GEMM_KERNEL_TC_TF32 7       /* tcgen05 1xTF32 */

/* governing roof predicted by the planner */
#define GEMM_BOUND_FP32 1           /* FP32 CUDA-core FMA peak */
#define GEMM_BOUND_TF32X3 2         /* one third of the dense TF32 tensor peak */
#define GEMM_BOUND_HBM 3            /* HBM bandwidth */
#define GEMM_BOUND_TF32 4           /* the dense TF32 tensor peak */

typedef struct gemm_plan {
  int32_t mode;            /* resolved mode, never GEMM_MODE_AUTO */
  int32_t kernel;          /* GEMM_KERNEL_* */
  int32_t bm, bn, bk;      /* CTA tile */
  int32_t stages;          /* shared-memory pipeline depth */
  int32_t split_k;         /* K slices; > 1 uses the workspace and a reduction */
  int32_t vec;             /* 1: 128-bit global access path, 0: scalar path */
  int32_t a_split_in_kernel; /* tensor-core modes: A split inside the GEMM kernel (1) or by a pre-pass (0) */
  int32_t bound;           /* GEMM_BOUND_* */
  int32_t threads;         /* threads per CTA */
  int32_t launches;        /* kernels one call launches (split pass, main, reduction) */
  int64_t grid_ctas;       /* CTAs of the main kernel */
  uint64_t workspace_bytes;/* device scratch the call needs (0: none) */
  double flops;            /* 2*M*N*K */
  double bytes;            /* algorithmic HBM bytes: A, B once, C once (+C read if beta != 0) */
  double intensity;        /* flops / bytes */
  int32_t b_concat;        /* TF32X3: A_hi*[B_hi|B_lo] issued as one MMA of width 2*bn (1) or two MMAs (0) */
  int32_t ctas_per_sm;     /* CTAs of the main kernel resident per SM (shared memory and TMEM budget) */
  int32_t stream_k;        /* tensor-core modes: grid_ctas persistent CTAs take whole tiles in
                              waves, then share the remaining tiles' K blocks evenly; a fix-up
                              kernel sums the parts of tiles shared between CTAs */
  int32_t a_hi_tmem;       /* tensor-core modes with A split on chip: A_hi kept in tensor memory (1)
                              or read from the landed tile in shared memory (0) */
  int32_t b_split_in_kernel; /* tensor-core modes: B read as stored and split inside the GEMM
                              kernel (1: no pass before it for B) or by a pre-pass (0) */
} gemm_plan_t;

typedef struct gemm_device_info {
  int32_t device;
  int32_t sm_count;
  int32_t cc_major, cc_minor;
  int32_t clock_khz;            /* cudaDevAttrClockRate (max SM clock) */
  int32_t mem_clock_khz;
  int32_t mem_bus_width_bits;
  int32_t fp32_lanes_per_sm;    /* 128 on sm_10x */
  int32_t regs_per_sm;
  int32_t smem_per_sm;
  int32_t smem_per_block_optin;
  int32_t from_device;          /* 1: queried from a device, 0: built-in GB300 defaults */
  int64_t l2_bytes;
  int64_t hbm_bytes;
  double fp32_peak_tflops;      /* sm_count * lanes * 2 * clock */
  char name[128];
} gemm_device_info_t;

/*
 * gemm_f32 -- C <- A * B  (alpha = 1, beta = 0: C is only written).
 * Equivalent to gemm_f32_ex(M,N,K, 1.0f, A,lda, B,ldb, 0.0f, C,ldc, mode,
 * NULL, 0, stream).
 * M, N, K >= 0.  M == 0 or N == 0 is a no-op.  K == 0 writes zeros to C.
 * A, B may be NULL only when the product is empty (K == 0 or M == 0 or
 * N == 0); C may be NULL only when M == 0 or N == 0.
 * stream: a cudaStream_t of the current device (0 = legacy default stream).
 * Returns GEMM_OK, or GEMM_ERR_INVALID_ARG (bad size, ld, pointer, mode),
 * GEMM_ERR_UNSUPPORTED, GEMM_ERR_CUDA, GEMM_ERR_NO_DEVICE.
 */
GEMM_API int gemm_f32(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
             const float *B, int64_t ldb, float *C, int64_t ldc, int mode,
             cudaStream_t stream);

/*
 * gemm_f32_ex -- C <- alpha * A * B + beta * C (BLAS semantics).
 * When beta == 0, C is not read (NaN/Inf in C do not propagate); when
 * alpha == 0, A and B are not read and C <- beta * C (one scaling kernel;
 * gemm_f32_plan describes the alpha != 0 call).
 * workspace/ws_bytes: device scratch of at least plan.workspace_bytes
 * (gemm_f32_plan), 256-byte aligned, owned by the caller and not used by
 * any other work in flight on the GPU during this call.  workspace == NULL
 * lets the library use its own per-device buffer, grown with cudaMalloc
 * when needed (which synchronises the device) and freed by gemm_shutdown();
 * that buffer is shared by every call on the device, so calls that use it
 * must not run at the same time on the GPU (issue them on one stream, or
 * give each concurrent stream its own workspace).
 * A call allocates nothing, synchronises nothing and reads nothing back to
 * the host when the workspace is given (or the library buffer is already
 * large enough), so it can be captured into a CUDA graph and replayed.
 * A non-NULL workspace smaller than the plan needs returns
 * GEMM_ERR_WORKSPACE_TOO_SMALL.
 */
GEMM_API int gemm_f32_ex(int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                int64_t lda, const float *B, int64_t ldb, float beta, float *C,
                int64_t ldc, int mode, void *workspace, size_t ws_bytes,
                cudaStream_t stream);

/*
 * gemm_f32_plan -- what gemm_f32/gemm_f32_ex would run for this shape, with
 * no launch and no allocation.
 *
 * The course page picks each rung's launch by hand: 16 x 16 thread blocks
 * and a grid that covers N x N for the naive and coalesced kernels, TILE x
 * TILE blocks for the shared-memory kernel, with TILE = 16 and 32 measured
 * side by side ("Project - tiled matrix multiply", sections "Stage 0 - the
 * naive baseline", "Stage 1 - global memory coalescing" and "Stage 2").  The
 * plan is that choice made by the library for any M, N, K: kernel, CTA tile,
 * pipeline depth, K slices, stream-K grid and workspace.  It also places the
 * shape on the roofline: arithmetic intensity = 2*M*N*K / algorithmic bytes,
 * compared with the ridge point = arithmetic rate / memory bandwidth of the
 * resolved mode ("Bandwidths and peak rate - exercises", exercise 3), which
 * gives plan.bound.
 *
 * Arguments: M, N, K >= 0 and the leading dimensions as gemm_f32_ex would
 * get them (row-major; a too-small ld returns GEMM_ERR_INVALID_ARG).
 * align_hint: the bitwise OR of the A, B and C addresses the call will use
 * (0 = assume 16-byte aligned); it decides between the 128-bit and the
 * scalar path.  beta_nonzero only changes the algorithmic byte count.  out:
 * caller-owned, written only on GEMM_OK.  Uses the current device's
 * properties when a device is visible, else built-in GB300 figures (152
 * SMs).  Host only: launches nothing, allocates nothing.  Returns GEMM_OK,
 * GEMM_ERR_INVALID_ARG (sizes, ld, mode, out == NULL) or
 * GEMM_ERR_UNSUPPORTED (a tensor-core mode on a device without sm_103a, or a
 * shape beyond its limits).
 */
GEMM_API int gemm_f32_plan(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                  int64_t ldc, int mode, uintptr_t align_hint,
                  int beta_nonzero, gemm_plan_t *out);

/*
 * gemm_f32_op -- C <- alpha * op(A) * op(B) + beta * C with the storage
 * order and operand ops of a BLAS SGEMM call.
 *
 * The course page's cuBLAS stage ("Project - tiled matrix multiply",
 * "Stage 3 - the reference ceiling: cuBLAS") calls a column-major library
 * on row-major data by computing C^T = B^T * A^T with the operands swapped;
 * this call takes either storage order and either op directly, so callers
 * with column-major or transposed matrices need no such rewrite.
 *
 * layout: GEMM_ROW_MAJOR (X(r,c) = X[r*ld + c]) or GEMM_COL_MAJOR
 *         (X(r,c) = X[c*ld + r]); applies to A, B and C alike.
 * op_a, op_b: GEMM_OP_N (op(X) = X) or GEMM_OP_T (op(X) = X^T).
 * op(A) is M x K, op(B) is K x N, C is M x N.  A is stored as the M x K
 * matrix (op_a = N) or the K x M matrix (op_a = T) in `layout`, and so on:
 *   stored rows x cols of A = op_a == N ? M x K : K x M, likewise B
 *   (K x N or N x K); ld >= the stored number of columns (row-major) or
 *   rows (column-major), and >= 1.
 * Everything else (device pointers, workspace, stream, beta == 0 not
 * reading C, return codes) is as gemm_f32_ex; mode must be AUTO,
 * FP32_SIMT, TF32X3 or TF32 (the teaching kernels take plain row-major
 * operands only: GEMM_ERR_UNSUPPORTED otherwise).  A layout or op outside
 * the constants below returns GEMM_ERR_INVALID_ARG.
 * Results equal gemm_f32_ex's on the same logical matrices, bit for bit,
 * whenever both run the same kernel configuration.  In the tensor-core
 * modes a B that the row-major problem sees stored N x K (row-major with
 * op_b = T) and 16-byte aligned with ldb a multiple of 4 can be read as
 * stored and split inside the GEMM kernel, with no pass before it (the
 * plan's b_split_in_kernel); the bits are those of the pass.
 */
#define GEMM_ROW_MAJOR 0
#define GEMM_COL_MAJOR 1
#define GEMM_OP_N 0
#define GEMM_OP_T 1

GEMM_API int gemm_f32_op(int layout, int op_a, int op_b, int64_t M, int64_t N, int64_t K,
                         float alpha, const float *A, int64_t lda, const float *B,
                         int64_t ldb, float beta, float *C, int64_t ldc, int mode,
                         void *workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * gemm_f32_op_plan -- gemm_f32_plan for a gemm_f32_op call.  The returned
 * plan describes the row-major problem the call runs (for GEMM_COL_MAJOR:
 * C^T = op(B)^T * op(A)^T, so M and N are exchanged in its tile grid).
 */
GEMM_API int gemm_f32_op_plan(int layout, int op_a, int op_b, int64_t M, int64_t N, int64_t K,
                              int64_t lda, int64_t ldb, int64_t ldc, int mode,
                              uintptr_t align_hint, int beta_nonzero, gemm_plan_t *out);

/*
 * gemm_f32_host -- C <- alpha * A * B + beta * C with A, B and C in HOST
 * memory (row-major, leading dimensions as gemm_f32_ex).  Blocking: returns
 * once C holds the result (or an error), with no copy still touching the
 * caller's buffers.
 *
 * The course page's scaffolding copies the operands to the GPU, runs the
 * kernel and copies the result back ("Project - tiled matrix multiply",
 * "Starter scaffolding"); this call does the same for the caller, cutting
 * the product into row blocks of A (and C) and column blocks of B (and C).
 * A and B blocks are copied in alternately, each GEMM starts as soon as its
 * two blocks are on the device, and each block of C is copied back as soon
 * as its GEMM is done, so copies in, GEMMs and copies out overlap.
 * Page-locked host buffers (cudaHostAlloc / cudaMallocHost) are needed for
 * the copies to overlap; pageable buffers give the same result, slower.
 *
 * mode: as gemm_f32_ex; AUTO is resolved once, for the whole product, and
 * that mode runs every block.  blocks: number of row blocks, 1 ..
 * GEMM_HOST_MAX_BLOCKS, with B in one column block; or 0 for the library's
 * choice (one block for short products; else for K >= 2048 up to 3 x 3
 * blocks of at least 1024 rows and 1024 columns, for shallower products up
 * to 4 row blocks).  Row blocks hold whole 128-row tiles and column blocks
 * whole 256-column tiles, except the last ones.
 * With the environment variable GEMM_HOST_STREAM=1 (and blocks == 0), a
 * product that resolves to the tensor-core kernel with A split on chip
 * (K % 4 == 0) runs in a streaming form instead: B is copied in whole, A
 * (and C) in row blocks, and one GEMM launch over the whole product starts
 * once B is in, each of its CTAs waiting (bounded) for its rows' block to
 * land; each row block of C is copied back as soon as the GEMM has stored
 * it.  Same results within the bound; faster on some shapes, slower on
 * others, so it is not the default.
 * The library stages the whole problem in device memory it owns (M*K + K*N
 * + M*N floats plus a GEMM workspace per column block), grown on demand and
 * freed by gemm_shutdown(); calls on one device are serialised.
 * Returns GEMM_OK, GEMM_ERR_INVALID_ARG (size, ld, pointer, mode, blocks),
 * GEMM_ERR_UNSUPPORTED, GEMM_ERR_CUDA (including a failed staging
 * allocation), GEMM_ERR_DEVICE_TIMEOUT (a bounded wait in the tensor-core
 * kernel ran out), GEMM_ERR_NO_DEVICE.
 */
#define GEMM_HOST_MAX_BLOCKS 64

GEMM_API int gemm_f32_host(int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                           int64_t lda, const float *B, int64_t ldb, float beta, float *C,
                           int64_t ldc, int mode, int blocks);

/*
 * hbm_copy_f32 -- dst[i] = src[i] for i < n on `stream` (the
 * device-to-device copy kernel of "Bandwidths and peak rate - exercises",
 * exercise 2: one read and one write per element).  Device pointers, must
 * not overlap.  Enqueue only.
 */
GEMM_API int hbm_copy_f32(const float *src, float *dst, size_t n, cudaStream_t stream);

/*
 * hbm_copy_calibrate -- measures achieved HBM bandwidth with hbm_copy_f32:
 * one untimed warm-up copy, then `iters` (>= 1) copies timed with CUDA
 * events on `stream`; *gbps_out = 2 * n * sizeof(float) * iters / seconds
 * / 1e9 (same exercise).  Blocks until the timed copies finish.  The
 * caller owns src and dst (n floats each; the exercise uses n = 256M, 1 GiB
 * per buffer).
 */
GEMM_API int hbm_copy_calibrate(const float *src, float *dst, size_t n, int iters,
                       cudaStream_t stream, double *gbps_out);

/*
 * fp32_fma_peak -- measures the FP32 FMA throughput of the CUDA cores with a
 * register-only kernel ("Bandwidths and peak rate - exercises", exercise 5:
 * long chains acc = acc * x + y, several independent chains per thread,
 * FLOP = threads x iterations x chains x 2).  packed = 1 uses the f32x2 FMA
 * (two lanes per instruction), 0 the scalar FMA.  One untimed warm-up
 * launch, then one launch of `iters` iterations timed with CUDA events on
 * `stream`; blocks until it finishes.  sink: device buffer of at least
 * fp32_fma_peak_sink_floats() floats (receives each thread's result).
 * *tflops_out = FLOP / seconds / 1e12.
 */
GEMM_API int fp32_fma_peak(int64_t iters, int packed, float *sink, cudaStream_t stream,
                           double *tflops_out);

/* Floats fp32_fma_peak writes to its sink on the current device. */
GEMM_API int64_t fp32_fma_peak_sink_floats(void);

/*
 * gemm_device_info -- SM count, clocks, register/shared-memory/L2/HBM sizes
 * of device `dev` (the device-property program of "Memory hierarchy in
 * hardware - solutions", exercise 1) and the FP32 CUDA-core peak derived as
 * in "Bandwidths and peak rate - exercises", exercise 1: SMs x 128 FP32
 * lanes x 2 x clock.  dev < 0 or no visible device fills built-in GB300
 * figures with from_device = 0 and returns GEMM_OK.
 */
GEMM_API int gemm_device_info(int dev, gemm_device_info_t *out);

/*
 * gemm_strerror -- a static, NUL-terminated description of a status code
 * (never NULL; unknown codes get "unknown status code"); the caller must not
 * free it.  The course page's scaffolding wraps every CUDA call in a
 * CUDA_CHECK macro that prints the error string and exits the process
 * ("Project - tiled matrix multiply", section "Starter scaffolding"); a
 * library must leave that decision to its caller, so every call returns a
 * code and this gives the text that macro would have printed.
 */
GEMM_API const char *gemm_strerror(int code);

/*
 * gemm_check_status -- the deferred half of that same CUDA_CHECK step
 * ("Starter scaffolding" checks cudaGetLastError and cudaDeviceSynchronize
 * after a launch): synchronises `stream`, then reads and clears the
 * library's device status words, set by the tensor-core kernel when one of
 * its bounded waits runs out and by the stream-K fix-up when a tile has more
 * parts than it can sum.  Returns GEMM_ERR_DEVICE_TIMEOUT or
 * GEMM_ERR_UNSUPPORTED if one was set (the result of the call that set it is
 * not valid), GEMM_ERR_CUDA if the synchronisation reported an error, else
 * GEMM_OK.  Blocking; not for use during stream capture.
 */
GEMM_API int gemm_check_status(cudaStream_t stream);

/*
 * gemm_set_profile_events -- measurement aid.  For the calling host thread,
 * the next GEMM calls record `before_main` on their stream immediately
 * before launching their main kernel (the SIMT or tensor-core GEMM kernel)
 * and `after_main` immediately after it, so that cudaEventElapsedTime gives
 * that kernel's device time.  Pass NULL, NULL to stop.  The caller owns the
 * events (created with cudaEventCreate on the current device).
 */
GEMM_API int gemm_set_profile_events(cudaEvent_t before_main, cudaEvent_t after_main);

/*
 * gemm_set_profile_stamps -- measurement aid that keeps the launch order of
 * a call unchanged (gemm_set_profile_events puts the main kernel in plain
 * stream order, which the events need; the split pass, GEMM kernel and
 * fix-up otherwise overlap their launches).  For the calling host thread,
 * the next GEMM calls' main kernel (the CUDA-core or tensor-core GEMM
 * kernel) reads the GPU's nanosecond clock (%globaltimer) and folds it into
 * stamps[0] with an atomic minimum when each of its CTAs starts work (past
 * its wait for the kernel before it), and into stamps[1] with an atomic
 * maximum when each CTA has finished, so stamps[1] - stamps[0] is that
 * launch's duration in ns.  stamps: DEVICE memory on the current device, 8-byte
 * aligned, owned by the caller, who sets stamps[0] = ~0 and stamps[1] = 0
 * before the call and passes a fresh pair for each launch it wants timed
 * separately.  NULL stops.  The course page times with cudaEvent pairs
 * ("Project - tiled matrix multiply", "Starter scaffolding"); these stamps
 * time one kernel inside a chain of launches that events would serialise.
 * Returns GEMM_ERR_INVALID_ARG for a misaligned pointer, else GEMM_OK.
 */
GEMM_API int gemm_set_profile_stamps(unsigned long long *stamps);

/*
 * gemm_f32_splitk_noalloc -- C <- alpha * A * B + beta * C on the CUDA cores
 * (the FP32_SIMT kernel), allocating no device memory at all.  The course
 * pages have no counterpart to this call; it exists for callers that cannot
 * allocate: code held to a device-memory budget fixed at start-up (for
 * example under a framework allocator that has already reserved the free
 * memory) and latency-critical loops that cannot take the device-wide
 * synchronisation of cudaMalloc/cudaFree.  The split-K partial sums go to a
 * static array of GEMM_NOALLOC_SCRATCH_BYTES that the library keeps in
 * device memory on every GPU that loads it, until the process exits.
 *
 * Arguments and layout are those of gemm_f32_ex (device pointers, row-major,
 * lda >= K, ldb >= N, ldc >= N).  split_k = 0 takes the planner's slice
 * count for FP32_SIMT, reduced if need be to the most slices whose partial
 * sums fit the array (at worst one slice, which needs no scratch), so it
 * never fails for want of scratch.  1 <= split_k <= GEMM_NOALLOC_MAX_SPLIT
 * asks for that many K slices (rounded to whole K tiles of the kernel, 16
 * deep by default, which can only lower the count); when their partial
 * sums, split_k * M * N * 4 bytes, exceed GEMM_NOALLOC_SCRATCH_BYTES the
 * call returns
 * GEMM_ERR_WORKSPACE_TOO_SMALL and launches nothing.  split_k < 0 or above
 * GEMM_NOALLOC_MAX_SPLIT returns GEMM_ERR_INVALID_ARG.  Other errors as
 * gemm_f32_ex.
 *
 * The first call on a device looks up the array's device address (with that
 * device current); make that first call before any stream capture.  All
 * calls share the one array, and a call leaves its partial sums there:
 * calls whose kernels overlap on the GPU (different streams, or different
 * host threads) race on it and must be serialised by the caller.  Nothing
 * in the array needs clearing between calls: each call writes every partial
 * sum before reading it.
 */
#define GEMM_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
#define GEMM_NOALLOC_MAX_SPLIT 256
GEMM_API int gemm_f32_splitk_noalloc(int64_t M, int64_t N, int64_t K, float alpha,
                                     const float *A, int64_t lda, const float *B,
                                     int64_t ldb, float beta, float *C, int64_t ldc,
                                     int split_k, cudaStream_t stream);

/* Frees the library's per-device workspace buffers.  Call with no library
 * work in flight. */
GEMM_API void gemm_shutdown(void);

/* ABI version this library was built with (GEMM_ABI_VERSION). */
GEMM_API int gemm_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* GB300_GEMM_H */
