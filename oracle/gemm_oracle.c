/*
 * CPU oracle for the FP32 GEMM library -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the bench's CPU-baseline leg may load
 * this file's library.  It shares no code, header, table or helper with the
 * CUDA path and must never be called by the product path.
 *
 * What it computes (one definition, written out):
 *
 *   C_ref(i,j) = float_rn( alpha * S(i,j) + beta * C_old(i,j) ),
 *   S(i,j)     = sum over k = 0 .. K-1, in ascending k, of
 *                (double)A(i,k) * (double)B(k,j), accumulated in double,
 *
 * with row-major storage A(i,k) = A[i*lda + k], B(k,j) = B[k*ldb + j],
 * C(i,j) = C[i*ldc + j].  This is the CPU reference of the tiled-matmul
 * course page ("Project - tiled matrix multiply", section "Starter
 * scaffolding": a triple loop that accumulates in double and rounds once to
 * float), generalised from N x N to M x N x K, leading dimensions, and the
 * alpha/beta scaling of the cuBLAS SGEMM call in section "Stage 3 - the
 * reference ceiling: cuBLAS".  When beta == 0, C_old is not read (BLAS
 * convention), so NaN in C_old does not propagate; likewise when alpha == 0
 * A and B are not read (S is taken as 0), so C_ref = float_rn(beta * C_old).
 *
 * Each product of two floats is exact in double (24 + 24 < 53 significand
 * bits); the only roundings are the double additions, the alpha/beta
 * products and the final cast.  Compile with -ffp-contract=off so the
 * compiler does not fuse the multiply and add.
 *
 * The per-entry bound  D(i,j) = |alpha| * sum_k |A(i,k)| |B(k,j)|
 * + |beta| |C_old(i,j)|  is the denominator of the normalised error metric.
 *
 * Parallelism: rows are independent outputs, so the full-matrix routine
 * splits rows across OpenMP threads; each entry is still summed in the
 * order above.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static float oracle_entry(int64_t i, int64_t j, int64_t K, double alpha,
                          const float *A, int64_t lda, const float *B,
                          int64_t ldb, double beta, const float *Cin,
                          int64_t ldc, double *bound) {
  double s = 0.0, sa = 0.0;
  const float *a = A + i * lda;
  if (alpha == 0.0) K = 0; /* A and B are not read */
  for (int64_t k = 0; k < K; ++k) {
    double p = (double)a[k] * (double)B[k * ldb + j];
    s += p;
    sa += fabs(p);
  }
  double r = alpha * s;
  double d = fabs(alpha) * sa;
  if (beta != 0.0) {
    double c = (double)Cin[i * ldc + j];
    r += beta * c;
    d += fabs(beta) * fabs(c);
  }
  if (bound) *bound = d;
  return (float)r;
}

/* Full C_ref (M x N into Cout with leading dimension ldo); optional bound
 * matrix D (M x N, leading dimension ldo) when D != NULL.  nthreads <= 0
 * uses the OpenMP default. */
int oracle_gemm(int64_t M, int64_t N, int64_t K, double alpha, const float *A,
                int64_t lda, const float *B, int64_t ldb, double beta,
                const float *Cin, int64_t ldc, float *Cout, double *D,
                int64_t ldo, int nthreads) {
  if (M < 0 || N < 0 || K < 0) return -1;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < M; ++i) {
    for (int64_t j = 0; j < N; ++j) {
      double bd;
      Cout[i * ldo + j] = oracle_entry(i, j, K, alpha, A, lda, B, ldb, beta,
                                       Cin, ldc, &bd);
      if (D) D[i * ldo + j] = bd;
    }
  }
  return 0;
}

/* C_ref and D at n listed positions (rows[t], cols[t]). */
int oracle_gemm_entries(int64_t M, int64_t N, int64_t K, double alpha,
                        const float *A, int64_t lda, const float *B,
                        int64_t ldb, double beta, const float *Cin,
                        int64_t ldc, int64_t n, const int64_t *rows,
                        const int64_t *cols, float *out, double *D,
                        int nthreads) {
  for (int64_t t = 0; t < n; ++t)
    if (rows[t] < 0 || rows[t] >= M || cols[t] < 0 || cols[t] >= N) return -1;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < n; ++t) {
    double bd;
    out[t] = oracle_entry(rows[t], cols[t], K, alpha, A, lda, B, ldb, beta,
                          Cin, ldc, &bd);
    if (D) D[t] = bd;
  }
  return 0;
}

/* Threads the OpenMP runtime would use (for reporting). */
int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
