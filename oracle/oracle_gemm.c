/*
 * CPU oracle for the dense matrix multiply C = A * B.  TEST INFRASTRUCTURE
 * ONLY: the tests, the smoke check and the benchmark's CPU-baseline leg call
 * it; the CUDA library never links, loads or calls it, and it shares no code,
 * header or constant with that library.
 *
 * What it computes is the plain definition the pages start from (and that
 * tiling leaves unchanged: tiling moves data closer to the arithmetic, it does
 * not change the arithmetic):
 *
 *     C[i][j] = sum over k = 0 .. K-1 of A[i][k] * B[k][j]
 *
 *   - "矩阵乘法 tiling:把分块搬进 shared memory,让 GFLOPS 翻百倍", section 一
 *     (the naive kernel: one output per thread, a dot product of a row of A
 *     and a column of B, row-major N x N floats);
 *   - "CUDA 深入浅出（二）：为什么分块可以减少 Global Memory 访问", section
 *     "naive kernel 怎么读数据" (the same dot product, and that tiling saves
 *     loads, never arithmetic);
 *   - the ijyty.com page on shared-memory tiling, opening paragraph
 *     (C[row][col] as the K-direction sum of A[row][k] * B[k][col]);
 *   - "CUDA 编程系列之三：内存墙与分块（tiling）的诞生", section 6
 *     (P[row][col] = sum_k M[row][k] * N[k][col]).
 *
 * Precision: every product is formed in double from the fp32 operands (the
 * product of two fp32 values is exact in double), summed in ascending k in
 * double, and rounded once to fp32 (round to nearest even).  The pages
 * accumulate in fp32; the fp64 sum is the stricter reading, against which
 * every GPU path is checked with one tolerance.
 *
 * Layout: row-major with leading dimensions, A[i*lda + k], B[k*ldb + j],
 * C[i*ldc + j].  Rectangular shapes and leading dimensions generalise the
 * pages' square N x N indexing; nothing outside the logical M x N block of C
 * is written.  K == 0 gives C == 0 (the empty sum).
 *
 * Threads: output rows are independent, so rows are shared among OpenMP
 * threads; each entry's summation order is unchanged by this.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1

static int bad_dims(const void* A, const void* B, int64_t M, int64_t N, int64_t K,
                    int64_t lda, int64_t ldb) {
  if (M < 0 || N < 0 || K < 0) return 1;
  if (K > 0 && (lda < K || ldb < N)) return 1;
  if (K > 0 && M > 0 && N > 0 && (A == NULL || B == NULL)) return 1;
  return 0;
}

/* One entry of the definition: sum_k A[i][k] * B[k][j] in double, k ascending.
 * Also returns sum_k |A[i][k]| * |B[k][j]|, the scale that the normalised
 * error max|C - C_ref| / sum_k |A_ik||B_kj| divides by. */
static double dot_entry(const float* A, const float* B, int64_t K, int64_t lda,
                        int64_t ldb, int64_t i, int64_t j, double* abs_sum) {
  double s = 0.0, a = 0.0;
  const float* arow = A + i * lda;
  for (int64_t k = 0; k < K; ++k) {
    double x = (double)arow[k];
    double y = (double)B[k * ldb + j];
    s += x * y;
    a += fabs(x) * fabs(y);
  }
  if (abs_sum) *abs_sum = a;
  return s;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Full product.  absC (optional, may be NULL) receives sum_k |A_ik||B_kj| in
 * double with leading dimension ldc.  nthreads <= 0 means the OpenMP default. */
int oracle_gemm(const float* A, const float* B, float* C, int64_t M, int64_t N,
                int64_t K, int64_t lda, int64_t ldb, int64_t ldc, double* absC,
                int nthreads) {
  if (bad_dims(A, B, M, N, K, lda, ldb) || (M > 0 && N > 0 && (C == NULL || ldc < N)))
    return ORACLE_BAD_ARG;
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
  for (int64_t i = 0; i < M; ++i) {
    for (int64_t j = 0; j < N; ++j) {
      double a = 0.0;
      double s = dot_entry(A, B, K, lda, ldb, i, j, &a);
      C[i * ldc + j] = (float)s;
      if (absC) absC[i * ldc + j] = a;
    }
  }
  (void)nthreads;
  return ORACLE_OK;
}

/* Selected entries (rows[t], cols[t]) of the product, for checks at sizes
 * where the full product is too slow on a CPU.  out[t] is the fp32 result,
 * abs_out[t] (optional) the sum of |A_ik||B_kj|. */
int oracle_gemm_entries(const float* A, const float* B, int64_t M, int64_t N,
                        int64_t K, int64_t lda, int64_t ldb, const int64_t* rows,
                        const int64_t* cols, int64_t n, float* out,
                        double* abs_out, int nthreads) {
  if (bad_dims(A, B, M, N, K, lda, ldb) || n < 0 || (n > 0 && (!rows || !cols || !out)))
    return ORACLE_BAD_ARG;
  for (int64_t t = 0; t < n; ++t)
    if (rows[t] < 0 || rows[t] >= M || cols[t] < 0 || cols[t] >= N) return ORACLE_BAD_ARG;
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 64) num_threads(nthreads)
#endif
  for (int64_t t = 0; t < n; ++t) {
    double a = 0.0;
    double s = dot_entry(A, B, K, lda, ldb, rows[t], cols[t], &a);
    out[t] = (float)s;
    if (abs_out) abs_out[t] = a;
  }
  (void)nthreads;
  return ORACLE_OK;
}
