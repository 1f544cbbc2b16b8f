/*
 * Cache-blocked CPU GEMM: C = A * B, row-major fp32, fp32 accumulation.
 *
 * The same method as the GPU kernels, one memory hierarchy over: the pages
 * note that tiling is not a GPU trick -- on a CPU the blocks are sized for
 * the caches instead of shared memory ("CUDA 编程系列之三：内存墙与分块
 * （tiling）的诞生", section 8; "矩阵乘法 tiling", section "这一篇在知识体系里
 * 的位置").  It serves as a realistic host comparator beside the deliberately
 * plain oracle; it shares no code with the oracle or the CUDA library.
 *
 * Blocking: C is cut into MC x NC blocks shared among OpenMP threads; for each
 * KC-deep slice of K, the thread copies the B slice block (KC x NC) into a
 * contiguous buffer that stays in L2, then sweeps the rows of A in the block,
 * each row's NC accumulators staying in L1 while KC multiply-adds per element
 * run (i-k-j order, the innermost j loop is unit-stride and vectorisable).
 * Each A element is reused NC times and each B element MC times from cache.
 * Edges are handled by clipping the block extents.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { MC = 64, NC = 256, KC = 256 };

int cpu_tiled_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

int cpu_tiled_gemm(const float* A, const float* B, float* C, int64_t M, int64_t N, int64_t K,
                   int64_t lda, int64_t ldb, int64_t ldc, int nthreads) {
  if (M < 0 || N < 0 || K < 0) return 1;
  if (M == 0 || N == 0) return 0;
  if (!C || ldc < N || (K > 0 && (!A || !B || lda < K || ldb < N))) return 1;
  const int64_t mb = (M + MC - 1) / MC, nb = (N + NC - 1) / NC;
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
#endif
  {
    float* bpack = (float*)malloc(sizeof(float) * KC * NC);
    float acc[NC];
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
    for (int64_t blk = 0; blk < mb * nb; ++blk) {
      const int64_t i0 = (blk / nb) * MC, j0 = (blk % nb) * NC;
      const int64_t ie = i0 + MC < M ? i0 + MC : M;
      const int64_t nw = j0 + NC < N ? NC : N - j0;
      for (int64_t i = i0; i < ie; ++i) memset(C + i * ldc + j0, 0, sizeof(float) * nw);
      for (int64_t k0 = 0; k0 < K; k0 += KC) {
        const int64_t kw = k0 + KC < K ? KC : K - k0;
        for (int64_t k = 0; k < kw; ++k)
          memcpy(bpack + k * NC, B + (k0 + k) * ldb + j0, sizeof(float) * nw);
        for (int64_t i = i0; i < ie; ++i) {
          float* crow = C + i * ldc + j0;
          for (int64_t j = 0; j < nw; ++j) acc[j] = crow[j];
          const float* arow = A + i * lda + k0;
          for (int64_t k = 0; k < kw; ++k) {
            const float a = arow[k];
            const float* brow = bpack + k * NC;
            for (int64_t j = 0; j < nw; ++j) acc[j] += a * brow[j];
          }
          for (int64_t j = 0; j < nw; ++j) crow[j] = acc[j];
        }
      }
    }
    free(bpack);
  }
  return 0;
}
