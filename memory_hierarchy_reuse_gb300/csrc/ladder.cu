// The pages' optimisation ladder, rebuilt for measurement on GB300: the
// one-output-per-thread kernel and the shared-memory tiled kernel at T = 16
// and T = 32.  They exist to test the pages' own claims on this hardware:
//   * naive: every output reads a row of A and a column of B straight from
//     global memory, 2MNK element loads in all ("矩阵乘法 tiling", section 一;
//     "CUDA 深入浅出（二）", section "naive kernel 怎么读数据");
//   * tiled T: a T x T block stages a T x T tile of A and of B per K step,
//     reuses each staged element T times, and loads 2MNK/T elements
//     ("矩阵乘法 tiling", sections 二-四; "CUDA 深入浅出（二）", section
//     "推广到整个 N×N 矩阵"; "CUDA 编程系列之三", section 6);
//   * the two barriers per K step -- one after the load, one before the next
//     load overwrites the tile ("矩阵乘法 tiling", section 四);
//   * threadIdx.x runs along a row of C, so a warp's global loads of B and
//     stores of C are consecutive (the ijyty.com page, step ②).
// Unlike the pages' listings, edges are handled: out-of-range inputs load as
// zero and out-of-range outputs are not stored ("矩阵乘法 tiling", section 六;
// "CUDA 编程系列之三", section 7).  The B tile is padded by one column so the
// column-wise reads of the compute loop do not share a bank.
#include <cuda_runtime.h>
#include <cstdint>

#include "mhr_internal.h"

namespace mhr {
namespace {

__global__ void ladder_naive_kernel(const float* __restrict__ A, const float* __restrict__ B,
                                    float* __restrict__ C, int64_t M, int64_t N, int64_t K,
                                    int64_t lda, int64_t ldb, int64_t ldc) {
  const int64_t row = static_cast<int64_t>(blockIdx.y) * blockDim.y + threadIdx.y;
  const int64_t col = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (row >= M || col >= N) return;
  float acc = 0.f;
  for (int64_t k = 0; k < K; ++k) acc = fmaf(A[row * lda + k], B[k * ldb + col], acc);
  C[row * ldc + col] = acc;
}

template <int T>
__global__ void __launch_bounds__(T * T)
    ladder_tiled_kernel(const float* __restrict__ A, const float* __restrict__ B,
                        float* __restrict__ C, int64_t M, int64_t N, int64_t K, int64_t lda,
                        int64_t ldb, int64_t ldc) {
  __shared__ float As[T][T];
  __shared__ float Bs[T][T + 1];
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int64_t row = static_cast<int64_t>(blockIdx.y) * T + ty;
  const int64_t col = static_cast<int64_t>(blockIdx.x) * T + tx;
  float acc = 0.f;
  for (int64_t k0 = 0; k0 < K; k0 += T) {
    // one element of each tile per thread; zero outside the matrices
    As[ty][tx] = (row < M && k0 + tx < K) ? A[row * lda + k0 + tx] : 0.f;
    Bs[ty][tx] = (k0 + ty < K && col < N) ? B[(k0 + ty) * ldb + col] : 0.f;
    __syncthreads();  // the tile is complete before anyone reads it
#pragma unroll
    for (int k = 0; k < T; ++k) acc = fmaf(As[ty][k], Bs[k][tx], acc);
    __syncthreads();  // everyone is done reading before the next load
  }
  if (row < M && col < N) C[row * ldc + col] = acc;
}

}  // namespace

cudaError_t launch_ladder(int rung, const float* A, const float* B, float* C, int64_t M, int64_t N,
                          int64_t K, int64_t lda, int64_t ldb, int64_t ldc, cudaStream_t s) {
  const int T = rung == 2 ? 32 : 16;
  const dim3 grid(static_cast<unsigned>((N + T - 1) / T), static_cast<unsigned>((M + T - 1) / T));
  const dim3 block(T, T);
  switch (rung) {
    case 0:
      note_main_kernel("ladder_naive_kernel", static_cast<int>(grid.x * grid.y), 0);
      ladder_naive_kernel<<<grid, block, 0, s>>>(A, B, C, M, N, K, lda, ldb, ldc);
      break;
    case 1:
      note_main_kernel("ladder_tiled_kernel<16>", static_cast<int>(grid.x * grid.y), 0);
      ladder_tiled_kernel<16><<<grid, block, 0, s>>>(A, B, C, M, N, K, lda, ldb, ldc);
      break;
    default:
      note_main_kernel("ladder_tiled_kernel<32>", static_cast<int>(grid.x * grid.y), 0);
      ladder_tiled_kernel<32><<<grid, block, 0, s>>>(A, B, C, M, N, K, lda, ldb, ldc);
      break;
  }
  return cudaGetLastError();
}

}  // namespace mhr
