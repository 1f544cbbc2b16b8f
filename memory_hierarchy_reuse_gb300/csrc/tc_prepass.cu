// Pre-passes of the tensor-core paths: the 3xTF32 split (each fp32 operand
// into tf32 big and small parts, B transposed to K-major), the bf16 repack for
// operands that TMA cannot address, and the K == 0 zero fill.
#include <cuda_runtime.h>
#include <cstdint>

#include "mhr_device.cuh"
#include "mhr_internal.h"
#include "tf32_split.cuh"

namespace mhr {
namespace {

__global__ void zero_fill_kernel(float* C, int64_t M, int64_t N, int64_t ldc) {
  for (int64_t r = blockIdx.y; r < M; r += gridDim.y)
    for (int64_t c = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; c < N;
         c += static_cast<int64_t>(gridDim.x) * blockDim.x)
      C[r * ldc + c] = 0.f;
}

__global__ void pack_u16_kernel(const uint16_t* __restrict__ src, int64_t rows, int64_t cols,
                                int64_t src_ld, uint16_t* __restrict__ dst, int64_t dst_ld) {
  grid_launch_dependents();  // the GEMM kernel after this one may start its set-up
  for (int64_t r = blockIdx.y; r < rows; r += gridDim.y)
    for (int64_t c = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; c < cols;
         c += static_cast<int64_t>(gridDim.x) * blockDim.x)
      dst[r * dst_ld + c] = src[r * src_ld + c];
}

// Split of both operands in one launch.  Blocks [0, a_blocks) split rows of
// A in place order (big part truncated, see split_tf32_trunc; with a_big null
// only the small part is written, A itself serving as A_big); the remaining
// blocks split 64 x 64 tiles of B (big part truncated too, as the fused split
// reads B itself as its big part) and write them transposed.  VA selects 16-byte loads of A when its address, leading
// dimension and K allow them, else 4-byte loads; VB is the width in floats of
// B's loads, 4, 2 or 1, the widest that B's address, leading dimension and N
// allow.  The outputs (pitch Kp, a multiple of 4, in the 16-byte-aligned
// workspace) are always written with 16-byte stores.  Each thread keeps
// several loads in flight.
constexpr int SPLIT_THREADS = 256;
constexpr int SPLIT_TILE = 64;

// With 16- or 8-byte loads of B the kernel keeps to 64 registers, so four
// blocks fit on an SM (the 8-byte form took 70, three blocks): fewer, fuller
// passes for problems too small to fill HBM's queues, where every pass is a
// round trip.  GB300, whole 3xTF32 calls in interleaved runs: 3000 x 2050 x
// 1000 70.4 -> 68.4 us, 4096^3 441.1 us either way.
template <bool VA, int VB>
__global__ void __launch_bounds__(SPLIT_THREADS, VB == 1 ? 1 : 4)
    split_vec_kernel(const float* __restrict__ A, const float* __restrict__ B, int64_t M,
                     int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t Kp, int a_blocks,
                     float* __restrict__ a_big, float* __restrict__ a_small,
                     float* __restrict__ bt_big, float* __restrict__ bt_small) {
  grid_launch_dependents();  // the GEMM kernel after this one may start its set-up
  __shared__ float tb[SPLIT_TILE][SPLIT_TILE + 1];
  __shared__ float ts[SPLIT_TILE][SPLIT_TILE + 1];
  const int t = threadIdx.x;
  if (static_cast<int>(blockIdx.x) < a_blocks) {
    const int64_t k4 = Kp / 4;  // 16-byte chunks of an output row (pad columns get zeros)
    if (k4 < 4 * SPLIT_THREADS) {
      // Short rows: a pass covers `rows` whole rows, slot t + 256 j taking
      // chunk co[j] of row ro[j], so every thread has four loads in flight.
      const int rows = static_cast<int>((4 * SPLIT_THREADS) / k4);
      int ro[4], co[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int slot = t + j * SPLIT_THREADS;
        ro[j] = slot < rows * k4 ? slot / static_cast<int>(k4) : -1;
        co[j] = slot - ro[j] * static_cast<int>(k4);
      }
      for (int64_t r0 = static_cast<int64_t>(blockIdx.x) * rows; r0 < M;
           r0 += static_cast<int64_t>(a_blocks) * rows) {
        float4 v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int64_t r = r0 + ro[j];
          v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (ro[j] < 0 || r >= M) continue;
          const float* src = A + r * lda;
          if (VA) {
            v[j] = __ldg(reinterpret_cast<const float4*>(src) + co[j]);
          } else {
            const int64_t k = 4 * co[j];
            v[j].x = k < K ? __ldg(src + k) : 0.f;
            v[j].y = k + 1 < K ? __ldg(src + k + 1) : 0.f;
            v[j].z = k + 2 < K ? __ldg(src + k + 2) : 0.f;
            v[j].w = k + 3 < K ? __ldg(src + k + 3) : 0.f;
          }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int64_t r = r0 + ro[j];
          if (ro[j] < 0 || r >= M) continue;
          float4 b, s;
          split4_trunc<VA>(v[j], b, s);
          if (a_big) reinterpret_cast<float4*>(a_big + r * Kp)[co[j]] = b;
          reinterpret_cast<float4*>(a_small + r * Kp)[co[j]] = s;
        }
      }
      return;
    }
    for (int64_t r = blockIdx.x; r < M; r += a_blocks) {
      const float* src = A + r * lda;
      float4* db = a_big ? reinterpret_cast<float4*>(a_big + r * Kp) : nullptr;
      float4* ds = reinterpret_cast<float4*>(a_small + r * Kp);
      for (int64_t c0 = t; c0 < k4; c0 += 4 * SPLIT_THREADS) {
        float4 v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int64_t c = c0 + j * SPLIT_THREADS;
          if (c >= k4) continue;
          if (VA) {
            v[j] = __ldg(reinterpret_cast<const float4*>(src) + c);
          } else {
            const int64_t k = 4 * c;
            v[j].x = k < K ? __ldg(src + k) : 0.f;
            v[j].y = k + 1 < K ? __ldg(src + k + 1) : 0.f;
            v[j].z = k + 2 < K ? __ldg(src + k + 2) : 0.f;
            v[j].w = k + 3 < K ? __ldg(src + k + 3) : 0.f;
          }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int64_t c = c0 + j * SPLIT_THREADS;
          if (c < k4) {
            float4 b, s;
            split4_trunc<VA>(v[j], b, s);  // conversion where 16-byte loads keep this memory-bound
            if (db) db[c] = b;
            ds[c] = s;
          }
        }
      }
    }
    return;
  }
  // B role: tile (k0, n0) of 64 x 64, transposed.
  const int64_t tiles_n = (N + SPLIT_TILE - 1) / SPLIT_TILE;
  const int64_t tiles = tiles_n * ((K + SPLIT_TILE - 1) / SPLIT_TILE);
  const int64_t nb = gridDim.x - a_blocks;
  for (int64_t tile = blockIdx.x - a_blocks; tile < tiles; tile += nb) {
    const int64_t n0 = (tile % tiles_n) * SPLIT_TILE, k0 = (tile / tiles_n) * SPLIT_TILE;
    if constexpr (VB == 4) {
      float4 v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {  // read: 64 k-rows x 16 float4 along n
        const int idx = t + j * SPLIT_THREADS;
        const int64_t k = k0 + (idx >> 4), n = n0 + (idx & 15) * 4;
        v[j] = (k < K && n < N) ? __ldg(reinterpret_cast<const float4*>(B + k * ldb + n))
                                : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int idx = t + j * SPLIT_THREADS;
        const int kr = idx >> 4, nc = (idx & 15) * 4;
        float4 b, s;
        split4_trunc<true>(v[j], b, s);
        tb[kr][nc] = b.x; tb[kr][nc + 1] = b.y; tb[kr][nc + 2] = b.z; tb[kr][nc + 3] = b.w;
        ts[kr][nc] = s.x; ts[kr][nc + 1] = s.y; ts[kr][nc + 2] = s.z; ts[kr][nc + 3] = s.w;
      }
    } else if constexpr (VB == 2) {
      float2 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {  // read: 64 k-rows x 32 float2 along n
        const int idx = t + j * SPLIT_THREADS;
        const int64_t k = k0 + (idx >> 5), n = n0 + (idx & 31) * 2;
        v[j] = (k < K && n < N) ? __ldg(reinterpret_cast<const float2*>(B + k * ldb + n))
                                : make_float2(0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int idx = t + j * SPLIT_THREADS;
        const int kr = idx >> 5, nc = (idx & 31) * 2;
        float b0, s0, b1, s1;
        split_tf32_trunc<false>(v[j].x, b0, s0);
        split_tf32_trunc<false>(v[j].y, b1, s1);
        tb[kr][nc] = b0; tb[kr][nc + 1] = b1;
        ts[kr][nc] = s0; ts[kr][nc + 1] = s1;
      }
    } else {
      float v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {  // read: 64 k-rows x 64 n, one float per load
        const int idx = t + j * SPLIT_THREADS;
        const int64_t k = k0 + (idx >> 6), n = n0 + (idx & 63);
        v[j] = (k < K && n < N) ? __ldg(B + k * ldb + n) : 0.f;
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int idx = t + j * SPLIT_THREADS;
        float b, sm;
        split_tf32_trunc<false>(v[j], b, sm);  // integer rounding: this 4-byte-load branch is latency-bound
        tb[idx >> 6][idx & 63] = b;
        ts[idx >> 6][idx & 63] = sm;
      }
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 4; ++j) {  // write: 64 n-rows x 16 float4 along k (zeros past K)
      const int idx = t + j * SPLIT_THREADS;
      const int nr = idx >> 4, kc = (idx & 15) * 4;
      const int64_t n = n0 + nr, k = k0 + kc;
      if (n < N && k < Kp) {
        *reinterpret_cast<float4*>(bt_big + n * Kp + k) =
            make_float4(tb[kc][nr], tb[kc + 1][nr], tb[kc + 2][nr], tb[kc + 3][nr]);
        *reinterpret_cast<float4*>(bt_small + n * Kp + k) =
            make_float4(ts[kc][nr], ts[kc + 1][nr], ts[kc + 2][nr], ts[kc + 3][nr]);
      }
    }
    __syncthreads();
  }
}

unsigned grid_rows(int64_t rows) { return static_cast<unsigned>(rows < 65535 ? rows : 65535); }


}  // namespace

cudaError_t launch_zero_fill(float* C, int64_t M, int64_t N, int64_t ldc, cudaStream_t s) {
  const unsigned gx = static_cast<unsigned>((N + 255) / 256 < 64 ? (N + 255) / 256 : 64);
  note_launch();
  zero_fill_kernel<<<dim3(gx, grid_rows(M)), 256, 0, s>>>(C, M, N, ldc);
  return cudaGetLastError();
}

cudaError_t launch_pack_u16(const uint16_t* src, int64_t rows, int64_t cols, int64_t src_ld,
                            uint16_t* dst, int64_t dst_ld, cudaStream_t s) {
  const unsigned gx = static_cast<unsigned>((cols + 255) / 256 < 64 ? (cols + 255) / 256 : 64);
  note_launch();
  pack_u16_kernel<<<dim3(gx, grid_rows(rows)), 256, 0, s>>>(src, rows, cols, src_ld, dst, dst_ld);
  return cudaGetLastError();
}

cudaError_t launch_split_tf32(const float* A, const float* B, int64_t M, int64_t N, int64_t K,
                              int64_t lda, int64_t ldb, int64_t Kp, float* a_big, float* a_small,
                              float* bt_big, float* bt_small, cudaStream_t s) {
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (Kp % 4 != 0 || !al16(a_big) || !al16(a_small) || !al16(bt_big) || !al16(bt_small))
    return cudaErrorInvalidValue;  // the workspace layout guarantees these (a_big may be null)
  const bool va = al16(A) && lda % 4 == 0 && K % 4 == 0;
  const int vb = al16(B) && ldb % 4 == 0 && N % 4 == 0                                   ? 4
                 : (reinterpret_cast<uintptr_t>(B) & 7u) == 0 && ldb % 2 == 0 && N % 2 == 0 ? 2
                                                                                          : 1;
  using Kern = void (*)(const float*, const float*, int64_t, int64_t, int64_t, int64_t, int64_t,
                       int64_t, int, float*, float*, float*, float*);
  const Kern kerns[2][3] = {{split_vec_kernel<false, 1>, split_vec_kernel<false, 2>,
                             split_vec_kernel<false, 4>},
                            {split_vec_kernel<true, 1>, split_vec_kernel<true, 2>,
                             split_vec_kernel<true, 4>}};
  const Kern kern = kerns[va ? 1 : 0][vb == 4 ? 2 : vb - 1];
  // Exactly one wave of resident blocks (registers decide how many fit: 5
  // per SM at 45 registers a thread, 3 at 70), shared between the operands in
  // proportion to their sizes.  Every block has an equal share of the work,
  // so a block left for a second wave would start when the others end and
  // run with too few loads in flight to keep HBM busy.
  int dev = 0, sms = 148, per_sm = 0;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, SPLIT_THREADS, 0) !=
          cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const int64_t total = static_cast<int64_t>(sms) * per_sm;
  const int64_t b_tiles = ((N + SPLIT_TILE - 1) / SPLIT_TILE) * ((K + SPLIT_TILE - 1) / SPLIT_TILE);
  // bytes per element: A 4 read + 8 written (4 without A_big), B 4 + 8
  const double a_w = a_big ? 12.0 : 8.0;
  const double a_share = a_w * M / (a_w * M + 12.0 * N);
  int64_t a_blocks = static_cast<int64_t>(a_share * total);
  a_blocks = a_blocks < 1 ? 1 : (a_blocks > M ? M : a_blocks);
  int64_t b_blocks = total - a_blocks;
  b_blocks = b_blocks < 1 ? 1 : (b_blocks > b_tiles ? b_tiles : b_blocks);
  const unsigned grid = static_cast<unsigned>(a_blocks + b_blocks);
  const int ab = static_cast<int>(a_blocks);
  note_launch();
  kern<<<grid, SPLIT_THREADS, 0, s>>>(A, B, M, N, K, lda, ldb, Kp, ab, a_big, a_small, bt_big,
                                      bt_small);
  return cudaGetLastError();
}

}  // namespace mhr
