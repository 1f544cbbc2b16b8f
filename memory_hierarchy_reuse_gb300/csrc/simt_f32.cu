// Strict-FP32 GEMM on the SIMT pipes: C = A * B, all row-major, fp32 FMA with
// fp32 accumulation.
//
// This is the pages' shared-memory tiled kernel ("矩阵乘法 tiling", section 四;
// "CUDA 编程系列之三", section 6) taken two levels further, as the pages point
// to in "矩阵乘法 tiling", sections 三 and 五 (one thread owns several outputs,
// the accumulator lives in registers):
//   * a 128 x 128 output tile per block: each A element staged in shared
//     memory feeds 128 outputs and each B element 128 outputs, so global
//     traffic is MNK (1/128 + 1/128) elements instead of 2MNK;
//   * an 8 x 8 register block per thread (register tiling): every value read
//     from shared memory feeds 8 FMAs;
//   * a double-buffered K ring (BK = 8): the next K-tile is fetched into
//     registers while the current one is consumed, so each K step needs one
//     __syncthreads() instead of the pages' two (the second barrier's job --
//     "do not overwrite a tile still being read" -- is done by writing the
//     other buffer);
//   * edge tiles: elements outside the matrix are loaded as zero and outputs
//     outside it are not stored ("矩阵乘法 tiling", section 六;
//     "CUDA 编程系列之三", section 7);
//   * problems with few tiles: a thread-block cluster of up to 8 CTAs shares
//     each tile, each CTA taking one run of K-steps, and the partial tiles
//     are summed through distributed shared memory -- the pages' reuse idea
//     applied to the partial sums, which never travel to global memory;
//   * aligned problems whose sizes are multiples of 128 x 256 x 8 go one
//     level further still: 128 x 256 tiles, 8 x 16 outputs per thread
//     (simt_f32_wide_kernel, below).
//
// Loads are coalesced where the tile crosses the global-memory boundary (a
// warp reads consecutive addresses of one row), the A tile is stored
// transposed (k-major) in shared memory with 4 floats of row padding so the
// transposing stores do not conflict, and the compute loop reads shared memory
// as float4 (two distinct A vectors per warp, broadcast; sixteen consecutive B
// vectors per warp).
//
// The multiply-adds use Blackwell's packed fp32 instruction fma.rn.f32x2: one
// instruction performs two independent fp32 fused multiply-adds (here
// acc[i][j] and acc[i][j+1] with the same a[i]), so the 64 FMAs per k step
// take 32 issue slots instead of 64 and the FMA pipe, not instruction issue,
// sets the pace.  Each lane is an ordinary round-to-nearest fp32 FMA, so the
// results are bit-identical to scalar fmaf in the same order.
#include <cuda_runtime.h>
#include <cstdint>

#include "mhr_internal.h"

namespace mhr {
namespace {

constexpr int BM = 128, BN = 128, BK = 8, NT = 256, APAD = 4;
constexpr int GROUP_M = 8;  // tile rows swept together (L2 reuse of B column strips)
// Cluster split: each CTA's partial 128 x 128 tile in shared memory, rows
// padded by 4 floats.
constexpr int RLD = BN + 4;
constexpr int RED_BYTES = BM * RLD * 4;

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_barrier() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// 16-byte load of shared address `addr` in the cluster's CTA `rank`.
__device__ __forceinline__ float4 ld_peer_v4(uint32_t addr, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(addr), "r"(rank));
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(a)
               : "memory");
  return v;
}

// d = a * b + c on two fp32 lanes packed in 64-bit registers.
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t dup2(float x) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %1};" : "=l"(d) : "f"(x));
  return d;
}
__device__ __forceinline__ float2 unpack2(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}

// k_mid > 0 splits every tile's K range in two at k_mid (a multiple of BK):
// blocks [0, tiles) take [0, k_mid), blocks [tiles, 2 tiles) take [k_mid, K),
// and both add their partial sums into C, which the caller has zeroed.  Two
// addends onto zero give the same fp32 sum in either order, so the result is
// reproducible bit for bit.
//
// CLUSTER: the kernel is launched in clusters of S CTAs (2, 4 or 8), one
// cluster per tile; rank r takes the r-th of S equal runs of K-steps (the
// last runs may be short or empty).  The S partial tiles meet in distributed
// shared memory: rank r sums rows [r * 128 / S, (r + 1) * 128 / S) of all S
// partial tiles, in rank order, and stores them.  One fixed order per
// element: bit-reproducible, with no atomics and no zeroing of C.  Used when
// the tiles alone would leave most SMs idle.
//
// WB, WC: the widest loads of B and stores of C that their alignment allows,
// in floats (4: 16-byte aligned with a leading dimension a multiple of 4; 2:
// 8-byte aligned with an even one; 1).  A column group of 4 starts at a
// multiple of 4 from the tile's first column, so either width divides it.
template <bool VA, int WB, int WC, bool CLUSTER>
__global__ void __launch_bounds__(NT, 2)
    simt_f32_kernel(const float* __restrict__ A, const float* __restrict__ B,
                    float* __restrict__ C, int64_t M, int64_t N, int64_t K, int64_t lda,
                    int64_t ldb, int64_t ldc, int64_t tiles_m, int64_t tiles_n, int64_t k_mid) {
  __shared__ __align__(16) float As[2][BK][BM + APAD];
  __shared__ __align__(16) float Bs[2][BK][BN];

  const int tid = threadIdx.x;
  int64_t t, k_begin, k_end;
  uint32_t crank = 0, csize = 1;
  if constexpr (CLUSTER) {
    crank = cluster_rank();
    csize = cluster_size();
    t = blockIdx.x / csize;
    const int64_t per = ((K + BK - 1) / BK + csize - 1) / csize * BK;  // K per rank
    k_begin = crank * per < K ? crank * per : K;
    k_end = k_begin + per < K ? k_begin + per : K;
  } else {
    const int64_t tiles = tiles_m * tiles_n;
    const bool second_half = k_mid > 0 && static_cast<int64_t>(blockIdx.x) >= tiles;
    k_begin = second_half ? k_mid : 0;
    k_end = k_mid > 0 && !second_half ? k_mid : K;
    t = second_half ? blockIdx.x - tiles : blockIdx.x;
  }
  // Grouped raster over a 1-D grid: blocks launched together cover GROUP_M
  // tile rows, column by column.
  const int64_t group_size = GROUP_M * tiles_n;
  const int64_t first_m = (t / group_size) * GROUP_M;
  const int64_t gm = tiles_m - first_m < GROUP_M ? tiles_m - first_m : GROUP_M;
  const int64_t r = t % group_size;
  const int64_t m0 = (first_m + r % gm) * BM;
  const int64_t n0 = (r / gm) * BN;

  // Load mapping: A tile 128 rows x 8 k, 4 consecutive k per thread; B tile
  // 8 k x 128 cols, 4 consecutive columns per thread.
  const int a_row = tid >> 1, a_k = (tid & 1) * 4;
  const int b_k = tid >> 5, b_col = (tid & 31) * 4;
  const bool a_row_ok = m0 + a_row < M;
  const int64_t b_col_g = n0 + b_col;
  const float* a_ptr = A + (a_row_ok ? (m0 + a_row) * lda : 0) + a_k;
  const float* b_ptr = B + static_cast<int64_t>(b_k) * ldb + b_col_g;

  // Compute mapping: thread (ty, tx) owns rows {4ty..4ty+3, 64+4ty..64+4ty+3}
  // and columns {4tx..4tx+3, 64+4tx..64+4tx+3} of the tile.
  const int ty = tid >> 4, tx = tid & 15;

  // acc2[i][p] holds outputs (i, 2p) and (i, 2p + 1) of the 8 x 8 block.
  uint64_t acc2[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int p = 0; p < 4; ++p) acc2[i][p] = 0ull;

  float ra[4], rb[4];
  auto fetch = [&](int64_t k0) {
    const int64_t ka = k0 + a_k;
    if (VA && a_row_ok && ka + 4 <= K) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(a_ptr + k0));
      ra[0] = v.x; ra[1] = v.y; ra[2] = v.z; ra[3] = v.w;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) ra[i] = (a_row_ok && ka + i < K) ? __ldg(a_ptr + k0 + i) : 0.f;
    }
    const int64_t kb = k0 + b_k;
    const float* bp = b_ptr + k0 * ldb;
    if (WB == 4 && kb < K && b_col_g + 4 <= N) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(bp));
      rb[0] = v.x; rb[1] = v.y; rb[2] = v.z; rb[3] = v.w;
    } else if (WB == 2 && kb < K && b_col_g + 4 <= N) {
      const float2 v0 = __ldg(reinterpret_cast<const float2*>(bp));
      const float2 v1 = __ldg(reinterpret_cast<const float2*>(bp + 2));
      rb[0] = v0.x; rb[1] = v0.y; rb[2] = v1.x; rb[3] = v1.y;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) rb[i] = (kb < K && b_col_g + i < N) ? __ldg(bp + i) : 0.f;
    }
  };
  auto stash = [&](int buf) {
#pragma unroll
    for (int i = 0; i < 4; ++i) As[buf][a_k + i][a_row] = ra[i];
    *reinterpret_cast<float4*>(&Bs[buf][b_k][b_col]) = make_float4(rb[0], rb[1], rb[2], rb[3]);
  };

  const int64_t nk = (k_end - k_begin + BK - 1) / BK;
  fetch(k_begin);
  stash(0);
  __syncthreads();

  for (int64_t kt = 0; kt < nk; ++kt) {
    const int cur = static_cast<int>(kt & 1);
    if (kt + 1 < nk) fetch(k_begin + (kt + 1) * BK);
#pragma unroll
    for (int k = 0; k < BK; ++k) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[cur][k][ty * 4]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[cur][k][64 + ty * 4]);
      const ulonglong2 b0 = *reinterpret_cast<const ulonglong2*>(&Bs[cur][k][tx * 4]);
      const ulonglong2 b1 = *reinterpret_cast<const ulonglong2*>(&Bs[cur][k][64 + tx * 4]);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const uint64_t b[4] = {b0.x, b0.y, b1.x, b1.y};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint64_t ai = dup2(a[i]);
#pragma unroll
        for (int p = 0; p < 4; ++p) acc2[i][p] = ffma2(ai, b[p], acc2[i][p]);
      }
    }
    if (kt + 1 < nk) stash(cur ^ 1);
    __syncthreads();
  }

  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const float2 v = unpack2(acc2[i][p]);
      acc[i][2 * p] = v.x;
      acc[i][2 * p + 1] = v.y;
    }
  if constexpr (CLUSTER) {
    extern __shared__ __align__(16) float red[];  // BM x RLD: this rank's partial tile
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int row = i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4);
#pragma unroll
      for (int h = 0; h < 2; ++h)
        *reinterpret_cast<float4*>(&red[row * RLD + h * 64 + tx * 4]) =
            make_float4(acc[i][4 * h], acc[i][4 * h + 1], acc[i][4 * h + 2], acc[i][4 * h + 3]);
    }
    cluster_barrier();  // every rank's partial tile is written
    const uint32_t red0 = static_cast<uint32_t>(__cvta_generic_to_shared(red));
    const int rows = BM / static_cast<int>(csize);
    for (int idx = tid; idx < rows * (BN / 4); idx += NT) {
      const int r = static_cast<int>(crank) * rows + idx / (BN / 4);
      const int c = (idx % (BN / 4)) * 4;
      const uint32_t addr = red0 + static_cast<uint32_t>((r * RLD + c) * 4);
      // all loads first (their latencies overlap), then the sum in rank order
      float4 w[8];
#pragma unroll
      for (uint32_t q = 0; q < 8; ++q)
        if (q < csize) w[q] = ld_peer_v4(addr, q);
      float4 v = w[0];
#pragma unroll
      for (uint32_t q = 1; q < 8; ++q)
        if (q < csize) {
          v.x += w[q].x;
          v.y += w[q].y;
          v.z += w[q].z;
          v.w += w[q].w;
        }
      const int64_t row = m0 + r, col = n0 + c;
      if (row >= M) continue;
      float* crow = C + row * ldc;
      if (WC == 4 && col + 4 <= N) {
        *reinterpret_cast<float4*>(crow + col) = v;
      } else if (WC == 2 && col + 4 <= N) {
        *reinterpret_cast<float2*>(crow + col) = make_float2(v.x, v.y);
        *reinterpret_cast<float2*>(crow + col + 2) = make_float2(v.z, v.w);
      } else {
        const float w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (col + j < N) crow[col + j] = w[j];
      }
    }
    cluster_barrier();  // no rank leaves while another still reads its tile
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int64_t row = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
      if (row >= M) continue;
      float* crow = C + row * ldc;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t col = n0 + h * 64 + tx * 4;
        const float4 v =
            make_float4(acc[i][4 * h], acc[i][4 * h + 1], acc[i][4 * h + 2], acc[i][4 * h + 3]);
        if (WC == 4 && col + 4 <= N) {
          if (k_mid > 0)
            atomicAdd(reinterpret_cast<float4*>(crow + col), v);
          else
            *reinterpret_cast<float4*>(crow + col) = v;
        } else if (WC == 2 && col + 4 <= N) {
          const float2 lo = make_float2(v.x, v.y), hi = make_float2(v.z, v.w);
          if (k_mid > 0) {
            atomicAdd(reinterpret_cast<float2*>(crow + col), lo);
            atomicAdd(reinterpret_cast<float2*>(crow + col + 2), hi);
          } else {
            *reinterpret_cast<float2*>(crow + col) = lo;
            *reinterpret_cast<float2*>(crow + col + 2) = hi;
          }
        } else {
          const float w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (col + j < N) {
              if (k_mid > 0)
                atomicAdd(crow + col + j, w[j]);
              else
                crow[col + j] = w[j];
            }
        }
      }
    }
  }
}

// ------------------------------------------------------------------ wide tiles
//
// Problems whose sizes are multiples of a 128 x 256 x 8 tile, with every
// operand 16-byte aligned (leading dimensions multiples of 4), can take a
// wider tile (simt_wide_plan decides, at the end of this file): one block of
// 256 threads per SM, each thread an 8 x 16 register
// block (rows {4ty..4ty+3, 64+4ty..64+4ty+3}, columns {64h+4tx..64h+4tx+3 :
// h = 0..3}).  Every A value read from shared memory then feeds 16 FMAs and
// every B value 8, so a k step issues 64 packed FMAs against 14 other
// instructions (8 against 6 in the kernel above), and global traffic falls to
// MNK (1/256 + 1/128) elements.  Nothing is masked.  Same double-buffered K
// ring, same k order per output (bit-identical to the kernel above for the
// same K split).  k_mid > 0: two K halves added into a zeroed C, as above.
// GB300, 4096^3 with the split, against the kernel above: 2406 -> 2188 us;
// 8192^3 18.2 -> 17.3 ms.
constexpr int WBN = 256;

__global__ void __launch_bounds__(NT, 1)
    simt_f32_wide_kernel(const float* __restrict__ A, const float* __restrict__ B,
                         float* __restrict__ C, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                         int64_t tiles_m, int64_t tiles_n, int64_t k_mid) {
  __shared__ __align__(16) float As[2][BK][BM + APAD];
  __shared__ __align__(16) float Bs[2][BK][WBN];
  const int tid = threadIdx.x;
  const int64_t tiles = tiles_m * tiles_n;
  const bool second_half = k_mid > 0 && static_cast<int64_t>(blockIdx.x) >= tiles;
  const int64_t k_begin = second_half ? k_mid : 0;
  const int64_t k_end = k_mid > 0 && !second_half ? k_mid : K;
  const int64_t t = second_half ? blockIdx.x - tiles : blockIdx.x;
  const int64_t group_size = GROUP_M * tiles_n;
  const int64_t first_m = (t / group_size) * GROUP_M;
  const int64_t gm = tiles_m - first_m < GROUP_M ? tiles_m - first_m : GROUP_M;
  const int64_t r = t % group_size;
  const int64_t m0 = (first_m + r % gm) * BM;
  const int64_t n0 = (r / gm) * WBN;

  // A tile 128 rows x 8 k: 4 consecutive k per thread; B tile 8 k x 256
  // columns: two runs of 4 columns per thread, 128 apart.
  const int a_row = tid >> 1, a_k = (tid & 1) * 4;
  const int b_k = tid >> 5, b_col = (tid & 31) * 4;
  const float* a_ptr = A + (m0 + a_row) * lda + a_k + k_begin;
  const float* b_ptr = B + (b_k + k_begin) * ldb + n0 + b_col;
  const int ty = tid >> 4, tx = tid & 15;

  uint64_t acc2[8][8];  // acc2[i][p]: outputs (i, 2p), (i, 2p + 1) of the 8 x 16 block
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int p = 0; p < 8; ++p) acc2[i][p] = 0ull;

  float4 ra, rb0, rb1;
  auto fetch = [&](int64_t k0) {
    ra = __ldg(reinterpret_cast<const float4*>(a_ptr + k0));
    const float* bp = b_ptr + k0 * ldb;
    rb0 = __ldg(reinterpret_cast<const float4*>(bp));
    rb1 = __ldg(reinterpret_cast<const float4*>(bp + 128));
  };
  auto stash = [&](int buf) {
    As[buf][a_k + 0][a_row] = ra.x;
    As[buf][a_k + 1][a_row] = ra.y;
    As[buf][a_k + 2][a_row] = ra.z;
    As[buf][a_k + 3][a_row] = ra.w;
    *reinterpret_cast<float4*>(&Bs[buf][b_k][b_col]) = rb0;
    *reinterpret_cast<float4*>(&Bs[buf][b_k][128 + b_col]) = rb1;
  };

  const int64_t nk = (k_end - k_begin) / BK;
  fetch(0);
  stash(0);
  __syncthreads();
  for (int64_t kt = 0; kt < nk; ++kt) {
    const int cur = static_cast<int>(kt & 1);
    if (kt + 1 < nk) fetch((kt + 1) * BK);
#pragma unroll
    for (int k = 0; k < BK; ++k) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[cur][k][ty * 4]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[cur][k][64 + ty * 4]);
      uint64_t b[8];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const ulonglong2 v = *reinterpret_cast<const ulonglong2*>(&Bs[cur][k][64 * h + tx * 4]);
        b[2 * h] = v.x;
        b[2 * h + 1] = v.y;
      }
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint64_t ai = dup2(a[i]);
#pragma unroll
        for (int p = 0; p < 8; ++p) acc2[i][p] = ffma2(ai, b[p], acc2[i][p]);
      }
    }
    if (kt + 1 < nk) stash(cur ^ 1);
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float* crow = C + (m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4))) * ldc + n0 + tx * 4;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const float2 v0 = unpack2(acc2[i][2 * h]), v1 = unpack2(acc2[i][2 * h + 1]);
      const float4 v = make_float4(v0.x, v0.y, v1.x, v1.y);
      if (k_mid > 0)
        atomicAdd(reinterpret_cast<float4*>(crow + 64 * h), v);
      else
        *reinterpret_cast<float4*>(crow + 64 * h) = v;
    }
  }
}

// C = 0 for the wide kernel's K halves: rows of N floats (N a multiple of 4,
// C 16-byte aligned, ldc a multiple of 4), 16-byte stores, a grid-stride
// loop over 16-byte chunks.
__global__ void zero_rows_v4_kernel(float* C, int64_t M, int64_t N, int64_t ldc) {
  const int64_t n4 = N / 4, total = M * n4;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    *reinterpret_cast<float4*>(C + (i / n4) * ldc + 4 * (i % n4)) = make_float4(0.f, 0.f, 0.f, 0.f);
}

// Whether splitting every one of `blocks` tiles into two K halves shortens
// the deepest queue of blocks on one SM by more than 7 % (see launch_t); each
// half keeps at least 64 K steps.
bool halves_pay(int64_t blocks, int64_t K, int sms) {
  const int64_t whole = (blocks + sms - 1) / sms;
  const int64_t halves = (2 * blocks + sms - 1) / sms;
  return K >= 2 * 64 * BK && blocks < (int64_t{1} << 30) && halves < 2 * whole * 0.93;
}

// Wide-tile launch, when simt_wide_plan picks it; returns false (launching
// nothing) when it does not.
bool launch_wide(const float* A, const float* B, float* C, int64_t M, int64_t N, int64_t K,
                 int64_t lda, int64_t ldb, int64_t ldc, int sms, int wide_mode, cudaStream_t s,
                 cudaError_t* err) {
  const int plan = simt_wide_plan(M, N, K, sms, wide_mode);
  if (plan == 0) return false;
  const int64_t tiles_m = M / BM, tiles_n = N / WBN, tiles = tiles_m * tiles_n;
  const int64_t k_mid = plan == 2 ? (K / 2 + BK - 1) / BK * BK : 0;
  if (k_mid > 0) {
    note_launch();
    zero_rows_v4_kernel<<<static_cast<unsigned>(4 * sms), 256, 0, s>>>(C, M, N, ldc);
    if ((*err = cudaGetLastError()) != cudaSuccess) return true;
  }
  const int64_t blocks = k_mid > 0 ? 2 * tiles : tiles;
  note_main_kernel(k_mid > 0 ? "simt_f32_kernel<wide,split-K>" : "simt_f32_kernel<wide>",
                   static_cast<int>(blocks), static_cast<int>(tiles));
  simt_f32_wide_kernel<<<static_cast<unsigned>(blocks), NT, 0, s>>>(A, B, C, K, lda, ldb, ldc,
                                                                     tiles_m, tiles_n, k_mid);
  *err = cudaGetLastError();
  return true;
}

template <bool VA, int WB, int WC>
cudaError_t launch_t(const float* A, const float* B, float* C, int64_t M, int64_t N, int64_t K,
                     int64_t lda, int64_t ldb, int64_t ldc, int wide_mode, cudaStream_t s) {
  const int64_t tiles_m = (M + BM - 1) / BM, tiles_n = (N + BN - 1) / BN;
  const int64_t tiles = tiles_m * tiles_n;
  // Split every tile along K when that shortens the busiest SM's queue.  On
  // GB300 the time of this kernel follows the largest number of blocks any
  // SM runs, ceil(tiles / SMs) -- a block alone on its SM finishes no sooner
  // than one sharing it -- so halves help when the last layer of blocks is
  // thin: ceil(2 tiles / SMs) / 2 against ceil(tiles / SMs).  Measured at
  // K = 4096: 320 tiles 40.2 -> 48.1 TFLOPS split (3 against 2.5 block
  // times); 400, 576 and 1024 tiles equal or 1 % slower split (3/3, 4/4,
  // 7/7), which is what the zero fill and the second add cost.  Each half
  // keeps at least 64 K steps.
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaError_t e;
  if (VA && WB == 4 && WC == 4 && launch_wide(A, B, C, M, N, K, lda, ldb, ldc, sms, wide_mode, s, &e))
    return e;
  // Few tiles (at most half as many as SMs): a cluster of S CTAs per tile,
  // the largest S in {8, 4, 2} that keeps one CTA per SM and at least two
  // K-steps per rank.
  const int64_t nk = (K + BK - 1) / BK;
  int cs = 1;
  if (2 * tiles <= sms)
    for (int c = 8; c >= 2; c /= 2)
      if (tiles * c <= sms && nk >= 2 * c) {
        cs = c;
        break;
      }
  if (cs > 1) {
    auto kern = simt_f32_kernel<VA, WB, WC, true>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  RED_BYTES)) != cudaSuccess)
      return e;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(tiles * cs));
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = RED_BYTES;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    note_main_kernel("simt_f32_kernel<cluster-K>", static_cast<int>(tiles * cs),
                     static_cast<int>(tiles));
    if ((e = cudaLaunchKernelEx(&cfg, kern, A, B, C, M, N, K, lda, ldb, ldc, tiles_m, tiles_n,
                                int64_t{0})) != cudaSuccess)
      return e;
    return cudaGetLastError();
  }
  const int64_t k_mid = halves_pay(tiles, K, sms) ? (K / 2 + BK - 1) / BK * BK : 0;
  if (k_mid > 0 && (e = launch_zero_fill(C, M, N, ldc, s)) != cudaSuccess) return e;
  const int64_t blocks = k_mid > 0 ? 2 * tiles : tiles;
  note_main_kernel(k_mid > 0 ? "simt_f32_kernel<split-K>" : "simt_f32_kernel",
                   static_cast<int>(blocks), static_cast<int>(tiles));
  simt_f32_kernel<VA, WB, WC, false><<<static_cast<unsigned>(blocks), NT, 0, s>>>(
      A, B, C, M, N, K, lda, ldb, ldc, tiles_m, tiles_n, k_mid);
  return cudaGetLastError();
}

// The widest access, in floats (4, 2 or 1), that every row of a matrix at `p`
// with leading dimension `ld` allows.
inline int vec_width(const void* p, int64_t ld) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  if ((a & 15u) == 0 && ld % 4 == 0) return 4;
  if ((a & 7u) == 0 && ld % 2 == 0) return 2;
  return 1;
}

template <bool VA, int WB>
cudaError_t launch_wc(const float* A, const float* B, float* C, int64_t M, int64_t N, int64_t K,
                      int64_t lda, int64_t ldb, int64_t ldc, int wc, int wide_mode,
                      cudaStream_t s) {
  switch (wc) {
    case 4: return launch_t<VA, WB, 4>(A, B, C, M, N, K, lda, ldb, ldc, wide_mode, s);
    case 2: return launch_t<VA, WB, 2>(A, B, C, M, N, K, lda, ldb, ldc, wide_mode, s);
    default: return launch_t<VA, WB, 1>(A, B, C, M, N, K, lda, ldb, ldc, wide_mode, s);
  }
}

template <bool VA>
cudaError_t launch_wb(const float* A, const float* B, float* C, int64_t M, int64_t N, int64_t K,
                      int64_t lda, int64_t ldb, int64_t ldc, int wb, int wc, int wide_mode,
                      cudaStream_t s) {
  switch (wb) {
    case 4: return launch_wc<VA, 4>(A, B, C, M, N, K, lda, ldb, ldc, wc, wide_mode, s);
    case 2: return launch_wc<VA, 2>(A, B, C, M, N, K, lda, ldb, ldc, wc, wide_mode, s);
    default: return launch_wc<VA, 1>(A, B, C, M, N, K, lda, ldb, ldc, wc, wide_mode, s);
  }
}

}  // namespace

// The estimate behind the wide kernel's choice: the time of either kernel
// follows the deepest queue of blocks on one SM, ceil(blocks / SMs) block
// times (half block times with K halves), and a 128 x 256 block takes 11/6 of
// a 128 x 128 block's time.  GB300, one kernel against the other on the same
// shape: 4096^3 3.5 wide block times, 2188 us, against 7 narrow ones,
// 2406 us (ratio 1.82); 2048^3 1.74; 4096 x 4096 x 1024 1.88; 8192^3 1.83.
int simt_wide_plan(int64_t M, int64_t N, int64_t K, int sms, int wide_mode) {
  if (wide_mode == 1 || sms < 1 || M % BM || N % WBN || K % BK) return 0;
  const int64_t tiles = (M / BM) * (N / WBN);
  if (tiles >= (int64_t{1} << 30)) return 0;
  const bool split = halves_pay(tiles, K, sms);
  if (wide_mode != 2) {
    // fewer wide tiles than half the SMs: the 128 x 128 kernel spreads wider
    if (2 * tiles < sms) return 0;
    const int64_t wide_q = split ? (2 * tiles + sms - 1) / sms : 2 * ((tiles + sms - 1) / sms);
    const int64_t narrow = 2 * tiles;
    const int64_t narrow_q = halves_pay(narrow, K, sms) ? (2 * narrow + sms - 1) / sms
                                                        : 2 * ((narrow + sms - 1) / sms);
    if (11 * wide_q >= 6 * narrow_q) return 0;
  }
  return split ? 2 : 1;
}

// Requires M, N, K >= 1 and ceil(M/128) * ceil(N/128) < 2^31.  Validation is the caller's.
cudaError_t launch_simt_f32(const float* A, const float* B, float* C, int64_t M, int64_t N,
                            int64_t K, int64_t lda, int64_t ldb, int64_t ldc, int wide_mode,
                            cudaStream_t s) {
  const int wb = vec_width(B, ldb), wc = vec_width(C, ldc);
  return vec_width(A, lda) == 4
             ? launch_wb<true>(A, B, C, M, N, K, lda, ldb, ldc, wb, wc, wide_mode, s)
             : launch_wb<false>(A, B, C, M, N, K, lda, ldb, ldc, wb, wc, wide_mode, s);
}

}  // namespace mhr
