// Shared pieces of the tensor-core GEMM kernels for sm_103a (TMA -> mbarrier
// shared-memory ring -> tcgen05.mma with a TMEM accumulator -> TMA-store
// epilogue): kinds, the parameter block, the tile schedule, bounded waits and
// the epilogue's chunk store.  The single-CTA kernel is in tc_gemm_1cta.cu,
// the CTA-pair kernel in tc_gemm_pair.cu.
//
// The method is the pages' tiling ("矩阵乘法 tiling", sections 二-四;
// "CUDA 深入浅出（二）", sections "分块之后怎么读" and "推广到整个 N×N 矩阵"):
// one output tile per work unit, K walked in BK-wide steps, each step staging
// an A box (BM x BK) and a B box (BK x BN) on chip and reusing every staged
// element across the whole tile.  What differs from the pages' 2016-era SIMT
// kernel is how each step is executed on Blackwell:
//
//   step                    pages                         here
//   ----------------------  ----------------------------  ------------------------------
//   global -> shared        each thread loads 1 element   one TMA box copy per operand,
//                                                          128-byte swizzle (no bank
//                                                          conflicts), OOB zero-fill
//   barrier one / two       __syncthreads() x 2           full[s] / empty[s] mbarriers
//                                                          of a STAGES-deep ring
//   multiply-accumulate     scalar FMA, acc in a register tcgen05.mma 128 x BN x K_instr,
//                                                          accumulator in TMEM
//   write C                 one store per thread          TMEM -> registers -> swizzled
//                                                          smem -> TMA store
//
// Warp roles (192 threads, one CTA per SM, persistent over tiles):
//   warp 0     TMA producer (lane 0 issues)
//   warp 1     TMEM allocator + MMA issuer (lane 0 issues)
//   warps 2-5  epilogue; warp w reads TMEM lanes 32*(w%4) .. 32*(w%4)+31
//   (the in-kernel split kinds add warps 6-13 as converters; in
//   KIND_3XTF32_SPLIT warp 0 idles)
// The accumulator is double-buffered in TMEM so the epilogue of tile i runs
// while the MMAs of tile i+1 are issued.  The kernels are launched with
// programmatic stream serialisation: their set-up overlaps the kernel before
// them, and griddepcontrol.wait precedes every access to inputs or C.
//
// Four kinds:
//   KIND_BF16:   A bf16 K-major (row-major M x K), B bf16 MN-major (row-major
//                K x N), kind::f16.
//   KIND_3XTF32: A_big, A_small K-major; B_big^T, B_small^T K-major (N x K),
//                kind::tf32, three MMAs per instruction-K step (small*big,
//                big*small, big*big).  The operands come from a split pre-pass.
//   KIND_3XTF32_SPLIT (CTA-pair kernel only): the same MMAs, but the split is
//                done in the kernel: converter warps load the fp32 operands
//                from global memory, split them and write the four tf32 parts
//                into the shared-memory ring in the layout TMA would produce.
//   KIND_3XTF32_SPLIT_TMA_A (CTA-pair kernel only): the same, except that TMA
//                stages A itself into the A_big box (the tensor core reads an
//                fp32 operand as its truncated tf32 big part) and the
//                converter warps read it there to write A_small; B goes
//                through the converters' registers as above.
//
// Every wait is bounded (DeviceCtl::wait_limit_ns).  A role that runs out of
// time sets its bit in the device status word and an abort flag in shared
// memory; the other roles see the flag and unwind; the CTA then waits
// (bounded) for its own copies and MMAs in flight, frees its TMEM and exits.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "mhr_device.cuh"
#include "mhr_internal.h"

namespace mhr {
namespace tc {

constexpr int KIND_BF16 = 0;
constexpr int KIND_3XTF32 = 1;
constexpr int KIND_3XTF32_SPLIT = 2;
constexpr int KIND_3XTF32_SPLIT_TMA_A = 3;

constexpr int EPI_WARPS = 4;
constexpr int EPI_BUF_BYTES = 32 * 32 * 4;                 // 32 rows x 32 fp32
constexpr int EPI_BYTES = EPI_WARPS * 2 * EPI_BUF_BYTES;   // 32 KB
constexpr int NUM_THREADS = 192;
// Default tile rows per raster group.  With 76 co-resident 256 x 256 pair
// tiles, 8 rows make each round of tiles about 8 x 9.5 instead of 16 x 4.75,
// so a round touches fewer A and B panels (DRAM reads of the 8192^3 bf16
// kernel: 1.11 GB against 1.30 GB at 16); on GB300 8 is 0.5-1 % faster than
// 16 at 4096^3 and 8192^3.
constexpr int GROUP_M = 8;

struct TcParams {
  int32_t M, N, K;
  // Output tile columns: 256 for the CTA-pair kernel's tiles unless the host
  // chose narrower ones (3xTF32 only, a multiple of 16), the kernel's BN
  // otherwise.
  int32_t bn;
  int32_t tiles_m, tiles_n, num_tiles, num_kb;
  // Work units of the pair kernel: tiles [0, full_units) whole; tiles
  // [full_units, num_tiles) split into two K halves, [0, kb_mid) and
  // [kb_mid, num_kb), whose results are reduce-added into a zeroed C.
  int32_t full_units, num_units, kb_mid;
  int32_t group_m;  // tile rows per raster group
  float* C;
  int64_t ldc;
  // C not TMA-aligned but its even rows are (16-byte aligned C, ldc even):
  // chunks wholly inside the tile and C store their even rows by TMA through
  // a map over rows 0, 2, 4, ... (c_even), and their odd rows through a map
  // over rows 1, 3, 5, ... whose base lies c_odd_shift columns (0, or 2 when
  // ldc is 2 mod 4) left of each odd row's start, so that it is 16-byte
  // aligned; -1: no odd-row map (the odd rows go out from registers).
  int32_t c_even, c_odd_shift;
  uint32_t* status;
  uint64_t wait_limit_ns;
  int32_t inject_stall;
  // The in-kernel split kinds only: the fp32 operands, row-major, and whether
  // A rows and B rows may be read with 16-byte loads (16-byte aligned,
  // leading dimension a multiple of 4).
  const float* A;
  const float* B;
  int64_t lda, ldb;
  int32_t vec_a, vec_b;
};

// Grouped raster: consecutive work units sweep GROUP_M tile rows column by
// column, so the CTAs resident at one time share A row strips and B column
// strips in L2 (a second level of the pages' reuse argument, one level up
// from shared memory).
__device__ __forceinline__ void tile_coords(int t, const TcParams& p, int& tm, int& tn) {
  const int group_size = p.group_m * p.tiles_n;
  const int g = t / group_size;
  const int first_m = g * p.group_m;
  const int gm = min(p.tiles_m - first_m, p.group_m);
  const int r = t - g * group_size;
  tm = first_m + r % gm;
  tn = r / gm;
}

// Work unit u of the pair kernel -> tile, K-block range, and whether its
// result is added into C (split unit) rather than stored.
struct Unit {
  int tile, kb0, kb1;
  bool reduce;
};
__device__ __forceinline__ Unit unit_of(int u, const TcParams& p) {
  Unit w;
  if (u < p.full_units) {
    w.tile = u;
    w.kb0 = 0;
    w.kb1 = p.num_kb;
    w.reduce = false;
  } else {
    const int v = u - p.full_units;
    w.tile = p.full_units + (v >> 1);
    w.kb0 = (v & 1) ? p.kb_mid : 0;
    w.kb1 = (v & 1) ? p.num_kb : p.kb_mid;
    w.reduce = true;
  }
  return w;
}

// Warp-uniform bounded wait: every lane polls; the warp agrees on the outcome.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint64_t limit,
                                          volatile int* abort_flag, uint32_t sleep_ns = 0) {
  const bool ok = mbar_wait_bounded(bar, parity, limit, abort_flag, sleep_ns);
  return __all_sync(0xffffffffu, ok);
}

// Called by a single thread: record why (first role to give up only) and
// raise the CTA's abort flag.
__device__ __forceinline__ void give_up_one(const TcParams& p, volatile int* abort_flag,
                                            uint32_t bit) {
  if (!*abort_flag) atomicOr(p.status, bit);
  *abort_flag = 1;
}

__device__ __forceinline__ void give_up(const TcParams& p, volatile int* abort_flag, uint32_t bit,
                                        int lane) {
  if (lane == 0) {
    if (!*abort_flag) atomicOr(p.status, bit);  // the first role to give up records why
    *abort_flag = 1;
  }
  __syncwarp();
}

// The odd-row part of an epilogue chunk under the even-row scheme
// (TcParams::c_even): whether the odd rows go out by TMA through the odd-row
// map, the chunk's columns 32 and 33 (the next chunk's first two, which a
// box shifted by 2 columns also covers), and which of the chunk's first two
// odd-row columns were written by the box of the chunk before it.
struct OddRows {
  bool tma = false;    // odd rows by one TMA store (or reduce-add) through tmC1
  bool lead2 = false;  // columns 0-1 of the odd rows: written by the previous chunk's box
  uint32_t e[2] = {0u, 0u};
};

// The odd-row plan of the chunk at col0 of a tile starting at n0.  With the
// map shifted by 2 columns, a box covers columns col0 + 2 .. col0 + 33, so it
// is used only when those lie inside the tile and C; the tile's first chunk
// then writes its odd rows' columns 0-1 from registers, and every later chunk
// finds them written.  Warp-uniform; TMEM columns col0 + 32 and + 33 of the
// accumulator at taddr_next are loaded when the box needs them.
__device__ __forceinline__ OddRows plan_odd_rows(const TcParams& p, int n0, int col0, int col_end,
                                                 uint32_t taddr_next) {
  OddRows o;
  if (!p.c_even || p.c_odd_shift < 0) return o;
  // the previous chunk (whole: this one starts inside the tile) had a box iff
  // its columns 2 .. 33 lay inside the tile and C
  o.lead2 = p.c_odd_shift == 2 && col0 > n0 && col0 + 2 <= col_end;
  if (col0 + 32 > col_end) return o;
  o.tma = col0 + 32 + p.c_odd_shift <= col_end;
  if (o.tma && p.c_odd_shift == 2) tmem_ld_2cols(taddr_next, o.e);
  return o;
}

// Epilogue of one 32 x 32 fp32 chunk held by a warp (lane = row, r[j] =
// column j): write it into the warp's staging box in shared memory (128-byte
// swizzle: 16-byte piece j of row r sits at position j ^ (r % 8), so both the
// row-wise writes here and the column-wise reads below are conflict-free),
// then either hand the box to one TMA store / reduce-add, or -- when C is not
// TMA-aligned -- store it two rows per warp instruction, masked to rows < M
// and columns < col_end (atomic adds for split-K units).  col_end is N, or
// the tile's last column + 1 when the tile is narrower than its last chunk
// (the TMA path is used only for tiles that are whole chunks).  `odd`: the
// odd rows' plan under the even-row scheme (plan_odd_rows).  The warp's two
// staging boxes alternate; before reusing one, the warp waits until the bulk
// group of the chunk two back has read it -- one group back when the chunk
// just before committed one (prev_group), else none.  Returns whether this
// chunk committed a bulk group.
template <bool TMA_STORE>
__device__ __forceinline__ bool stage_and_store_chunk(const uint32_t (&r)[32], uint32_t epi_base,
                                                      int ew, uint32_t chunk, int lane,
                                                      const CUtensorMap* tmC,
                                                      const CUtensorMap* tmC1, const TcParams& p,
                                                      int row0, int col0, int col_end,
                                                      bool reduce, const OddRows& odd,
                                                      bool prev_group) {
  const uint32_t stg = epi_base + (ew * 2 + (chunk & 1u)) * EPI_BUF_BYTES;
  const bool even_rows = !TMA_STORE && p.c_even;
  if (even_rows && col0 + 32 <= col_end) {
    // Even rows 0, 2, .., 30 of the chunk into the buffer's first 16 swizzled
    // rows, odd rows into the last 16; one TMA store (or reduce-add) writes
    // the even half to rows row0 / 2 .. of the even-row map.  The odd half
    // goes out through the odd-row map (staged c_odd_shift columns on, the
    // next chunk's first columns at the end) or from registers two rows per
    // warp instruction as below.
    if (lane == 0) {
      if (prev_group)
        bulk_wait_group_read<1>();
      else
        bulk_wait_group_read<0>();
    }
    __syncwarp();
    const int brow = (lane >> 1) + (lane & 1) * 16;
    const uint32_t brow_addr = stg + brow * 128;
    const bool shifted = odd.tma && p.c_odd_shift == 2 && (lane & 1);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t a = brow_addr + ((j ^ (brow & 7)) << 4);
      // a shifted odd row holds columns 2 .. 33: r[2 ..], then the next
      // chunk's two
      const uint32_t v0 = shifted ? r[4 * j + 2] : r[4 * j];
      const uint32_t v1 = shifted ? r[4 * j + 3] : r[4 * j + 1];
      const uint32_t v2 = shifted ? (j < 7 ? r[4 * j + 4] : odd.e[0]) : r[4 * j + 2];
      const uint32_t v3 = shifted ? (j < 7 ? r[4 * j + 5] : odd.e[1]) : r[4 * j + 3];
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v0), "r"(v1),
                   "r"(v2), "r"(v3)
                   : "memory");
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      if (reduce)
        tma_reduce_add_2d(tmC, stg, col0, row0 / 2);
      else
        tma_store_2d(tmC, stg, col0, row0 / 2);
      if (odd.tma) {
        const int x = col0 + 2 * p.c_odd_shift;  // the odd map's column of col0 + shift
        if (reduce)
          tma_reduce_add_2d(tmC1, stg + 16 * 128, x, row0 / 2);
        else
          tma_store_2d(tmC1, stg + 16 * 128, x, row0 / 2);
      }
      bulk_commit_group();
    }
    if (odd.tma) {
      // a box shifted by 2 columns starts at the chunk's column 2: the tile's
      // first chunk writes its odd rows' columns 0-1 itself (8-byte aligned:
      // C 16-byte aligned, ldc 2 mod 4, col0 a multiple of 16)
      if (p.c_odd_shift == 2 && !odd.lead2 && (lane & 1) && row0 + lane < p.M) {
        float* dst = p.C + static_cast<int64_t>(row0 + lane) * p.ldc + col0;
        const float2 v = make_float2(__uint_as_float(r[0]), __uint_as_float(r[1]));
        if (reduce)
          atomicAdd(reinterpret_cast<float2*>(dst), v);
        else
          *reinterpret_cast<float2*>(dst) = v;
      }
      __syncwarp();
      return true;
    }
    const int half = lane >> 4;
    const int cp = (lane & 15) * 2;
    const int col = col0 + cp;
    float2 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int rr = 16 + 2 * i + half;  // buffer row: odd row 2 (rr - 16) + 1
      const uint32_t a = stg + rr * 128 + ((((cp >> 2) ^ rr) & 7) << 4) + (cp & 3) * 4;
      asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];"
                   : "=f"(v[i].x), "=f"(v[i].y)
                   : "r"(a)
                   : "memory");
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int row = row0 + 2 * (2 * i + half) + 1;
      // (columns 0-1 of a chunk after one whose odd rows went out by TMA are
      // written already: a reduce-add must not add them twice)
      if (row < p.M && !(odd.lead2 && cp == 0)) {
        float* dst = p.C + static_cast<int64_t>(row) * p.ldc + col;  // 8-byte aligned: ldc even
        if (reduce)
          atomicAdd(reinterpret_cast<float2*>(dst), v[i]);
        else
          *reinterpret_cast<float2*>(dst) = v[i];
      }
    }
    __syncwarp();
    return true;
  }
  if (TMA_STORE) {
    if (lane == 0) bulk_wait_group_read<1>();  // the store that last used this buffer has read it
  } else if (even_rows && lane == 0) {         // (a chunk at the tile's edge; see above)
    if (prev_group)
      bulk_wait_group_read<1>();
    else
      bulk_wait_group_read<0>();
  }
  __syncwarp();
  const uint32_t row_addr = stg + lane * 128;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t a = row_addr + ((j ^ (lane & 7)) << 4);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(r[4 * j]),
                 "r"(r[4 * j + 1]), "r"(r[4 * j + 2]), "r"(r[4 * j + 3])
                 : "memory");
  }
  if (TMA_STORE) {
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      if (reduce)
        tma_reduce_add_2d(tmC, stg, col0, row0);
      else
        tma_store_2d(tmC, stg, col0, row0);
      bulk_commit_group();
    }
    return true;
  } else {
    __syncwarp();
    // Two rows per step, two adjacent columns per lane: lanes 0-15 take row
    // i, lanes 16-31 row i + 1.  A pair whose address is 8-byte aligned (all
    // of them when C and ldc are even) goes out as one 8-byte store or atomic
    // add, else as two 4-byte ones.  All sixteen shared-memory reads are
    // issued before the first store, so the chunk waits for one shared-memory
    // round trip, not one per step.
    const int half = lane >> 4;
    const int cp = (lane & 15) * 2;  // column pair within the chunk
    const int col = col0 + cp;
    float2 v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int rr = 2 * i + half;
      const uint32_t a = stg + rr * 128 + ((((cp >> 2) ^ rr) & 7) << 4) + (cp & 3) * 4;
      asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];"
                   : "=f"(v[i].x), "=f"(v[i].y)
                   : "r"(a)
                   : "memory");
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int row = row0 + 2 * i + half;
      // (odd rows: see above; half = 1 is the odd rows)
      if (row < p.M && col < col_end && !(odd.lead2 && half == 1 && cp == 0)) {
        float* dst = p.C + static_cast<int64_t>(row) * p.ldc + col;
        if (col + 1 < col_end && (reinterpret_cast<uintptr_t>(dst) & 7u) == 0) {
          if (reduce)
            atomicAdd(reinterpret_cast<float2*>(dst), v[i]);
          else
            *reinterpret_cast<float2*>(dst) = v[i];
        } else {
          if (reduce) {
            atomicAdd(dst, v[i].x);
            if (col + 1 < col_end) atomicAdd(dst + 1, v[i].y);
          } else {
            dst[0] = v[i].x;
            if (col + 1 < col_end) dst[1] = v[i].y;
          }
        }
      }
    }
    __syncwarp();  // the box is free for the next chunk
  }
  return false;
}

// ------------------------------------------------------------------ host side

// Parameter block for a grid of tile_m x tile_n tiles walking K in bk steps.
inline TcParams make_params(int64_t M, int64_t N, int64_t K, int tile_m, int tile_n, int bk,
                            float* C, int64_t ldc, const DeviceCtl& ctl) {
  TcParams p;
  p.M = static_cast<int32_t>(M);
  p.N = static_cast<int32_t>(N);
  p.K = static_cast<int32_t>(K);
  p.bn = tile_n;
  p.tiles_m = static_cast<int32_t>((M + tile_m - 1) / tile_m);
  p.tiles_n = static_cast<int32_t>((N + tile_n - 1) / tile_n);
  p.num_tiles = p.tiles_m * p.tiles_n;
  p.num_kb = static_cast<int32_t>((K + bk - 1) / bk);
  p.full_units = p.num_tiles;
  p.num_units = p.num_tiles;
  p.kb_mid = p.num_kb;
  p.group_m = ctl.raster_group > 0 ? ctl.raster_group : GROUP_M;
  p.C = C;
  p.ldc = ldc;
  p.c_even = 0;
  p.c_odd_shift = -1;
  p.status = ctl.status;
  p.wait_limit_ns = ctl.wait_limit_ns;
  p.inject_stall = ctl.inject_stall;
  p.A = nullptr;
  p.B = nullptr;
  p.lda = p.ldb = 0;
  p.vec_a = p.vec_b = 0;
  return p;
}

// The CTA pair's output tile (both kinds).
constexpr int PAIR_TILE_M = 256, PAIR_TILE_N = 256;

// Tensor maps of one launch: A parts, B parts (the bf16 kind uses a0 / b0
// only) and C (unused without TMA stores).  c_even: `c` maps C's even rows
// (boxes of 32 columns x 16 of those rows) for the register-store kernels.
struct TcMaps {
  CUtensorMap a0, a1, b0, b1, c, c1;
  bool c_even = false;
  int c_odd_shift = -1;  // c1: C's odd rows (TcParams::c_odd_shift); -1: none
};

// tc_gemm_1cta.cu.  bn: KIND_3XTF32's tile columns (128, or 96, 64 or 32
// with the B maps' boxes of bn rows; 0 = 128); the bf16 kind plans its own
// (256 or 128 columns over B's 64-column boxes; DeviceCtl::single_tile_n
// forces either).
cudaError_t launch_single_cta(int kind, const TcMaps& maps, float* C, int64_t M, int64_t N,
                              int64_t K, int64_t ldc, bool c_tma, bool after_prepass, int bn,
                              const DeviceCtl& ctl, cudaStream_t s);
// tc_gemm_1cta.cu: KIND_3XTF32_SPLIT_TMA_A on the single-CTA kernel, for small
// problems (one launch): maps.a0 is A's map (K-major boxes of 32 k x 128
// rows), maps.c C's map when c_tma.
cudaError_t launch_single_cta_split(const TcMaps& maps, const float* A, const float* B, float* C,
                                    int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                                    int64_t ldc, bool c_tma, const DeviceCtl& ctl,
                                    cudaStream_t s);
// tc_gemm_pair.cu.  after_prepass: the call launched a pre-pass (split or
// repack) just before this, in plain stream order; a kernel zeroing C for a
// K-split schedule then runs alongside it as a programmatic dependent.  bn:
// the pair tiles' columns (256; KIND_3XTF32 also a multiple of 16 from 128,
// a multiple of 32 with c_tma), matching the B maps' boxes of bn / 2 rows.
cudaError_t launch_cta_pair(int kind, const TcMaps& maps, float* C, int64_t M, int64_t N,
                            int64_t K, int64_t ldc, bool c_tma, bool after_prepass, int bn,
                            const DeviceCtl& ctl, cudaStream_t s);
// Zero the C tiles [q.full_units, q.num_tiles) of tile_rows x tile_cols that
// a K-split schedule reduce-adds into; after_prepass as for launch_cta_pair.
cudaError_t launch_zero_split_tiles(const TcParams& q, int tile_rows, int tile_cols,
                                    bool after_prepass, cudaStream_t s);
// The CTA-pair kernel with the 3xTF32 split done in the kernel (no workspace):
// A (M x K, pitch lda) and B (K x N, pitch ldb) row-major fp32.  `maps` holds
// the C map (TMA stores) and, with tma_a, A's map (K-major boxes of 32 k x
// 128 rows) for KIND_3XTF32_SPLIT_TMA_A; else KIND_3XTF32_SPLIT runs.
cudaError_t launch_cta_pair_split(bool tma_a, const float* A, const float* B, const TcMaps& maps,
                                  float* C, int64_t M, int64_t N, int64_t K, int64_t lda,
                                  int64_t ldb, int64_t ldc, bool c_tma, const DeviceCtl& ctl,
                                  cudaStream_t s);

}  // namespace tc
}  // namespace mhr
