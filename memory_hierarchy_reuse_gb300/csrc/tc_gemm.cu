// Tensor-core GEMM for sm_103a: TMA -> mbarrier shared-memory ring ->
// tcgen05.mma with a TMEM accumulator -> TMA-store epilogue.
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
// The accumulator is double-buffered in TMEM so the epilogue of tile i runs
// while the MMAs of tile i+1 are issued.
//
// Two kinds:
//   KIND_BF16:   A bf16 K-major (row-major M x K), B bf16 MN-major (row-major
//                K x N), BM x BN x BK = 128 x 256 x 64, 4 stages, kind::f16.
//   KIND_3XTF32: A_big, A_small K-major; B_big^T, B_small^T K-major (N x K),
//                128 x 128 x 32, 3 stages, kind::tf32, three MMAs per
//                instruction-K step (small*big, big*small, big*big).
//
// Every wait is bounded (DeviceCtl::wait_limit_ns).  A role that runs out of
// time sets its bit in the device status word and an abort flag in shared
// memory; the other roles see the flag and unwind; the CTA then waits
// (bounded) for its own copies and MMAs in flight, frees its TMEM and exits.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "mhr_device.cuh"
#include "mhr_internal.h"

namespace mhr {
namespace {

constexpr int KIND_BF16 = 0;
constexpr int KIND_3XTF32 = 1;

template <int KIND>
struct Cfg;

template <>
struct Cfg<KIND_BF16> {
  static constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
  static constexpr int A_BYTES = BM * BK * 2;              // 16 KB
  static constexpr int B_BOX_BYTES = 64 * BK * 2;          // 64 cols x 64 k = 8 KB
  static constexpr int B_BYTES = BK * BN * 2;              // 32 KB
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;    // 48 KB
  static constexpr int INSTR_K = 16;
  static constexpr uint32_t IDESC = make_idesc(1, false, true, BM, BN);
  static constexpr uint32_t TMEM_COLS = 2 * BN;            // 512
};

template <>
struct Cfg<KIND_3XTF32> {
  static constexpr int BM = 128, BN = 128, BK = 32, STAGES = 3;
  static constexpr int A_BYTES = BM * BK * 4;              // 16 KB each (big, small)
  static constexpr int B_BYTES = BN * BK * 4;              // 16 KB each (big, small)
  static constexpr int STAGE_BYTES = 2 * A_BYTES + 2 * B_BYTES;  // 64 KB
  static constexpr int INSTR_K = 8;
  static constexpr uint32_t IDESC = make_idesc(2, false, false, BM, BN);
  static constexpr uint32_t TMEM_COLS = 2 * BN;            // 256
};

constexpr int EPI_WARPS = 4;
constexpr int EPI_BUF_BYTES = 32 * 32 * 4;                 // 32 rows x 32 fp32
constexpr int EPI_BYTES = EPI_WARPS * 2 * EPI_BUF_BYTES;   // 32 KB
constexpr int NUM_THREADS = 192;
constexpr int GROUP_M = 16;  // default tile rows per raster group

template <int KIND>
struct Layout {
  using C = Cfg<KIND>;
  static constexpr int EPI_OFF = C::STAGES * C::STAGE_BYTES;
  static constexpr int BAR_OFF = EPI_OFF + EPI_BYTES;
  static constexpr int NUM_BARS = 2 * C::STAGES + 5;        // full, empty, acc_full x2, acc_empty x2, drain
  static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;   // tmem slot, abort flag
  static constexpr int USED = MISC_OFF + 16;
  static constexpr int ALLOC = USED + 1024;                 // slack for 1024-byte alignment
};

struct TcParams {
  int32_t M, N, K;
  int32_t tiles_m, tiles_n, num_tiles, num_kb;
  // Work units of the pair kernel: tiles [0, full_units) whole; tiles
  // [full_units, num_tiles) split into two K halves, [0, kb_mid) and
  // [kb_mid, num_kb), whose results are reduce-added into a zeroed C.
  int32_t full_units, num_units, kb_mid;
  int32_t group_m;  // tile rows per raster group
  float* C;
  int64_t ldc;
  uint32_t* status;
  uint64_t wait_limit_ns;
  int32_t inject_stall;
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

__device__ __forceinline__ void give_up(const TcParams& p, volatile int* abort_flag, uint32_t bit,
                                        int lane) {
  if (lane == 0) {
    if (!*abort_flag) atomicOr(p.status, bit);  // the first role to give up records why
    *abort_flag = 1;
  }
  __syncwarp();
}

// Epilogue of one 32 x 32 fp32 chunk held by a warp (lane = row, r[j] =
// column j): write it into the warp's staging box in shared memory (128-byte
// swizzle: 16-byte piece j of row r sits at position j ^ (r % 8), so both the
// row-wise writes here and the column-wise reads below are conflict-free),
// then either hand the box to one TMA store / reduce-add, or -- when C is not
// TMA-aligned -- store it row by row so each warp instruction writes 32
// consecutive floats of one row of C (masked at the edges; atomic adds for
// split-K units).
template <bool TMA_STORE>
__device__ __forceinline__ void stage_and_store_chunk(const uint32_t (&r)[32], uint32_t epi_base,
                                                      int ew, uint32_t chunk, int lane,
                                                      const CUtensorMap* tmC, const TcParams& p,
                                                      int row0, int col0, bool reduce) {
  const uint32_t stg = epi_base + (ew * 2 + (chunk & 1u)) * EPI_BUF_BYTES;
  if (TMA_STORE) {
    if (lane == 0) bulk_wait_group_read<1>();  // the store that last used this buffer has read it
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
  } else {
    __syncwarp();
    const int col = col0 + lane;
#pragma unroll 4
    for (int i = 0; i < 32; ++i) {
      const int row = row0 + i;
      const uint32_t a = stg + i * 128 + ((((lane >> 2) ^ i) & 7) << 4) + (lane & 3) * 4;
      float v;
      asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
      if (row < p.M && col < p.N) {
        float* dst = p.C + static_cast<int64_t>(row) * p.ldc + col;
        if (reduce)
          atomicAdd(dst, v);
        else
          *dst = v;
      }
    }
    __syncwarp();  // the box is free for the next chunk
  }
}

template <int KIND, bool TMA_STORE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                   const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
                   const __grid_constant__ CUtensorMap tmC, const TcParams p) {
  using Cf = Cfg<KIND>;
  using L = Layout<KIND>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + L::BAR_OFF;
  auto full_bar = [&](uint32_t s) { return bar0 + 8u * s; };
  auto empty_bar = [&](uint32_t s) { return bar0 + 8u * (Cf::STAGES + s); };
  auto accf_bar = [&](uint32_t b) { return bar0 + 8u * (2 * Cf::STAGES + b); };
  auto acce_bar = [&](uint32_t b) { return bar0 + 8u * (2 * Cf::STAGES + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * Cf::STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::MISC_OFF + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cf::STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), EPI_WARPS);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA0);
    tma_prefetch_desc(&tmB0);
    if constexpr (KIND == KIND_3XTF32) {
      tma_prefetch_desc(&tmA1);
      tma_prefetch_desc(&tmB1);
    }
    if (TMA_STORE) tma_prefetch_desc(&tmC);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Cf::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint64_t limit = p.wait_limit_ns;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    uint32_t it = 0;
    uint32_t inflight = 0;  // bit s: the latest fill of stage s had a TMA issued
    bool ok = true;
    for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
      int tm, tn;
      tile_coords(t, p, tm, tn);
      const int m0 = tm * Cf::BM, n0 = tn * Cf::BN;
      for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
        const uint32_t s = it % Cf::STAGES, ph = (it / Cf::STAGES) & 1u;
        if (!warp_wait(empty_bar(s), ph ^ 1u, limit, abort_flag)) {
          give_up(p, abort_flag, kErrTimeoutProducer, lane);
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t st = sbase + s * Cf::STAGE_BYTES;
          const int k0 = kb * Cf::BK;
          mbar_arrive_expect_tx(full_bar(s), Cf::STAGE_BYTES);
          const bool stall = p.inject_stall && blockIdx.x == 0 && it == 0;
          if (!stall) {
            if constexpr (KIND == KIND_BF16) {
              tma_load_2d(st, &tmA0, full_bar(s), k0, m0);
#pragma unroll
              for (int j = 0; j < Cf::BN / 64; ++j)
                tma_load_2d(st + Cf::A_BYTES + j * Cf::B_BOX_BYTES, &tmB0, full_bar(s), n0 + 64 * j,
                            k0);
            } else {
              tma_load_2d(st, &tmA0, full_bar(s), k0, m0);
              tma_load_2d(st + Cf::A_BYTES, &tmA1, full_bar(s), k0, m0);
              tma_load_2d(st + 2 * Cf::A_BYTES, &tmB0, full_bar(s), k0, n0);
              tma_load_2d(st + 2 * Cf::A_BYTES + Cf::B_BYTES, &tmB1, full_bar(s), k0, n0);
            }
            inflight |= 1u << s;
          } else {
            inflight &= ~(1u << s);
          }
        }
        __syncwarp();
      }
    }
    // Drain: every TMA this CTA issued must have landed before it exits.
    if (lane == 0) {
      for (uint32_t s = 0; s < static_cast<uint32_t>(Cf::STAGES) && s < it; ++s) {
        if (!(inflight & (1u << s))) continue;
        const uint32_t last = it - 1 - ((it - 1 - s) % Cf::STAGES);  // latest fill of stage s
        volatile int never = 0;
        if (!mbar_wait_bounded(full_bar(s), (last / Cf::STAGES) & 1u, limit, &never))
          atomicOr(p.status, kErrTimeoutDrain);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    uint32_t it = 0, tcount = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x, ++tcount) {
      const uint32_t buf = tcount & 1u, aph = (tcount >> 1) & 1u;
      if (!warp_wait(acce_bar(buf), aph ^ 1u, limit, abort_flag)) {
        give_up(p, abort_flag, kErrTimeoutMma, lane);
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + buf * Cf::BN;
      for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
        const uint32_t s = it % Cf::STAGES, ph = (it / Cf::STAGES) & 1u;
        if (!warp_wait(full_bar(s), ph, limit, abort_flag)) {
          give_up(p, abort_flag, kErrTimeoutMma, lane);
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t st = sbase + s * Cf::STAGE_BYTES;
          if constexpr (KIND == KIND_BF16) {
            // A: 128 rows x 128 B, K-major, 8-row groups 1024 B apart.
            // B: four 64-column boxes (8 KB apart) of 64 k-rows x 128 B,
            //    MN-major: LBO = next 64 columns, SBO = next 8 k-rows.
#pragma unroll
            for (int kk = 0; kk < Cf::BK / Cf::INSTR_K; ++kk) {
              const uint64_t ad = smem_desc_sw128(st + kk * 32, 16, 1024);
              const uint64_t bd = smem_desc_sw128(st + Cf::A_BYTES + kk * 2048, Cf::B_BOX_BYTES, 1024);
              mma_f16(d_tmem, ad, bd, Cf::IDESC, (kb > 0 || kk > 0) ? 1u : 0u);
            }
          } else {
            // All four operands K-major, 128 B rows (32 floats), 8-row groups
            // 1024 B apart; one instruction-K step (8 tf32) = 32 B.
            const uint32_t a_big = st, a_small = st + Cf::A_BYTES;
            const uint32_t b_big = st + 2 * Cf::A_BYTES, b_small = b_big + Cf::B_BYTES;
#pragma unroll
            for (int kk = 0; kk < Cf::BK / Cf::INSTR_K; ++kk) {
              const uint32_t off = kk * 32;
              const uint64_t abd = smem_desc_sw128(a_big + off, 16, 1024);
              const uint64_t asd = smem_desc_sw128(a_small + off, 16, 1024);
              const uint64_t bbd = smem_desc_sw128(b_big + off, 16, 1024);
              const uint64_t bsd = smem_desc_sw128(b_small + off, 16, 1024);
              mma_tf32(d_tmem, asd, bbd, Cf::IDESC, (kb > 0 || kk > 0) ? 1u : 0u);
              mma_tf32(d_tmem, abd, bsd, Cf::IDESC, 1u);
              mma_tf32(d_tmem, abd, bbd, Cf::IDESC, 1u);
            }
          }
          mma_commit(empty_bar(s));  // stage s may be refilled once these MMAs finish
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) mma_commit(accf_bar(buf));  // accumulator `buf` complete
      __syncwarp();
    }
    // Drain: all MMAs issued by this thread complete before TMEM is freed.
    if (lane == 0) {
      mma_commit(drain_bar);
      volatile int never = 0;
      if (!mbar_wait_bounded(drain_bar, 0, limit, &never)) atomicOr(p.status, kErrTimeoutDrain);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;           // TMEM lane quarter this warp may access
    const int ew = warp - 2;          // epilogue warp index 0..3
    uint32_t tcount = 0, chunk = 0;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x, ++tcount) {
      const uint32_t buf = tcount & 1u, aph = (tcount >> 1) & 1u;
      if (!warp_wait(accf_bar(buf), aph, limit, abort_flag)) {
        give_up(p, abort_flag, kErrTimeoutEpilogue, lane);
        break;
      }
      tc_fence_after();
      int tm, tn;
      tile_coords(t, p, tm, tn);
      const int m0 = tm * Cf::BM, n0 = tn * Cf::BN;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * Cf::BN;
#pragma unroll 1
      for (int c = 0; c < Cf::BN / 32; ++c) {
        uint32_t r[32];
        tmem_ld_32cols(taddr + c * 32, r);
        tmem_ld_wait();
        stage_and_store_chunk<TMA_STORE>(r, sbase + L::EPI_OFF, ew, chunk, lane, &tmC, p,
                                         m0 + q * 32, n0 + c * 32, false);
        ++chunk;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce_bar(buf));  // TMEM buffer `buf` may be overwritten
    }
    if constexpr (TMA_STORE) {
      if (lane == 0) bulk_wait_group<0>();
      __syncwarp();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cf::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ CTA pairs
//
// The same method one level up: two CTAs on two SMs (a cluster of 2) share
// one 256 x BN output tile.  Each CTA stages its own 128 rows of A and its own
// half of B's columns; one tcgen05.mma.cta_group::2 instruction (M = 256)
// reads both CTAs' shared memory and writes each CTA's 128 accumulator rows
// into that CTA's TMEM.  Every staged B element now feeds 256 output rows
// instead of 128, so each SM reads half as many B bytes from shared memory
// per FLOP -- the shared-memory bandwidth that binds the 1-CTA kernel.
//
// Synchronisation across the pair:
//   full[s]      (rank 0 only) both CTAs' TMA bytes complete on it; rank 0's
//                producer arms it for the pair's bytes
//   empty[s]     (both) rank 0's MMA thread commits to both CTAs' copy
//   acc_full[b]  (both) likewise, when accumulator b is complete
//   acc_empty[b] (rank 0 only) all 8 epilogue warps of the pair arrive
// On a timeout, the role that gave up raises the abort flag in both CTAs.

template <int KIND>
struct PairCfg;

#ifndef MHR_PAIR_BF16_BK
#define MHR_PAIR_BF16_BK 64
#endif
template <>
struct PairCfg<KIND_BF16> {
  static constexpr int BM = 128;                            // rows per CTA (pair: 256)
  static constexpr int BN = 256, BN_HALF = 128, BK = MHR_PAIR_BF16_BK;
  static constexpr int STAGES = BK == 64 ? 6 : 3;
  static constexpr int A_BOX_BYTES = BM * 64 * 2;           // 128 rows x 64 k = 16 KB
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BOX_BYTES = 64 * BK * 2;           // 64 columns x BK k-rows
  static constexpr int B_BYTES = BN_HALF * BK * 2;          // this CTA's half
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;     // 32 or 64 KB per CTA
  static constexpr int INSTR_K = 16;
  static constexpr uint32_t IDESC = make_idesc(1, false, true, 2 * BM, BN);
  static constexpr uint32_t TMEM_COLS = 2 * BN;             // 512
};

template <>
struct PairCfg<KIND_3XTF32> {
  static constexpr int BM = 128;
  static constexpr int BN = 256, BN_HALF = 128, BK = 32, STAGES = 3;
  static constexpr int A_BYTES = BM * BK * 4;               // 16 KB each (big, small)
  static constexpr int B_BYTES = BN_HALF * BK * 4;          // 16 KB each (big, small)
  static constexpr int STAGE_BYTES = 2 * A_BYTES + 2 * B_BYTES;  // 64 KB per CTA
  static constexpr int INSTR_K = 8;
  static constexpr uint32_t IDESC = make_idesc(2, false, false, 2 * BM, BN);
  static constexpr uint32_t TMEM_COLS = 2 * BN;             // 512
};

template <int KIND>
struct PairLayout {
  using C = PairCfg<KIND>;
  static constexpr int EPI_OFF = C::STAGES * C::STAGE_BYTES;
  static constexpr int BAR_OFF = EPI_OFF + EPI_BYTES;
  static constexpr int NUM_BARS = 2 * C::STAGES + 5;
  static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
  static constexpr int USED = MISC_OFF + 16;
  static constexpr int ALLOC = USED + 1024;
};

// Pause for `ns` nanoseconds (bounded).
__device__ __forceinline__ void pause_ns(uint64_t ns) {
  const uint64_t t0 = global_timer_ns();
  while (global_timer_ns() - t0 < ns) {
  }
}

template <int KIND, bool TMA_STORE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    tc_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA0,
                        const __grid_constant__ CUtensorMap tmA1,
                        const __grid_constant__ CUtensorMap tmB0,
                        const __grid_constant__ CUtensorMap tmB1,
                        const __grid_constant__ CUtensorMap tmC, const TcParams p) {
  using Cf = PairCfg<KIND>;
  using L = PairLayout<KIND>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + L::BAR_OFF;
  auto full_bar = [&](uint32_t s) { return bar0 + 8u * s; };
  auto empty_bar = [&](uint32_t s) { return bar0 + 8u * (Cf::STAGES + s); };
  auto accf_bar = [&](uint32_t b) { return bar0 + 8u * (2 * Cf::STAGES + b); };
  auto acce_bar = [&](uint32_t b) { return bar0 + 8u * (2 * Cf::STAGES + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * Cf::STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::MISC_OFF + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cluster = blockIdx.x >> 1, num_clusters = gridDim.x >> 1;
  const uint32_t peer_abort = mapa_shared(smem_u32(const_cast<int*>(abort_flag)), rank ^ 1u);

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cf::STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), 2 * EPI_WARPS);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA0);
    tma_prefetch_desc(&tmB0);
    if constexpr (KIND == KIND_3XTF32) {
      tma_prefetch_desc(&tmA1);
      tma_prefetch_desc(&tmB1);
    }
    if (TMA_STORE) tma_prefetch_desc(&tmC);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), Cf::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // both CTAs' barriers initialised, TMEM allocated in both
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint64_t limit = p.wait_limit_ns;

  // Give up: record why (first role only), raise the abort flag in both CTAs.
  auto give_up_one = [&](uint32_t bit) {  // called by a single thread
    if (!*abort_flag) atomicOr(p.status, bit);
    *abort_flag = 1;
    st_shared_cluster_u32(peer_abort, 1u);
  };
  auto give_up_pair = [&](uint32_t bit) {  // called by a whole warp
    if (lane == 0) give_up_one(bit);
    __syncwarp();
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producers (both CTAs)
    // One thread waits, arms and issues; the rest of the warp idles.
    if (lane == 0) {
      uint32_t it = 0, inflight = 0;
      bool ok = true;
      for (int u = cluster; ok && u < p.num_units; u += num_clusters) {
        const Unit w = unit_of(u, p);
        int tm, tn;
        tile_coords(w.tile, p, tm, tn);
        const int m0 = tm * 2 * Cf::BM + static_cast<int>(rank) * Cf::BM;
        const int nb0 = tn * Cf::BN + static_cast<int>(rank) * Cf::BN_HALF;
        for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
          const uint32_t s = it % Cf::STAGES, ph = (it / Cf::STAGES) & 1u;
          if (!mbar_wait_bounded(empty_bar(s), ph ^ 1u, limit, abort_flag)) {
            give_up_one(kErrTimeoutProducer);
            ok = false;
            break;
          }
          const uint32_t st = sbase + s * Cf::STAGE_BYTES;
          const uint32_t fb = mapa_shared(full_bar(s), 0);  // rank 0's full[s]
          const int k0 = kb * Cf::BK;
          if (leader) mbar_arrive_expect_tx(full_bar(s), 2 * Cf::STAGE_BYTES);
          const bool stall = p.inject_stall && blockIdx.x == 0 && it == 0;
          if (!stall) {
            if constexpr (KIND == KIND_BF16) {
#pragma unroll
              for (int i = 0; i < Cf::BK / 64; ++i)
                tma_load_2d_pair(st + i * Cf::A_BOX_BYTES, &tmA0, fb, k0 + 64 * i, m0);
#pragma unroll
              for (int j = 0; j < Cf::BN_HALF / 64; ++j)
#pragma unroll
                for (int i = 0; i < Cf::BK / 64; ++i)  // 64 k-rows per box, stacked
                  tma_load_2d_pair(st + Cf::A_BYTES + j * Cf::B_BOX_BYTES + i * 8192, &tmB0, fb,
                                   nb0 + 64 * j, k0 + 64 * i);
            } else {
              tma_load_2d_pair(st, &tmA0, fb, k0, m0);
              tma_load_2d_pair(st + Cf::A_BYTES, &tmA1, fb, k0, m0);
              tma_load_2d_pair(st + 2 * Cf::A_BYTES, &tmB0, fb, k0, nb0);
              tma_load_2d_pair(st + 2 * Cf::A_BYTES + Cf::B_BYTES, &tmB1, fb, k0, nb0);
            }
            inflight |= 1u << s;
          } else {
            inflight &= ~(1u << s);
          }
        }
      }
      if (leader) {
        // Rank 0 can see its full barriers: wait for every fill it armed and loaded.
        for (uint32_t s = 0; s < static_cast<uint32_t>(Cf::STAGES) && s < it; ++s) {
          if (!(inflight & (1u << s))) continue;
          const uint32_t last = it - 1 - ((it - 1 - s) % Cf::STAGES);
          volatile int never = 0;
          if (!mbar_wait_bounded(full_bar(s), (last / Cf::STAGES) & 1u, limit, &never))
            atomicOr(p.status, kErrTimeoutDrain);
        }
      }
      // After an abort, the loads this CTA issued signal rank 0's barriers,
      // which rank 1 cannot poll: give them time to land (a TMA load takes
      // microseconds) before the CTA may leave.
      if (*abort_flag) pause_ns(100000);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (rank 0)
    // One thread of rank 0 waits and issues every MMA of the pair.
    if (leader && lane == 0) {
      uint32_t it = 0, tcount = 0;
      bool ok = true;
      for (int u = cluster; ok && u < p.num_units; u += num_clusters, ++tcount) {
        const Unit w = unit_of(u, p);
        const uint32_t buf = tcount & 1u, aph = (tcount >> 1) & 1u;
        if (!mbar_wait_bounded(acce_bar(buf), aph ^ 1u, limit, abort_flag)) {
          give_up_one(kErrTimeoutMma);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * Cf::BN;
        for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
          const uint32_t s = it % Cf::STAGES, ph = (it / Cf::STAGES) & 1u;
          if (!mbar_wait_bounded(full_bar(s), ph, limit, abort_flag)) {
            give_up_one(kErrTimeoutMma);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = sbase + s * Cf::STAGE_BYTES;
          if constexpr (KIND == KIND_BF16) {
            // A: 128 rows x 128 B per CTA, K-major.  B: this CTA's two
            // 64-column boxes (8 KB apart), MN-major.
#pragma unroll
            for (int kk = 0; kk < Cf::BK / Cf::INSTR_K; ++kk) {
              const uint64_t ad =
                  smem_desc_sw128(st + (kk / 4) * Cf::A_BOX_BYTES + (kk % 4) * 32, 16, 1024);
              const uint64_t bd =
                  smem_desc_sw128(st + Cf::A_BYTES + kk * 2048, Cf::B_BOX_BYTES, 1024);
              mma_f16_pair(d_tmem, ad, bd, Cf::IDESC, (kb > w.kb0 || kk > 0) ? 1u : 0u);
            }
          } else {
            const uint32_t a_big = st, a_small = st + Cf::A_BYTES;
            const uint32_t b_big = st + 2 * Cf::A_BYTES, b_small = b_big + Cf::B_BYTES;
#pragma unroll
            for (int kk = 0; kk < Cf::BK / Cf::INSTR_K; ++kk) {
              const uint32_t off = kk * 32;
              const uint64_t abd = smem_desc_sw128(a_big + off, 16, 1024);
              const uint64_t asd = smem_desc_sw128(a_small + off, 16, 1024);
              const uint64_t bbd = smem_desc_sw128(b_big + off, 16, 1024);
              const uint64_t bsd = smem_desc_sw128(b_small + off, 16, 1024);
              mma_tf32_pair(d_tmem, asd, bbd, Cf::IDESC, (kb > w.kb0 || kk > 0) ? 1u : 0u);
              mma_tf32_pair(d_tmem, abd, bsd, Cf::IDESC, 1u);
              mma_tf32_pair(d_tmem, abd, bbd, Cf::IDESC, 1u);
            }
          }
          mma_commit_pair_multicast(empty_bar(s), 0x3);  // stage s free in both CTAs
        }
        if (!ok) break;
        mma_commit_pair_multicast(accf_bar(buf), 0x3);  // accumulator `buf` complete
      }
      mma_commit_pair(drain_bar);
      volatile int never = 0;
      if (!mbar_wait_bounded(drain_bar, 0, limit, &never)) atomicOr(p.status, kErrTimeoutDrain);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    const int ew = warp - 2;
    uint32_t tcount = 0, chunk = 0;
    for (int u = cluster; u < p.num_units; u += num_clusters, ++tcount) {
      const Unit w = unit_of(u, p);
      const uint32_t buf = tcount & 1u, aph = (tcount >> 1) & 1u;
      // The accumulator takes a whole tile's main loop to fill: back off
      // between polls instead of spinning at full issue rate.
      if (!warp_wait(accf_bar(buf), aph, limit, abort_flag, 128)) {
        give_up_pair(kErrTimeoutEpilogue);
        break;
      }
      tc_fence_after();
      int tm, tn;
      tile_coords(w.tile, p, tm, tn);
      const int m0 = tm * 2 * Cf::BM + static_cast<int>(rank) * Cf::BM;
      const int n0 = tn * Cf::BN;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * Cf::BN;
#pragma unroll 1
      for (int c = 0; c < Cf::BN / 32; ++c) {
        uint32_t r[32];
        tmem_ld_32cols(taddr + c * 32, r);
        tmem_ld_wait();
        stage_and_store_chunk<TMA_STORE>(r, sbase + L::EPI_OFF, ew, chunk, lane, &tmC, p,
                                         m0 + q * 32, n0 + c * 32, w.reduce);
        ++chunk;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(acce_bar(buf), 0));
    }
    if constexpr (TMA_STORE) {
      if (lane == 0) bulk_wait_group<0>();
      __syncwarp();
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // neither CTA leaves while the pair's MMAs or arrivals may touch it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, Cf::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ pre-passes

// Zero the C tiles of the split work units (pair tiles [full_units,
// num_tiles)), which both K halves then add into.  Block (x, y) clears rows
// [8y, 8y + 8) of split tile x.
__global__ void zero_split_tiles_kernel(TcParams p, int tile_cols) {
  const int tile = p.full_units + blockIdx.x;
  int tm, tn;
  tile_coords(tile, p, tm, tn);
  const int64_t row = static_cast<int64_t>(tm) * (8 * gridDim.y) + 8 * blockIdx.y + threadIdx.y;
  if (row >= p.M) return;
  const int64_t c0 = static_cast<int64_t>(tn) * tile_cols;
  float* crow = p.C + row * p.ldc;
  for (int c = threadIdx.x; c < tile_cols; c += blockDim.x)
    if (c0 + c < p.N) crow[c0 + c] = 0.f;
}

__global__ void zero_fill_kernel(float* C, int64_t M, int64_t N, int64_t ldc) {
  for (int64_t r = blockIdx.y; r < M; r += gridDim.y)
    for (int64_t c = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; c < N;
         c += static_cast<int64_t>(gridDim.x) * blockDim.x)
      C[r * ldc + c] = 0.f;
}

__global__ void pack_u16_kernel(const uint16_t* __restrict__ src, int64_t rows, int64_t cols,
                                int64_t src_ld, uint16_t* __restrict__ dst, int64_t dst_ld) {
  for (int64_t r = blockIdx.y; r < rows; r += gridDim.y)
    for (int64_t c = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; c < cols;
         c += static_cast<int64_t>(gridDim.x) * blockDim.x)
      dst[r * dst_ld + c] = src[r * src_ld + c];
}

// Round an fp32 value to tf32 (10 explicit mantissa bits) to nearest, ties to
// even, by integer arithmetic on the bit pattern; Inf and NaN pass unchanged.
__device__ __forceinline__ float tf32_rne(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u & 0x7F800000u) == 0x7F800000u) return x;
  u += 0x0FFFu + ((u >> 13) & 1u);
  return __uint_as_float(u & 0xFFFFE000u);
}

__device__ __forceinline__ void split_tf32(float x, float& big, float& small) {
  big = tf32_rne(x);
  const float rest = x - big;  // exact: the discarded low bits
  small = isfinite(x) ? tf32_rne(rest) : 0.f;
}

// Split of both operands in one launch.  Blocks [0, a_blocks) split rows of
// A in place order; the remaining blocks split 64 x 64 tiles of B and write
// them transposed.  VA / VB select 16-byte loads when the operand's address,
// leading dimension (and, for A, K) allow them, else 4-byte loads; the
// outputs (pitch Kp, a multiple of 4, in the 16-byte-aligned workspace) are
// always written with 16-byte stores.  Each thread keeps several loads in
// flight.
constexpr int SPLIT_THREADS = 256;
constexpr int SPLIT_TILE = 64;

__device__ __forceinline__ void split4(const float4 v, float4& b, float4& s) {
  split_tf32(v.x, b.x, s.x);
  split_tf32(v.y, b.y, s.y);
  split_tf32(v.z, b.z, s.z);
  split_tf32(v.w, b.w, s.w);
}

template <bool VA, bool VB>
__global__ void __launch_bounds__(SPLIT_THREADS)
    split_vec_kernel(const float* __restrict__ A, const float* __restrict__ B, int64_t M,
                     int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t Kp, int a_blocks,
                     float* __restrict__ a_big, float* __restrict__ a_small,
                     float* __restrict__ bt_big, float* __restrict__ bt_small) {
  __shared__ float tb[SPLIT_TILE][SPLIT_TILE + 1];
  __shared__ float ts[SPLIT_TILE][SPLIT_TILE + 1];
  const int t = threadIdx.x;
  if (static_cast<int>(blockIdx.x) < a_blocks) {
    const int64_t k4 = Kp / 4;  // 16-byte chunks of an output row (pad columns get zeros)
    for (int64_t r = blockIdx.x; r < M; r += a_blocks) {
      const float* src = A + r * lda;
      float4* db = reinterpret_cast<float4*>(a_big + r * Kp);
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
            split4(v[j], b, s);
            db[c] = b;
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
    if (VB) {
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
        split4(v[j], b, s);
        tb[kr][nc] = b.x; tb[kr][nc + 1] = b.y; tb[kr][nc + 2] = b.z; tb[kr][nc + 3] = b.w;
        ts[kr][nc] = s.x; ts[kr][nc + 1] = s.y; ts[kr][nc + 2] = s.z; ts[kr][nc + 3] = s.w;
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
        split_tf32(v[j], b, sm);
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

template <int KIND, bool TMA_STORE>
cudaError_t prepare_kernel() {
  // cudaFuncSetAttribute is per device; callers run it on every launch (cheap).
  return cudaFuncSetAttribute(tc_gemm_kernel<KIND, TMA_STORE>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, Layout<KIND>::ALLOC);
}

template <int KIND>
cudaError_t launch_tc(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b0,
                      const CUtensorMap& b1, const CUtensorMap& cm, float* C, int64_t M, int64_t N,
                      int64_t K, int64_t ldc, bool c_tma, const DeviceCtl& ctl, cudaStream_t s) {
  using Cf = Cfg<KIND>;
  TcParams p;
  p.M = static_cast<int32_t>(M);
  p.N = static_cast<int32_t>(N);
  p.K = static_cast<int32_t>(K);
  p.tiles_m = static_cast<int32_t>((M + Cf::BM - 1) / Cf::BM);
  p.tiles_n = static_cast<int32_t>((N + Cf::BN - 1) / Cf::BN);
  p.num_tiles = p.tiles_m * p.tiles_n;
  p.num_kb = static_cast<int32_t>((K + Cf::BK - 1) / Cf::BK);
  p.full_units = p.num_tiles;
  p.num_units = p.num_tiles;
  p.kb_mid = p.num_kb;
  p.group_m = ctl.raster_group > 0 ? ctl.raster_group : GROUP_M;
  p.C = C;
  p.ldc = ldc;
  p.status = ctl.status;
  p.wait_limit_ns = ctl.wait_limit_ns;
  p.inject_stall = ctl.inject_stall;
  const int grid = p.num_tiles < ctl.sm_count ? p.num_tiles : ctl.sm_count;
  note_main_kernel(KIND == KIND_BF16 ? "tc_gemm_kernel<bf16>" : "tc_gemm_kernel<3xtf32>", grid,
                   p.num_tiles);
  cudaError_t e;
  if (c_tma) {
    if ((e = prepare_kernel<KIND, true>()) != cudaSuccess) return e;
    tc_gemm_kernel<KIND, true><<<grid, NUM_THREADS, Layout<KIND>::ALLOC, s>>>(a0, a1, b0, b1, cm, p);
  } else {
    if ((e = prepare_kernel<KIND, false>()) != cudaSuccess) return e;
    tc_gemm_kernel<KIND, false><<<grid, NUM_THREADS, Layout<KIND>::ALLOC, s>>>(a0, a1, b0, b1, cm, p);
  }
  return cudaGetLastError();
}

// Pair kernel launch: clusters of 2 CTAs, persistent over 256 x BN pair
// tiles, as many clusters as can be co-resident (at most one per pair tile).
template <int KIND, bool TMA_STORE>
cudaError_t launch_pair_t(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b0,
                          const CUtensorMap& b1, const CUtensorMap& cm, const TcParams& p,
                          const DeviceCtl& ctl, cudaStream_t s) {
  auto kern = tc_gemm_pair_kernel<KIND, TMA_STORE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       PairLayout<KIND>::ALLOC);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = PairLayout<KIND>::ALLOC;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(2 * (ctl.sm_count / 2));
  int max_clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg);
  if (e != cudaSuccess) return e;
  if (max_clusters < 1) return cudaErrorInvalidConfiguration;
  const int clusters = p.num_tiles < max_clusters ? p.num_tiles : max_clusters;
  // A last round that would leave more than half of the clusters idle is
  // split along K: its tiles become two half-K units each, reduce-added into
  // C (zeroed first).  Two addends onto zero give the same sum in either
  // order, so results stay bit-reproducible.
  TcParams q = p;
  const int rem = p.num_tiles % clusters;
  if (p.num_tiles > clusters && rem > 0 && 2 * rem <= clusters && p.num_kb >= 2) {
    q.full_units = p.num_tiles - rem;
    q.num_units = q.full_units + 2 * rem;
    q.kb_mid = p.num_kb / 2;
    zero_split_tiles_kernel<<<dim3(rem, 2 * PairCfg<KIND>::BM / 8), dim3(128, 8), 0, s>>>(
        q, PairCfg<KIND>::BN);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  cfg.gridDim = dim3(2 * clusters);
  note_main_kernel(KIND == KIND_BF16 ? "tc_gemm_pair_kernel<bf16>" : "tc_gemm_pair_kernel<3xtf32>",
                   2 * clusters, p.num_tiles);
  e = cudaLaunchKernelEx(&cfg, kern, a0, a1, b0, b1, cm, q);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// 1-CTA or CTA-pair kernel: the pair kernel when its 256 x BN tiles can keep
// every cluster of the GPU busy, the 1-CTA kernel for smaller problems (more,
// smaller tiles).  DeviceCtl::pair_mode forces one of them (tests).
template <int KIND>
cudaError_t launch_tc_any(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b0,
                          const CUtensorMap& b1, const CUtensorMap& cm, float* C, int64_t M,
                          int64_t N, int64_t K, int64_t ldc, bool c_tma, const DeviceCtl& ctl,
                          cudaStream_t s) {
  using Pc = PairCfg<KIND>;
  const int64_t pair_tiles = ((M + 2 * Pc::BM - 1) / (2 * Pc::BM)) * ((N + Pc::BN - 1) / Pc::BN);
  bool pair = pair_tiles >= ctl.sm_count / 2;
  if (ctl.pair_mode == 1) pair = false;
  if (ctl.pair_mode == 2) pair = true;
  if (!pair) return launch_tc<KIND>(a0, a1, b0, b1, cm, C, M, N, K, ldc, c_tma, ctl, s);
  TcParams p;
  p.M = static_cast<int32_t>(M);
  p.N = static_cast<int32_t>(N);
  p.K = static_cast<int32_t>(K);
  p.tiles_m = static_cast<int32_t>((M + 2 * Pc::BM - 1) / (2 * Pc::BM));
  p.tiles_n = static_cast<int32_t>((N + Pc::BN - 1) / Pc::BN);
  p.num_tiles = p.tiles_m * p.tiles_n;
  p.num_kb = static_cast<int32_t>((K + Pc::BK - 1) / Pc::BK);
  p.full_units = p.num_tiles;
  p.num_units = p.num_tiles;
  p.kb_mid = p.num_kb;
  p.group_m = ctl.raster_group > 0 ? ctl.raster_group : GROUP_M;
  p.C = C;
  p.ldc = ldc;
  p.status = ctl.status;
  p.wait_limit_ns = ctl.wait_limit_ns;
  p.inject_stall = ctl.inject_stall;
  return c_tma ? launch_pair_t<KIND, true>(a0, a1, b0, b1, cm, p, ctl, s)
               : launch_pair_t<KIND, false>(a0, a1, b0, b1, cm, p, ctl, s);
}

unsigned grid_rows(int64_t rows) { return static_cast<unsigned>(rows < 65535 ? rows : 65535); }

CUresult encode_c_map(CUtensorMap* cm, float* C, int64_t M, int64_t N, int64_t ldc, bool c_tma) {
  if (!c_tma) return CUDA_SUCCESS;
  return encode_tmap_2d(cm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, C, N, M, ldc * 4, 32, 32,
                        CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

size_t tc_bf16_smem_bytes() { return Layout<KIND_BF16>::ALLOC; }
size_t tc_3xtf32_smem_bytes() { return Layout<KIND_3XTF32>::ALLOC; }

cudaError_t launch_zero_fill(float* C, int64_t M, int64_t N, int64_t ldc, cudaStream_t s) {
  const unsigned gx = static_cast<unsigned>((N + 255) / 256 < 64 ? (N + 255) / 256 : 64);
  zero_fill_kernel<<<dim3(gx, grid_rows(M)), 256, 0, s>>>(C, M, N, ldc);
  return cudaGetLastError();
}

cudaError_t launch_pack_u16(const uint16_t* src, int64_t rows, int64_t cols, int64_t src_ld,
                            uint16_t* dst, int64_t dst_ld, cudaStream_t s) {
  const unsigned gx = static_cast<unsigned>((cols + 255) / 256 < 64 ? (cols + 255) / 256 : 64);
  pack_u16_kernel<<<dim3(gx, grid_rows(rows)), 256, 0, s>>>(src, rows, cols, src_ld, dst, dst_ld);
  return cudaGetLastError();
}

cudaError_t launch_split_tf32(const float* A, const float* B, int64_t M, int64_t N, int64_t K,
                              int64_t lda, int64_t ldb, int64_t Kp, float* a_big, float* a_small,
                              float* bt_big, float* bt_small, cudaStream_t s) {
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (Kp % 4 != 0 || !al16(a_big) || !al16(a_small) || !al16(bt_big) || !al16(bt_small))
    return cudaErrorInvalidValue;  // the workspace layout guarantees these
  const bool va = al16(A) && lda % 4 == 0 && K % 4 == 0;
  const bool vb = al16(B) && ldb % 4 == 0 && N % 4 == 0;
  // One wave of resident blocks (6 per SM fit), shared between the operands
  // in proportion to their sizes.
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t total = static_cast<int64_t>(sms) * 6;
  const int64_t b_tiles = ((N + SPLIT_TILE - 1) / SPLIT_TILE) * ((K + SPLIT_TILE - 1) / SPLIT_TILE);
  const double a_share = static_cast<double>(M) / static_cast<double>(M + N);
  int64_t a_blocks = static_cast<int64_t>(a_share * total);
  a_blocks = a_blocks < 1 ? 1 : (a_blocks > M ? M : a_blocks);
  int64_t b_blocks = total - a_blocks;
  b_blocks = b_blocks < 1 ? 1 : (b_blocks > b_tiles ? b_tiles : b_blocks);
  const unsigned grid = static_cast<unsigned>(a_blocks + b_blocks);
  const int ab = static_cast<int>(a_blocks);
  if (va && vb)
    split_vec_kernel<true, true><<<grid, SPLIT_THREADS, 0, s>>>(A, B, M, N, K, lda, ldb, Kp, ab,
                                                                a_big, a_small, bt_big, bt_small);
  else if (va)
    split_vec_kernel<true, false><<<grid, SPLIT_THREADS, 0, s>>>(A, B, M, N, K, lda, ldb, Kp, ab,
                                                                 a_big, a_small, bt_big, bt_small);
  else if (vb)
    split_vec_kernel<false, true><<<grid, SPLIT_THREADS, 0, s>>>(A, B, M, N, K, lda, ldb, Kp, ab,
                                                                 a_big, a_small, bt_big, bt_small);
  else
    split_vec_kernel<false, false><<<grid, SPLIT_THREADS, 0, s>>>(A, B, M, N, K, lda, ldb, Kp, ab,
                                                                  a_big, a_small, bt_big, bt_small);
  return cudaGetLastError();
}

cudaError_t launch_tc_bf16(const uint16_t* A, const uint16_t* B, float* C, int64_t M, int64_t N,
                           int64_t K, int64_t lda, int64_t ldb, int64_t ldc, bool c_tma,
                           const DeviceCtl& ctl, cudaStream_t s) {
  CUtensorMap a, b, cm;
  if (encode_tmap_2d(&a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A, K, M, lda * 2, 64, 128,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
      encode_tmap_2d(&b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, B, N, K, ldb * 2, 64, 64,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
      encode_c_map(&cm, C, M, N, ldc, c_tma) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  if (!c_tma) cm = a;  // unused by the kernel
  return launch_tc_any<KIND_BF16>(a, a, b, b, cm, C, M, N, K, ldc, c_tma, ctl, s);
}

cudaError_t launch_tc_3xtf32(const float* a_big, const float* a_small, const float* bt_big,
                             const float* bt_small, float* C, int64_t M, int64_t N, int64_t K,
                             int64_t Kp, int64_t ldc, bool c_tma, const DeviceCtl& ctl,
                             cudaStream_t s) {
  CUtensorMap a0, a1, b0, b1, cm;
  const auto f32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  if (encode_tmap_2d(&a0, f32, a_big, K, M, Kp * 4, 32, 128, sw) != CUDA_SUCCESS ||
      encode_tmap_2d(&a1, f32, a_small, K, M, Kp * 4, 32, 128, sw) != CUDA_SUCCESS ||
      encode_tmap_2d(&b0, f32, bt_big, K, N, Kp * 4, 32, 128, sw) != CUDA_SUCCESS ||
      encode_tmap_2d(&b1, f32, bt_small, K, N, Kp * 4, 32, 128, sw) != CUDA_SUCCESS ||
      encode_c_map(&cm, C, M, N, ldc, c_tma) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  if (!c_tma) cm = a0;
  return launch_tc_any<KIND_3XTF32>(a0, a1, b0, b1, cm, C, M, N, K, ldc, c_tma, ctl, s);
}

}  // namespace mhr
