// Single-CTA tensor-core GEMM kernel (one SM per output tile, persistent):
//   bf16:   128 x 256 x 64 tiles, 4 stages of 48 KB, kind::f16 M128 N256 K16;
//   3xTF32: 128 x 128 x 32 tiles, 3 stages of 64 KB, kind::tf32 M128 N128 K8.
// Used for problems whose 256-row CTA-pair tiles would not keep the GPU busy.
// The method and the warp roles are described in tc_common.cuh.
#include <array>
#include <cstdio>
#include <map>
#include <type_traits>

#include "tc_common.cuh"
#include "tc_split.cuh"

namespace mhr {
namespace tc {
namespace {

template <int KIND>
struct Cfg;

template <>
struct Cfg<KIND_BF16> {
  static constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
  static constexpr int A_BYTES = BM * BK * 2;              // 16 KB
  static constexpr int B_BOX_BYTES = 64 * BK * 2;          // 64 cols x 64 k = 8 KB
  static constexpr int B_BYTES = BK * BN * 2;              // 32 KB
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;    // 48 KB
  static constexpr int MAX_STAGES = STAGES;
  static constexpr int INSTR_K = 16;
  static constexpr uint32_t TMEM_COLS = 2 * BN;            // 512
};

// BN is the widest tile; with a pre-pass the kernel runs the width the host
// planned (TcParams::bn: 128, 96, 64 or 32), and its ring holds as many
// stages of 2 x 16 KB of A and 2 x bn x 128 bytes of B as fit in the same
// 192 KB, up to MAX_STAGES (ring_stages below): four at bn = 32 and 64.
template <>
struct Cfg<KIND_3XTF32> {
  static constexpr int BM = 128, BN = 128, BK = 32, STAGES = 3, MAX_STAGES = 4;
  static constexpr int A_BYTES = BM * BK * 4;              // 16 KB each (big, small)
  static constexpr int B_BYTES = BN * BK * 4;              // 16 KB each (big, small)
  static constexpr int STAGE_BYTES = 2 * A_BYTES + 2 * B_BYTES;  // 64 KB
  static constexpr int INSTR_K = 8;
  static constexpr uint32_t TMEM_COLS = 2 * BN;            // 256
};

// The 3xTF32 split done in the kernel, for problems too small to amortise a
// pre-pass launch: TMA stages A itself into the A_big box and two groups of
// converter warps (tc_split.cuh) write A_small, B_big^T and B_small^T.  One
// launch, no workspace.
template <>
struct Cfg<KIND_3XTF32_SPLIT_TMA_A> : Cfg<KIND_3XTF32> {};

// Ring stages and bytes per stage for tiles of bn columns (KIND_3XTF32
// outside the cluster split; every other case has the kind's fixed ring).
template <int KIND>
__host__ __device__ constexpr int ring_stage_bytes(int bn) {
  return KIND == KIND_3XTF32 ? 2 * Cfg<KIND>::A_BYTES + 2 * bn * Cfg<KIND>::BK * 4
                             : Cfg<KIND>::STAGE_BYTES;
}
template <int KIND>
__host__ __device__ constexpr int ring_stages(int bn) {
  return KIND == KIND_3XTF32
             ? (Cfg<KIND>::STAGES * Cfg<KIND>::STAGE_BYTES / ring_stage_bytes<KIND>(bn) <
                        Cfg<KIND>::MAX_STAGES
                    ? Cfg<KIND>::STAGES * Cfg<KIND>::STAGE_BYTES / ring_stage_bytes<KIND>(bn)
                    : Cfg<KIND>::MAX_STAGES)
             : Cfg<KIND>::STAGES;
}

template <int KIND>
__host__ __device__ constexpr int cta_threads() {
  return KIND == KIND_3XTF32_SPLIT_TMA_A ? NUM_THREADS + 2 * SPLIT_THREADS : NUM_THREADS;
}

// ------------------------------------------------------------------ cluster split
//
// Few tiles: the kernel can run as clusters of S CTAs (2 to 8; 16 for
// 3xTF32, beyond the portable cluster size, with the kernel's opt-in), one
// cluster per output tile.  Rank r takes the r-th run of ceil(num_kb / S)
// K-blocks (trailing runs may be short or empty), accumulates it in TMEM as
// usual, and its epilogue writes the partial 128 x BN fp32 tile into its own
// shared memory, over the ring, which no longer holds operands once the
// accumulator is complete.  After a cluster barrier rank r sums the r-th of
// S equal runs of the tile's float4s (row-major; whole rows [r * 128 / S,
// (r + 1) * 128 / S) when S divides 128) of all S partial tiles through
// distributed shared memory, in rank order, and stores them to C; a second
// barrier keeps every partial tile alive until the peers have read it.  One fixed order
// per element: bit-reproducible, with no zeroing of C and no atomics.
template <int KIND>
constexpr int MAX_CLUSTER = KIND == KIND_3XTF32 ? 16 : 8;

__device__ __forceinline__ uint32_t cluster_ctas() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ float4 ld_cluster_v4(uint32_t cluster_addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(cluster_addr)
               : "memory");
  return v;
}

// Work unit u: the persistent schedule's (tile, K range), or with CLUSTER
// tile u / S and the K-run u % S.
template <bool CLUSTER>
__device__ __forceinline__ Unit unit_1cta(int u, const TcParams& p) {
  if constexpr (CLUSTER) {
    const int S = static_cast<int>(cluster_ctas());
    const int per = (p.num_kb + S - 1) / S;
    Unit w;
    w.tile = u / S;
    w.kb0 = min(p.num_kb, (u % S) * per);
    w.kb1 = min(p.num_kb, w.kb0 + per);
    w.reduce = false;
    return w;
  } else {
    return unit_of(u, p);
  }
}

// Row pitch (floats) of the cluster split's partial tile: BN + 4.
template <int KIND>
constexpr int PART_LD = Cfg<KIND>::BN + 4;

template <int KIND>
struct Layout {
  using C = Cfg<KIND>;
  static constexpr int EPI_OFF = C::STAGES * C::STAGE_BYTES;
  static constexpr int BAR_OFF = EPI_OFF + EPI_BYTES;
  // full, empty, acc_full x2, acc_empty x2, drain, and the converters' stores
  static constexpr int NUM_BARS = 3 * C::MAX_STAGES + 5;
  static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;   // tmem slot, abort flag
  static constexpr int USED = MISC_OFF + 16;
  static constexpr int ALLOC = USED + 1024;                 // slack for 1024-byte alignment
  // the cluster split's partial tile lives over the ring
  static_assert(C::BM * PART_LD<KIND> * 4 <= C::STAGES * C::STAGE_BYTES, "partial tile");
};

// The converter warps' walk over this CTA's units (A rows m0.., 128 of them,
// B columns n0.., bn of them, and a K-block range).
template <bool CLUSTER>
struct SingleWalk {
  int bn;
  __device__ __forceinline__ int cols() const { return bn; }
  __device__ __forceinline__ bool box(const TcParams& p, int u, int& m0, int& nb0, int& kb0,
                                      int& kb1) const {
    if (u >= p.num_units) return false;
    const Unit w = unit_1cta<CLUSTER>(u, p);
    int tm, tn;
    tile_coords(w.tile, p, tm, tn);
    m0 = tm * SPLIT_BOX_ROWS;
    nb0 = tn * bn;
    kb0 = w.kb0;
    kb1 = w.kb1;
    return true;
  }
};

template <int KIND, bool TMA_STORE, bool CLUSTER>
__global__ void __launch_bounds__(cta_threads<KIND>(), 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                   const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
                   const __grid_constant__ CUtensorMap tmC,
                   const __grid_constant__ CUtensorMap tmC1, const TcParams p) {
  using Cf = Cfg<KIND>;
  using L = Layout<KIND>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + L::BAR_OFF;
  auto full_bar = [&](uint32_t s) { return bar0 + 8u * s; };
  auto empty_bar = [&](uint32_t s) { return bar0 + 8u * (Cf::MAX_STAGES + s); };
  auto accf_bar = [&](uint32_t b) { return bar0 + 8u * (2 * Cf::MAX_STAGES + b); };
  auto acce_bar = [&](uint32_t b) { return bar0 + 8u * (2 * Cf::MAX_STAGES + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * Cf::MAX_STAGES + 4);
  // KIND_3XTF32_SPLIT_TMA_A: the converter warps' stores of stage s are done
  auto cvt_bar = [&](uint32_t s) { return bar0 + 8u * (2 * Cf::MAX_STAGES + 5 + s); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::MISC_OFF + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // The tile's columns (with a pre-pass, the cluster split runs whole tiles
  // only), and the ring.
  const int bn = p.bn;
  const uint32_t stages = static_cast<uint32_t>(ring_stages<KIND>(bn));
  const uint32_t stage_bytes = static_cast<uint32_t>(ring_stage_bytes<KIND>(bn));

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cf::MAX_STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      if constexpr (KIND == KIND_3XTF32_SPLIT_TMA_A) mbar_init(cvt_bar(s), SPLIT_WARPS);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), EPI_WARPS);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA0);
    if constexpr (KIND != KIND_3XTF32_SPLIT_TMA_A) tma_prefetch_desc(&tmB0);
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
  // The set-up above may overlap the pre-pass kernel before this one; its
  // outputs (split or repacked operands, zeroed C tiles) are read from here on.
  grid_dependency_wait();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // One thread waits, arms and issues; the rest of the warp idles.
    if (lane == 0) {
      uint32_t it = 0;
      uint32_t inflight = 0;  // bit s: the latest fill of stage s had a TMA issued
      bool ok = true;
      for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x) {
        const Unit w = unit_1cta<CLUSTER>(u, p);
        int tm, tn;
        tile_coords(w.tile, p, tm, tn);
        const int m0 = tm * Cf::BM, n0 = tn * bn;
        for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
          const uint32_t s = it % stages, ph = (it / stages) & 1u;
          if (!mbar_wait_bounded(empty_bar(s), ph ^ 1u, limit, abort_flag)) {
            give_up_one(p, abort_flag, kErrTimeoutProducer);
            ok = false;
            break;
          }
          const uint32_t st = sbase + s * stage_bytes;
          const int k0 = kb * Cf::BK;
          // the split kind loads A alone (its converters fill the rest)
          mbar_arrive_expect_tx(full_bar(s), KIND == KIND_3XTF32_SPLIT_TMA_A ? Cf::A_BYTES
                                             : KIND == KIND_BF16 ? Cf::A_BYTES + bn * Cf::BK * 2
                                                                 : stage_bytes);
          const bool stall = p.inject_stall && blockIdx.x == 0 && it == 0;
          if (!stall) {
            if constexpr (KIND == KIND_3XTF32_SPLIT_TMA_A) {
              tma_load_2d(st, &tmA0, full_bar(s), k0, m0);
            } else if constexpr (KIND == KIND_BF16) {
              tma_load_2d(st, &tmA0, full_bar(s), k0, m0);
              for (int j = 0; j < bn / 64; ++j)
                tma_load_2d(st + Cf::A_BYTES + j * Cf::B_BOX_BYTES, &tmB0, full_bar(s), n0 + 64 * j,
                            k0);
            } else {
              tma_load_2d(st, &tmA0, full_bar(s), k0, m0);
              tma_load_2d(st + Cf::A_BYTES, &tmA1, full_bar(s), k0, m0);
              tma_load_2d(st + 2 * Cf::A_BYTES, &tmB0, full_bar(s), k0, n0);
              tma_load_2d(st + 2 * Cf::A_BYTES + bn * Cf::BK * 4, &tmB1, full_bar(s), k0, n0);
            }
            inflight |= 1u << s;
          } else {
            inflight &= ~(1u << s);
          }
        }
      }
      // Drain: every TMA this CTA issued must have landed before it exits.
      for (uint32_t s = 0; s < stages && s < it; ++s) {
        if (!(inflight & (1u << s))) continue;
        const uint32_t last = it - 1 - ((it - 1 - s) % stages);  // latest fill of stage s
        volatile int never = 0;
        if (!mbar_wait_bounded(full_bar(s), (last / stages) & 1u, limit, &never))
          atomicOr(p.status, kErrTimeoutDrain);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // One thread waits and issues every MMA.
    if (lane == 0) {
      uint32_t it = 0, tcount = 0;
      bool ok = true;
      const uint32_t idesc = KIND == KIND_BF16 ? make_idesc(1, false, true, Cf::BM, bn)
                                               : make_idesc(2, false, false, Cf::BM, bn);
      for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x, ++tcount) {
        const Unit w = unit_1cta<CLUSTER>(u, p);
        const uint32_t buf = tcount & 1u, aph = (tcount >> 1) & 1u;
        if (!mbar_wait_bounded(acce_bar(buf), aph ^ 1u, limit, abort_flag)) {
          give_up_one(p, abort_flag, kErrTimeoutMma);
          break;
        }
        tc_fence_after();  // the epilogue's TMEM reads precede these MMAs' writes
        const uint32_t d_tmem = tmem_base + buf * Cf::BN;
        for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
          const uint32_t s = it % stages, ph = (it / stages) & 1u;
          // the split kind: the converters' stores, which follow the A load
          if (!mbar_wait_bounded(KIND == KIND_3XTF32_SPLIT_TMA_A ? cvt_bar(s) : full_bar(s), ph,
                                 limit, abort_flag)) {
            give_up_one(p, abort_flag, kErrTimeoutMma);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = sbase + s * stage_bytes;
          if constexpr (KIND == KIND_BF16) {
            // A: 128 rows x 128 B, K-major, 8-row groups 1024 B apart.
            // B: bn / 64 (4 or 2) 64-column boxes (8 KB apart) of 64 k-rows x
            //    128 B, MN-major: LBO = next 64 columns, SBO = next 8 k-rows.
#pragma unroll
            for (int kk = 0; kk < Cf::BK / Cf::INSTR_K; ++kk) {
              const uint64_t ad = smem_desc_sw128(st + kk * 32, 16, 1024);
              const uint64_t bd = smem_desc_sw128(st + Cf::A_BYTES + kk * 2048, Cf::B_BOX_BYTES, 1024);
              mma_f16(d_tmem, ad, bd, idesc, (kb > w.kb0 || kk > 0) ? 1u : 0u);
            }
          } else {
            // All four operands K-major, 128 B rows (32 floats), 8-row groups
            // 1024 B apart; one instruction-K step (8 tf32) = 32 B.
            const uint32_t a_big = st, a_small = st + Cf::A_BYTES;
            const uint32_t b_big = st + 2 * Cf::A_BYTES, b_small = b_big + bn * Cf::BK * 4;
#pragma unroll
            for (int kk = 0; kk < Cf::BK / Cf::INSTR_K; ++kk) {
              const uint32_t off = kk * 32;
              const uint64_t abd = smem_desc_sw128(a_big + off, 16, 1024);
              const uint64_t asd = smem_desc_sw128(a_small + off, 16, 1024);
              const uint64_t bbd = smem_desc_sw128(b_big + off, 16, 1024);
              const uint64_t bsd = smem_desc_sw128(b_small + off, 16, 1024);
              mma_tf32(d_tmem, asd, bbd, idesc, (kb > w.kb0 || kk > 0) ? 1u : 0u);
              mma_tf32(d_tmem, abd, bsd, idesc, 1u);
              mma_tf32(d_tmem, abd, bbd, idesc, 1u);
            }
          }
          mma_commit(empty_bar(s));  // stage s may be refilled once these MMAs finish
        }
        if (!ok) break;
        mma_commit(accf_bar(buf));  // accumulator `buf` complete
      }
      // Drain: all MMAs issued by this thread complete before TMEM is freed.
      mma_commit(drain_bar);
      volatile int never = 0;
      if (!mbar_wait_bounded(drain_bar, 0, limit, &never)) atomicOr(p.status, kErrTimeoutDrain);
    }
    __syncwarp();
  } else if (KIND == KIND_3XTF32_SPLIT_TMA_A && warp >= NUM_THREADS / 32) {
    // ------------------------------------------------------------ converters
    // Group g takes this CTA's K-blocks g, g + 2, ... (tc_split.cuh).
    const int g = (threadIdx.x - NUM_THREADS) / SPLIT_THREADS;
    const int ct = (threadIdx.x - NUM_THREADS) % SPLIT_THREADS;
    const StoreOffsets so(ct);
    const SingleWalk<CLUSTER> walk{bn};
    // this thread's B columns 4 nb .. 4 nb + 3 lie inside the tile
    const bool has_b = 4 * (((ct & 31) >> 3) + 4 * (ct >> 5)) < bn;
    const int stride = static_cast<int>(gridDim.x);
    auto convert = [&](auto vec_b) {
      constexpr bool VB = decltype(vec_b)::value;
      // The group's first loads go out before the rest of the set-up: on a
      // small problem that set-up is most of the time to the first MMA.
      LoadCursor<SingleWalk<CLUSTER>> ld;
      ld.seek_work(p, walk, blockIdx.x, stride, ct);  // (a cluster rank's K run may be empty)
      for (int d = 0; d < g; ++d) ld.advance(p, walk, stride, ct);
      BRegs r;
      if (ld.valid) load_b<VB>(r, p, ld, ct);
      int total = 0;  // how many K-blocks this CTA stores
      for (int u = blockIdx.x; u < p.num_units; u += stride) {
        const Unit w = unit_1cta<CLUSTER>(u, p);
        total += w.kb1 - w.kb0;
      }
      // L2 prefetches run SPLIT_PREFETCH K-blocks ahead of the loads; with at
      // most one K-block per group there is nothing ahead to fetch.
      const bool prefetch = total > 2;
      PrefetchCursor<SingleWalk<CLUSTER>> pf;
      if (prefetch) {
        pf.seek_work(p, walk, blockIdx.x, stride);
        for (int d = 0; d < g + 2 + SPLIT_PREFETCH; ++d) {
          if (d >= g + 2 && ((d - g) & 1) == 0) split_prefetch_l2(p, ct, pf);
          pf.advance(p, walk, stride);
        }
      }
      for (int it = g; it < total; it += 2) {
        const uint32_t s = it % stages, ph = (it / stages) & 1u;
        if (!warp_wait(empty_bar(s), ph ^ 1u, limit, abort_flag) ||
            !warp_wait(full_bar(s), ph, limit, abort_flag)) {
          give_up(p, abort_flag, kErrTimeoutProducer, lane);
          break;
        }
        split_store_tma_a(r, sbase + s * stage_bytes, so, bn * Cf::BK * 4, has_b);
        fence_proxy_async_smem();  // the stores, visible to the MMA's reads
        __syncwarp();
        if (lane == 0) mbar_arrive(cvt_bar(s));
        ld.advance(p, walk, stride, ct);
        ld.advance(p, walk, stride, ct);
        if (it + 2 < total) load_b<VB>(r, p, ld, ct);
        if (prefetch) {
          split_prefetch_l2(p, ct, pf);
          pf.advance(p, walk, stride);
          pf.advance(p, walk, stride);
        }
      }
    };
    if (p.vec_b)
      convert(std::true_type{});
    else
      convert(std::false_type{});
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;           // TMEM lane quarter this warp may access
    const int ew = warp - 2;          // epilogue warp index 0..3
    uint32_t tcount = 0, chunk = 0;
    bool prev_group = false;  // the warp's previous chunk committed a bulk group
    for (int u = blockIdx.x; u < p.num_units; u += gridDim.x, ++tcount) {
      const Unit w = unit_1cta<CLUSTER>(u, p);
      const uint32_t buf = tcount & 1u, aph = (tcount >> 1) & 1u;
      if (!warp_wait(accf_bar(buf), aph, limit, abort_flag, 128)) {
        give_up(p, abort_flag, kErrTimeoutEpilogue, lane);
        break;
      }
      tc_fence_after();
      int tm, tn;
      tile_coords(w.tile, p, tm, tn);
      const int m0 = tm * Cf::BM, n0 = tn * bn;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * Cf::BN;
      if constexpr (CLUSTER) {
        // this thread's row of the partial tile, into shared memory (a rank
        // with no K-blocks contributes zeros)
        const uint32_t prow = sbase + static_cast<uint32_t>((q * 32 + lane) * PART_LD<KIND> * 4);
        const bool has_k = w.kb1 > w.kb0;
#pragma unroll 1
        for (int c = 0; c < bn / 32; ++c) {
          uint32_t r[32];
          if (has_k) {
            tmem_ld_32cols(taddr + c * 32, r);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = 0u;
          }
#pragma unroll
          for (int j = 0; j < 8; ++j)
            st_shared_v4(prow + static_cast<uint32_t>((c * 32 + 4 * j) * 4),
                         make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                     __uint_as_float(r[4 * j + 2]),
                                     __uint_as_float(r[4 * j + 3])));
        }
      } else {
        const int col_end = n0 + bn < p.N ? n0 + bn : p.N;
#pragma unroll 1
        for (int c = 0; c < bn / 32; ++c) {
          uint32_t r[32];
          tmem_ld_32cols(taddr + c * 32, r);
          // (the converter kind, held to 80 registers, keeps its odd rows in
          // registers)
          const OddRows odd =
              KIND == KIND_3XTF32_SPLIT_TMA_A
                  ? OddRows{}
                  : plan_odd_rows(p, n0, n0 + c * 32, col_end, taddr + c * 32 + 32);
          tmem_ld_wait();
          prev_group = stage_and_store_chunk<TMA_STORE>(r, sbase + L::EPI_OFF, ew, chunk, lane,
                                                        &tmC, &tmC1, p, m0 + q * 32,
                                                        n0 + c * 32, col_end, w.reduce, odd,
                                                        prev_group);
          ++chunk;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce_bar(buf));  // TMEM buffer `buf` may be overwritten
    }
    if (TMA_STORE || p.c_even) {  // every store of this warp has completed
      if (lane == 0) bulk_wait_group<0>();
      __syncwarp();
    }
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (CLUSTER) {
    cluster_sync_all();  // every rank's partial tile is in its shared memory
    const int S = static_cast<int>(cluster_ctas());
    const int rank = static_cast<int>(cluster_ctarank());
    // rank r sums the r-th of S equal runs of the tile's float4s, row-major
    const int quads = bn / 4;
    const int end = (rank + 1) * (Cf::BM * quads) / S;
    int tm, tn;
    tile_coords(static_cast<int>(blockIdx.x) / S, p, tm, tn);
    const int64_t m0 = static_cast<int64_t>(tm) * Cf::BM;
    const int n0 = tn * bn;
    const bool vec = (reinterpret_cast<uintptr_t>(p.C) & 15u) == 0 && (p.ldc & 3) == 0;
    for (int idx = rank * (Cf::BM * quads) / S + static_cast<int>(threadIdx.x); idx < end;
         idx += cta_threads<KIND>()) {
      const int r = idx / quads;
      const int c = (idx % quads) * 4;
      const uint32_t off = sbase + static_cast<uint32_t>((r * PART_LD<KIND> + c) * 4);
      // all loads first (their latencies overlap), then the sum in rank order
      float4 t[MAX_CLUSTER<KIND>];
#pragma unroll
      for (int k = 0; k < MAX_CLUSTER<KIND>; ++k)
        if (k < S) t[k] = ld_cluster_v4(mapa_shared(off, static_cast<uint32_t>(k)));
      float4 v = t[0];
#pragma unroll
      for (int k = 1; k < MAX_CLUSTER<KIND>; ++k)
        if (k < S) {
          v.x += t[k].x;
          v.y += t[k].y;
          v.z += t[k].z;
          v.w += t[k].w;
        }
      const int64_t row = m0 + r;
      const int col = n0 + c;
      if (row >= p.M || col >= p.N) continue;
      float* dst = p.C + row * p.ldc + col;
      if (vec && col + 4 <= p.N) {
        *reinterpret_cast<float4*>(dst) = v;
      } else {
        dst[0] = v.x;
        if (col + 1 < p.N) dst[1] = v.y;
        if (col + 2 < p.N) dst[2] = v.z;
        if (col + 3 < p.N) dst[3] = v.w;
      }
    }
    cluster_sync_all();  // no rank leaves while a peer still reads its partial tile
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cf::TMEM_COLS);
  }
}

template <int KIND, bool TMA_STORE, bool CLUSTER>
cudaError_t prepare_kernel() {
  // cudaFuncSetAttribute is per device; callers run it on every launch (cheap).
  cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<KIND, TMA_STORE, CLUSTER>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Layout<KIND>::ALLOC);
  if (e == cudaSuccess && CLUSTER && MAX_CLUSTER<KIND> > 8)
    e = cudaFuncSetAttribute(tc_gemm_kernel<KIND, TMA_STORE, CLUSTER>,
                             cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

// Cluster size for the cluster split of a problem with few tiles: the
// largest S in 8, 7, ..., 4 (3xTF32: 16 first) with one CTA per SM for all
// tiles x S CTAs, at least 16 K-blocks per rank (8 at S = 16), and every
// cluster co-resident; 1 = no cluster split.  Sizes between the powers of
// two fit where the next power does not: 16 tiles of 128 x 128 take
// clusters of 7 (112 CTAs) where sixteen clusters of 8 are more than fit.  Each rank pulls about one tile of
// partial sums from its peers whatever S is, so a larger S shortens the K
// runs at the same reduction cost: 3xTF32, 256 x 256 x 8192 37.5 -> 29.3 us
// and 512 x 128 x 4136 27.3 -> 23.2 us with S = 16; bf16, at half the MMA
// time per K-block, gained nothing from it (256 x 256 x 8192 17.1 / 17.0).
// Measured on GB300 (whole calls), the split's fixed costs -- the cluster
// launch, the partial tiles through shared memory, two cluster barriers --
// pay off only on long K runs: 512 x 512 x 8192 3xTF32 95.9 -> 64.1 us (S =
// 4, against two K halves), bf16 33.4 -> 21.1 us (S = 8); 1024 x 1024 x 4096
// bf16 23.2 -> 21.2 us (S = 4); but 256^3 3xTF32 14.0 -> 15.0 us (S = 8, one
// K-block per rank), bf16 10.9 -> 12.9 us, and S = 2 in place of the K
// halves 63.1 -> 66.2 us (1024 x 1024 x 4096 3xTF32).
template <int KIND>
int cluster_split_size(const TcParams& p, cudaLaunchConfig_t cfg, const DeviceCtl& ctl) {
  if (2 * p.num_tiles > ctl.sm_count || p.num_kb < 16 * 4) return 1;
  if (prepare_kernel<KIND, false, true>() != cudaSuccess) {
    cudaGetLastError();
    return 1;
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // Clusters of S CTAs that fit on the GPU at once: the occupancy query
  // depends on the kernel and S only, so it is made once per device (calls
  // are serialised by the library's lock).
  static std::map<int, std::array<int, 17>> fit_cache;
  int dev = 0;
  cudaGetDevice(&dev);
  auto fit = fit_cache.emplace(dev, std::array<int, 17>{}).first;
  for (int S = MAX_CLUSTER<KIND>; S >= 4; S = S > 8 ? 8 : S - 1) {
    if (p.num_tiles * S > ctl.sm_count || p.num_kb < (S > 8 ? 8 : 16) * S) continue;
    int& clusters = fit->second[S];
    if (clusters == 0) {
      attr[0].val.clusterDim.x = static_cast<unsigned>(S);
      cfg.gridDim = dim3(static_cast<unsigned>(8 * S));
      if (cudaOccupancyMaxActiveClusters(&clusters, tc_gemm_kernel<KIND, false, true>, &cfg) !=
          cudaSuccess) {
        cudaGetLastError();
        clusters = -1;
      }
    }
    if (clusters >= p.num_tiles) return S;
  }
  return 1;
}

// Whether launch_t splits every tile into two K halves (see there): all the
// halves fit on the SMs at once, and without a pre-pass to hide the zeroing
// of C behind, K has at least 32 steps.
inline bool k_halves_chosen(const TcParams& p, bool after_prepass, const DeviceCtl& ctl) {
  return 2 * p.num_tiles <= ctl.sm_count && p.num_kb >= (after_prepass ? 4 : 32);
}

// How many CTAs the single-CTA kernel puts to work on tiles of bn columns:
// clusters for the cluster split, two K halves per tile when they all fit,
// else one CTA per tile up to the SM count (as launch_t below decides).
template <int KIND>
int64_t working_ctas(int64_t M, int64_t N, int64_t K, float* C, int64_t ldc, int bn,
                     bool after_prepass, cudaLaunchConfig_t cfg, const DeviceCtl& ctl) {
  const TcParams q = make_params(M, N, K, Cfg<KIND>::BM, bn, Cfg<KIND>::BK, C, ldc, ctl);
  const int S = cluster_split_size<KIND>(q, cfg, ctl);
  if (S > 1) return q.num_tiles * S;
  if (k_halves_chosen(q, after_prepass, ctl)) return 2 * q.num_tiles;
  return q.num_tiles < ctl.sm_count ? q.num_tiles : ctl.sm_count;
}

// bf16 tile columns, 256 or 128: 128 when its tiles, split as launch_t splits
// them, put more CTAs to work in a single round.  An MMA of 128 columns reads
// 32 KB of shared memory per 64-deep K-block against 48 KB for 256 columns
// at half the work, so it only pays where it brings SMs that would idle.
template <int KIND>
int bf16_tile_n(int64_t M, int64_t N, int64_t K, float* C, int64_t ldc, bool after_prepass,
                cudaLaunchConfig_t cfg, const DeviceCtl& ctl) {
  const int64_t narrow = working_ctas<KIND>(M, N, K, C, ldc, 128, after_prepass, cfg, ctl);
  const int64_t wide = working_ctas<KIND>(M, N, K, C, ldc, Cfg<KIND>::BN, after_prepass, cfg, ctl);
  const int64_t tiles128 = ((M + Cfg<KIND>::BM - 1) / Cfg<KIND>::BM) * ((N + 127) / 128);
  return narrow > wide && tiles128 <= ctl.sm_count ? 128 : Cfg<KIND>::BN;
}

template <int KIND>
cudaError_t launch_t(const TcMaps& mp, float* C, int64_t M, int64_t N, int64_t K, int64_t ldc,
                     bool c_tma, bool after_prepass, int bn, const DeviceCtl& ctl,
                     cudaStream_t s) {
  using Cf = Cfg<KIND>;
  cudaError_t e;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = Layout<KIND>::ALLOC;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // bf16: 256 or 128 columns, forced or planned; 3xTF32: the width the
  // caller planned (128, 96, 64 or 32)
  if (KIND == KIND_BF16 && bn != 128 && bn != Cf::BN)
    bn = bf16_tile_n<KIND>(M, N, K, C, ldc, after_prepass, cfg, ctl);
  if ((KIND != KIND_3XTF32 && KIND != KIND_BF16) || bn <= 0 || bn > Cf::BN) bn = Cf::BN;
  TcParams p = make_params(M, N, K, Cf::BM, bn, Cf::BK, C, ldc, ctl);
  p.c_even = !c_tma && mp.c_even;
  p.c_odd_shift = p.c_even ? mp.c_odd_shift : -1;
  // Few tiles with long K runs: a cluster of S CTAs per tile, each on one
  // run of K-blocks, summing through distributed shared memory (see above).
  const int S = cluster_split_size<KIND>(p, cfg, ctl);
  if (S > 1) {
    p.num_units = p.num_tiles * S;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(S);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
    cfg.gridDim = dim3(static_cast<unsigned>(p.num_units));
    char cname[48];
    if (bn == Cf::BN)
      snprintf(cname, sizeof(cname), "tc_gemm_kernel<%s,cluster-K>",
               KIND == KIND_BF16 ? "bf16" : "3xtf32");
    else
      snprintf(cname, sizeof(cname), "tc_gemm_kernel<%s,n%d,cluster-K>",
               KIND == KIND_BF16 ? "bf16" : "3xtf32", bn);
    note_main_kernel(cname, p.num_units, p.num_tiles);
    e = cudaLaunchKernelEx(&cfg, tc_gemm_kernel<KIND, false, true>, mp.a0, mp.a1, mp.b0, mp.b1,
                           mp.c, mp.c1, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  // Otherwise, few tiles (all of them, halved, fit on the SMs at once):
  // split every tile into two half-K units that reduce-add into C, zeroed
  // first, so that twice as many SMs share the work.  Two addends onto zero
  // give the same sum in either order: results stay bit-reproducible.  The
  // zeroing runs alongside a pre-pass when there is one; without, it is a
  // launch of its own, which only pays for itself with a long K loop.  GB300,
  // whole calls: 3xTF32 1024 x 1024 x 4096 95.9 -> 63.1 us, 1024^3 31.4 ->
  // 24.2, 256^3 15.0 -> 14.0; bf16 1024^3 (16 K-steps) 15.0 either way, 256^3
  // (4) 10.9 -> 13.0.
  if (k_halves_chosen(p, after_prepass, ctl)) {
    p.full_units = 0;
    p.num_units = 2 * p.num_tiles;
    p.kb_mid = p.num_kb / 2;
    if ((e = launch_zero_split_tiles(p, Cf::BM, bn, after_prepass, s)) != cudaSuccess) return e;
  }
  const int grid = p.num_units < ctl.sm_count ? p.num_units : ctl.sm_count;
  char name[48];
  if (bn != Cf::BN)
    snprintf(name, sizeof(name), "tc_gemm_kernel<%s,n%d>",
             KIND == KIND_BF16 ? "bf16" : "3xtf32", bn);
  else
    snprintf(name, sizeof(name), "%s",
             KIND == KIND_BF16 ? "tc_gemm_kernel<bf16>" : "tc_gemm_kernel<3xtf32>");
  note_main_kernel(name, grid, p.num_tiles);
  cfg.gridDim = dim3(grid);
  if (c_tma) {
    if ((e = prepare_kernel<KIND, true, false>()) != cudaSuccess) return e;
    e = cudaLaunchKernelEx(&cfg, tc_gemm_kernel<KIND, true, false>, mp.a0, mp.a1, mp.b0, mp.b1,
                           mp.c, mp.c1, p);
  } else {
    if ((e = prepare_kernel<KIND, false, false>()) != cudaSuccess) return e;
    e = cudaLaunchKernelEx(&cfg, tc_gemm_kernel<KIND, false, false>, mp.a0, mp.a1, mp.b0, mp.b1,
                           mp.c, mp.c1, p);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

// The largest cluster size the one-launch split tries (8, 4 or 2; 1 = none).
#ifndef MHR_SMALL_MAX_CLUSTER
#define MHR_SMALL_MAX_CLUSTER 8
#endif

cudaError_t launch_single_cta_split(const TcMaps& maps, const float* A, const float* B, float* C,
                                    int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                                    int64_t ldc, bool c_tma, const DeviceCtl& ctl,
                                    cudaStream_t s) {
  constexpr int KIND = KIND_3XTF32_SPLIT_TMA_A;
  using Cf = Cfg<KIND>;
  cudaError_t e;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(cta_threads<KIND>());
  cfg.dynamicSmemBytes = Layout<KIND>::ALLOC;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if ((e = prepare_kernel<KIND, false, true>()) != cudaSuccess) return e;
  // Clusters of c CTAs that fit on the GPU at once (c = 2, 4, 8): the
  // occupancy query depends on the kernel and c only, so it is made once per
  // device (calls are serialised by the library's lock).
  static std::map<int, std::array<int, 9>> fit_cache;
  int dev = 0;
  cudaGetDevice(&dev);
  auto fit = fit_cache.emplace(dev, std::array<int, 9>{}).first;
  auto clusters_fit = [&](int c) {
    int& n = fit->second[c];
    if (n == 0) {
      attr[1].val.clusterDim.x = static_cast<unsigned>(c);
      cfg.numAttrs = 2;
      cfg.gridDim = dim3(static_cast<unsigned>(8 * c));
      if (cudaOccupancyMaxActiveClusters(&n, tc_gemm_kernel<KIND, false, true>, &cfg) !=
          cudaSuccess) {
        cudaGetLastError();
        n = -1;
      }
      cfg.numAttrs = 1;
    }
    return n;
  };
  // With few tiles, a cluster of S CTAs per tile, each on one run of
  // K-blocks, summing through distributed shared memory: the largest S in
  // {8, 4, 2} that gives every rank a K-block and every CTA its own SM.
  const int num_kb = static_cast<int>((K + Cf::BK - 1) / Cf::BK);
  auto cluster_size = [&](int64_t tiles) {
    for (int c = MHR_SMALL_MAX_CLUSTER; c >= 2; c /= 2)
      if (tiles * c <= ctl.sm_count && num_kb >= c && clusters_fit(c) >= tiles) return c;
    return 1;
  };
  // Tile width: the one that puts the most CTAs to work (128, 64 or 32
  // columns; a tie goes to the wider tile), unless the test hook forces one.
  // GB300, whole calls: 256^3 15.1 / 13.1 / 13.0 us at 128 / 64 / 32 columns,
  // 512^3 18.7 / 15.1 / 17.1, 300 x 520 x 1000 19.1 / 19.2 / 23.1,
  // 256 x 512 x 1000 19.1 / 19.1 / 17.1, 256 x 256 x 2048 25.2 / 19.1 / 23.0.
  int bn = ctl.single_tile_n <= Cf::BN ? ctl.single_tile_n : 0;
  if (bn <= 0) {
    int64_t best_grid = 0;
    for (int w = Cf::BN; w >= 32; w /= 2) {
      const int64_t tiles = ((M + Cf::BM - 1) / Cf::BM) * ((N + w - 1) / w);
      const int c = cluster_size(tiles);
      const int64_t grid = c > 1 ? tiles * c : (tiles < ctl.sm_count ? tiles : ctl.sm_count);
      if (grid > best_grid) {
        best_grid = grid;
        bn = w;
      }
    }
  }
  TcParams p = make_params(M, N, K, Cf::BM, bn, Cf::BK, C, ldc, ctl);
  p.A = A;
  p.B = B;
  p.lda = lda;
  p.ldb = ldb;
  p.vec_a = 1;  // the TMA map of A requires what the 16-byte loads do
  p.vec_b = (reinterpret_cast<uintptr_t>(B) % 16 == 0) && (ldb % 4 == 0);
  p.c_even = !c_tma && maps.c_even;
  p.c_odd_shift = -1;  // see the epilogue
  const int S = cluster_size(p.num_tiles);
  if (S > 1) {
    attr[1].val.clusterDim.x = static_cast<unsigned>(S);
    p.num_units = p.num_tiles * S;
    cfg.numAttrs = 2;
    cfg.gridDim = dim3(static_cast<unsigned>(p.num_units));
    char name[64];
    if (bn == Cf::BN)
      snprintf(name, sizeof(name), "tc_gemm_kernel<3xtf32,split,tma-a,cluster-K>");
    else
      snprintf(name, sizeof(name), "tc_gemm_kernel<3xtf32,split,tma-a,n%d,cluster-K>", bn);
    note_main_kernel(name, p.num_units, p.num_tiles);
    e = cudaLaunchKernelEx(&cfg, tc_gemm_kernel<KIND, false, true>, maps.a0, maps.a1, maps.b0,
                           maps.b1, maps.c, maps.c1, p);
  } else {
    cfg.numAttrs = 1;
    const int grid = p.num_units < ctl.sm_count ? p.num_units : ctl.sm_count;
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    char name[64];
    if (bn == Cf::BN)
      snprintf(name, sizeof(name), "tc_gemm_kernel<3xtf32,split,tma-a>");
    else
      snprintf(name, sizeof(name), "tc_gemm_kernel<3xtf32,split,tma-a,n%d>", bn);
    note_main_kernel(name, grid, p.num_tiles);
    if (c_tma) {
      if ((e = prepare_kernel<KIND, true, false>()) != cudaSuccess) return e;
      e = cudaLaunchKernelEx(&cfg, tc_gemm_kernel<KIND, true, false>, maps.a0, maps.a1, maps.b0,
                             maps.b1, maps.c, maps.c1, p);
    } else {
      if ((e = prepare_kernel<KIND, false, false>()) != cudaSuccess) return e;
      e = cudaLaunchKernelEx(&cfg, tc_gemm_kernel<KIND, false, false>, maps.a0, maps.a1, maps.b0,
                             maps.b1, maps.c, maps.c1, p);
    }
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_single_cta(int kind, const TcMaps& maps, float* C, int64_t M, int64_t N,
                              int64_t K, int64_t ldc, bool c_tma, bool after_prepass, int bn,
                              const DeviceCtl& ctl, cudaStream_t s) {
  return kind == KIND_BF16
             ? launch_t<KIND_BF16>(maps, C, M, N, K, ldc, c_tma, after_prepass,
                                   ctl.single_tile_n, ctl, s)
             : launch_t<KIND_3XTF32>(maps, C, M, N, K, ldc, c_tma, after_prepass, bn, ctl, s);
}

}  // namespace tc
}  // namespace mhr
