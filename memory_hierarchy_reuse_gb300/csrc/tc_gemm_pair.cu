// CTA-pair tensor-core GEMM kernel (tcgen05.mma.cta_group::2): two CTAs on
// two SMs share one 256 x 256 output tile; persistent over tiles, with the
// sparse last round split along K.  Used for large problems.  The method and
// the warp roles are described in tc_common.cuh.
#include <cstdio>
#include <type_traits>

#include "tc_common.cuh"
#include "tc_split.cuh"
#include "tf32_split.cuh"

namespace mhr {
namespace tc {
namespace {

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

// bf16 K step: 128 (3 stages of 64 KB) by default, 64 (6 stages of 32 KB)
// when built with -DMHR_PAIR_BF16_BK=64.  Both keep 192 KB of operands in
// flight; they differ in how many MMAs share one commit and one ring-barrier
// round trip (8 against 4).  On GB300 each round trip costs the tensor pipe
// some 40 cycles against 128 per 256x256x16 instruction: with loads taken out,
// the pipe is busy 98% of the time at 128 against 91.5% at 64, and with loads
// the 8192^3 kernel runs 2-3% faster at 128.
#ifndef MHR_PAIR_BF16_BK
#define MHR_PAIR_BF16_BK 128
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

// BN is the widest tile; the kernel runs the tile width the host planned
// (TcParams::bn, a multiple of 16), loading bn / 2 rows of each B part per CTA
// into the start of its 16 KB box.
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

// The in-kernel split runs the 3xTF32 main loop unchanged; only the producer
// differs (converter warps instead of TMA).
template <>
struct PairCfg<KIND_3XTF32_SPLIT> : PairCfg<KIND_3XTF32> {};
template <>
struct PairCfg<KIND_3XTF32_SPLIT_TMA_A> : PairCfg<KIND_3XTF32> {};

// Kinds whose ring stages are filled (wholly or partly) by converter warps.
template <int KIND>
__host__ __device__ constexpr bool has_converters() {
  return KIND == KIND_3XTF32_SPLIT || KIND == KIND_3XTF32_SPLIT_TMA_A;
}

// Groups of SPLIT_WARPS converter warps that take K-blocks in turn (see
// tc_split.cuh and the split kinds below).
template <int KIND>
constexpr int converter_groups() {
  return KIND == KIND_3XTF32_SPLIT_TMA_A ? 2 : has_converters<KIND>() ? 1 : 0;
}

template <int KIND>
constexpr int pair_threads() {
  return NUM_THREADS + converter_groups<KIND>() * SPLIT_THREADS;
}

// This CTA's boxes of work unit u, and the unit's K-block range.
__device__ __forceinline__ bool unit_boxes(const TcParams& p, int u, uint32_t rank, int& m0,
                                           int& nb0, int& kb0, int& kb1) {
  if (u >= p.num_units) return false;
  const Unit w = unit_of(u, p);
  int tm, tn;
  tile_coords(w.tile, p, tm, tn);
  m0 = tm * PAIR_TILE_M + static_cast<int>(rank) * (PAIR_TILE_M / 2);
  nb0 = tn * PAIR_TILE_N + static_cast<int>(rank) * (PAIR_TILE_N / 2);
  kb0 = w.kb0;
  kb1 = w.kb1;
  return true;
}

// The converter warps' walk over this CTA's boxes: units cluster,
// cluster + clusters, ...
struct PairWalk {
  uint32_t rank;
  __device__ __forceinline__ int cols() const { return PAIR_TILE_N / 2; }
  __device__ __forceinline__ bool box(const TcParams& p, int u, int& m0, int& nb0, int& kb0,
                                      int& kb1) const {
    return unit_boxes(p, u, rank, m0, nb0, kb0, kb1);
  }
};

template <int KIND>
struct PairLayout {
  using C = PairCfg<KIND>;
  static constexpr int EPI_OFF = C::STAGES * C::STAGE_BYTES;
  static constexpr int BAR_OFF = EPI_OFF + EPI_BYTES;
  static constexpr int NUM_BARS = 3 * C::STAGES + 6;
  static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
  static constexpr int USED = MISC_OFF + 16;
  static constexpr int ALLOC = USED + 1024;
};

template <int KIND, bool TMA_STORE>
__global__ void __launch_bounds__(pair_threads<KIND>(), 1)
    tc_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA0,
                        const __grid_constant__ CUtensorMap tmA1,
                        const __grid_constant__ CUtensorMap tmB0,
                        const __grid_constant__ CUtensorMap tmB1,
                        const __grid_constant__ CUtensorMap tmC,
                        const __grid_constant__ CUtensorMap tmC1, const TcParams p) {
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
  // rank 0 only: rank 1's producer arrives here once it has issued its last load
  const uint32_t peer_done_bar = bar0 + 8u * (2 * Cf::STAGES + 5);
  // KIND_3XTF32_SPLIT_TMA_A, each CTA: its own TMA load of A's box into stage s
  auto a_full_bar = [&](uint32_t s) { return bar0 + 8u * (2 * Cf::STAGES + 6 + s); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::MISC_OFF + 4);
  // rank 0 only: how many ring stages rank 1's producer loaded
  volatile uint32_t* peer_loaded = reinterpret_cast<volatile uint32_t*>(smem + L::MISC_OFF + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cluster = blockIdx.x >> 1, num_clusters = gridDim.x >> 1;
  const uint32_t peer_abort = mapa_shared(smem_u32(const_cast<int*>(abort_flag)), rank ^ 1u);
  // The pair tile's columns, and the bytes one CTA loads into a ring stage.
  const int bn = KIND == KIND_3XTF32 ? p.bn : Cf::BN;
  const uint32_t stage_tx =
      KIND == KIND_3XTF32 ? static_cast<uint32_t>(2 * Cf::A_BYTES + 2 * (bn / 2) * Cf::BK * 4)
                          : static_cast<uint32_t>(Cf::STAGE_BYTES);

  if (threadIdx.x == 0) {
    // full[s]: one arrive.expect_tx by the TMA producer, or one arrive per
    // converter warp of both CTAs (split kind)
    constexpr uint32_t full_count = has_converters<KIND>() ? 2 * SPLIT_WARPS : 1;
    for (int s = 0; s < Cf::STAGES; ++s) {
      mbar_init(full_bar(s), full_count);
      mbar_init(empty_bar(s), 1);
      if constexpr (KIND == KIND_3XTF32_SPLIT_TMA_A) mbar_init(a_full_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), 2 * EPI_WARPS);
    }
    mbar_init(drain_bar, 1);
    mbar_init(peer_done_bar, 1);
    *abort_flag = 0;
    *peer_loaded = 0;
    fence_mbar_init();
    if constexpr (KIND != KIND_3XTF32_SPLIT) tma_prefetch_desc(&tmA0);
    if constexpr (!has_converters<KIND>()) tma_prefetch_desc(&tmB0);
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
  // The set-up above may overlap the pre-pass kernel before this one; its
  // outputs (split or repacked operands, zeroed C tiles) are read from here on.
  grid_dependency_wait();

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
    // One thread waits, arms and issues; the rest of the warp idles.  (The
    // split kind has converter warps instead; its warp 0 only idles.)
    if (KIND == KIND_3XTF32_SPLIT_TMA_A && lane == 0) {
      // This CTA's A boxes, into the A_big box of each stage, on its own
      // barriers (its converter warps wait for them).
      uint32_t it = 0;
      bool stalled_first = false;
      for (int u = cluster; u < p.num_units; u += num_clusters) {
        const Unit w = unit_of(u, p);
        int tm, tn;
        tile_coords(w.tile, p, tm, tn);
        const int m0 = tm * 2 * Cf::BM + static_cast<int>(rank) * Cf::BM;
        bool ok = true;
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          const uint32_t s = it % Cf::STAGES, ph = (it / Cf::STAGES) & 1u;
          if (!mbar_wait_bounded(empty_bar(s), ph ^ 1u, limit, abort_flag)) {
            give_up_one(kErrTimeoutProducer);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(a_full_bar(s), Cf::A_BYTES);
          // test hook: block 0 arms its first stage without loading it
          if (!(p.inject_stall && blockIdx.x == 0 && it == 0))
            tma_load_2d(sbase + s * Cf::STAGE_BYTES, &tmA0, a_full_bar(s), kb * Cf::BK, m0);
          else
            stalled_first = true;
          ++it;
        }
        if (!ok) break;
      }
      // Drain: wait for this CTA's loads of the last STAGES iterations (earlier
      // phases were waited for by the converters before the stage was reused).
      // A stage armed without its load is counted as done.
      volatile int never = 0;
      for (uint32_t i = it > static_cast<uint32_t>(Cf::STAGES) ? it - Cf::STAGES : 0; i < it;
           ++i) {
        const uint32_t s = i % Cf::STAGES, ph = (i / Cf::STAGES) & 1u;
        if (stalled_first && i == 0) mbar_complete_tx(a_full_bar(s), Cf::A_BYTES);
        if (!mbar_wait_bounded(a_full_bar(s), ph, limit, &never))
          atomicOr(p.status, kErrTimeoutDrain);
      }
    } else if (!has_converters<KIND>() && lane == 0) {
      // `it` counts the ring stages this producer armed (rank 0) and loaded;
      // with the injected stall, block 0's first stage is armed but not loaded.
      uint32_t it = 0;
      bool stalled_first = false;
      for (int u = cluster; u < p.num_units; u += num_clusters) {
        const Unit w = unit_of(u, p);
        int tm, tn;
        tile_coords(w.tile, p, tm, tn);
        const int m0 = tm * 2 * Cf::BM + static_cast<int>(rank) * Cf::BM;
        const int nb0 = tn * bn + static_cast<int>(rank) * (bn / 2);
        bool ok = true;
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          const uint32_t s = it % Cf::STAGES, ph = (it / Cf::STAGES) & 1u;
          if (!mbar_wait_bounded(empty_bar(s), ph ^ 1u, limit, abort_flag)) {
            give_up_one(kErrTimeoutProducer);
            ok = false;
            break;
          }
          const uint32_t st = sbase + s * Cf::STAGE_BYTES;
          const uint32_t fb = mapa_shared(full_bar(s), 0);  // rank 0's full[s]
          const int k0 = kb * Cf::BK;
          if (leader) mbar_arrive_expect_tx(full_bar(s), 2 * stage_tx);
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
          } else {
            stalled_first = true;
          }
          ++it;
        }
        if (!ok) break;
      }
      // Drain.  Both CTAs' loads complete on rank 0's full barriers, which
      // rank 1 cannot poll, so rank 0 waits for them all: rank 1 tells it how
      // many stages it loaded; rank 0 then completes the phase of each of the
      // last STAGES iterations -- arming it for rank 1's bytes if rank 0 never
      // got that far, or counting as done the bytes that either CTA never
      // issued -- and waits for it.  Earlier phases are complete already: a
      // stage is armed or loaded again only after the MMAs have consumed it.
      // Neither CTA passes the final cluster barrier before this ends, so no
      // load can land in the shared memory of a CTA that has exited.
      volatile int never = 0;
      if (!leader) {
        st_shared_cluster_u32(mapa_shared(smem_u32(const_cast<uint32_t*>(peer_loaded)), 0), it);
        mbar_arrive_cluster(mapa_shared(peer_done_bar, 0));
      } else {
        uint32_t it1 = 0;
        if (mbar_wait_bounded<true>(peer_done_bar, 0, limit, &never)) {
          it1 = *peer_loaded;
        } else {
          atomicOr(p.status, kErrTimeoutDrain);
          it1 = it;  // unknown: wait for what rank 0 armed
        }
        const uint32_t hi = it > it1 ? it : it1;
        for (uint32_t i = hi > static_cast<uint32_t>(Cf::STAGES) ? hi - Cf::STAGES : 0; i < hi;
             ++i) {
          const uint32_t s = i % Cf::STAGES, ph = (i / Cf::STAGES) & 1u;
          const bool armed0 = i < it, loaded0 = armed0 && !(stalled_first && i == 0);
          const bool loaded1 = i < it1;
          if (!armed0) {
            mbar_arrive_expect_tx(full_bar(s), stage_tx);  // rank 1's bytes only
          } else {
            const uint32_t missing = (loaded0 ? 0u : stage_tx) + (loaded1 ? 0u : stage_tx);
            if (missing) mbar_complete_tx(full_bar(s), missing);
          }
          if (!mbar_wait_bounded(full_bar(s), ph, limit, &never))
            atomicOr(p.status, kErrTimeoutDrain);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (rank 0)
    // One thread of rank 0 waits and issues every MMA of the pair.
    if (leader && lane == 0) {
      uint32_t it = 0, tcount = 0;
      bool ok = true;
      // M = 256 (the pair), N = the tile's columns
      const uint32_t idesc =
          KIND == KIND_3XTF32 ? make_idesc(2, false, false, 2 * Cf::BM, bn) : Cf::IDESC;
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
          // the split kind's stages are completed by plain stores from both
          // CTAs, released at cluster scope
          if (!mbar_wait_bounded<has_converters<KIND>()>(full_bar(s), ph, limit, abort_flag)) {
            give_up_one(kErrTimeoutMma);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = sbase + s * Cf::STAGE_BYTES;
          if constexpr (KIND == KIND_BF16) {
            // A: BK/64 boxes of 128 rows x 128 B per CTA, K-major.  B: this
            // CTA's two 64-column boxes (B_BOX_BYTES apart), MN-major, each
            // holding BK k-rows of 128 B.
#pragma unroll
            for (int kk = 0; kk < Cf::BK / Cf::INSTR_K; ++kk) {
              const uint64_t ad =
                  smem_desc_sw128(st + (kk / 4) * Cf::A_BOX_BYTES + (kk % 4) * 32, 16, 1024);
              const uint64_t bd =
                  smem_desc_sw128(st + Cf::A_BYTES + kk * 2048, Cf::B_BOX_BYTES, 1024);
              mma_f16_pair(d_tmem, ad, bd, idesc, (kb > w.kb0 || kk > 0) ? 1u : 0u);
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
              mma_tf32_pair(d_tmem, asd, bbd, idesc, (kb > w.kb0 || kk > 0) ? 1u : 0u);
              mma_tf32_pair(d_tmem, abd, bsd, idesc, 1u);
              mma_tf32_pair(d_tmem, abd, bbd, idesc, 1u);
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
  } else if (warp < NUM_THREADS / 32) {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    const int ew = warp - 2;
    uint32_t tcount = 0, chunk = 0;
    bool prev_group = false;  // the warp's previous chunk committed a bulk group
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
      const int n0 = tn * bn;
      const int col_end = n0 + bn < p.N ? n0 + bn : p.N;
      // (accumulator b occupies TMEM columns [256 b, 256 b + bn); a last
      // chunk of 16 columns reads 16 allocated, unwritten ones, masked off)
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * Cf::BN;
#pragma unroll 1
      for (int c = 0; c < (bn + 31) / 32; ++c) {
        uint32_t r[32];
        tmem_ld_32cols(taddr + c * 32, r);
        // (the converter kinds, held to 80 or 128 registers, keep their odd
        // rows in registers)
        const OddRows odd = has_converters<KIND>()
                                ? OddRows{}
                                : plan_odd_rows(p, n0, n0 + c * 32, col_end, taddr + c * 32 + 32);
        tmem_ld_wait();
        prev_group = stage_and_store_chunk<TMA_STORE>(r, sbase + L::EPI_OFF, ew, chunk, lane,
                                                      &tmC, &tmC1, p, m0 + q * 32, n0 + c * 32,
                                                      col_end, w.reduce, odd, prev_group);
        ++chunk;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(acce_bar(buf), 0));
    }
    if (TMA_STORE || p.c_even) {  // every store of this warp has completed
      if (lane == 0) bulk_wait_group<0>();
      __syncwarp();
    }
  } else if constexpr (KIND == KIND_3XTF32_SPLIT_TMA_A) {
    // ------------------------------------------------------------ converters (both CTAs)
    // Group g takes the cluster's K-blocks g, g + 2, g + 4, ...
    const int g = (threadIdx.x - NUM_THREADS) / SPLIT_THREADS;
    const int ct = (threadIdx.x - NUM_THREADS) % SPLIT_THREADS;
    const StoreOffsets so(ct);
    const PairWalk walk{rank};
    auto convert = [&](auto vec_b) {
      constexpr bool VB = decltype(vec_b)::value;
      int total = 0;  // how many K-blocks this cluster stores
      for (int u = cluster; u < p.num_units; u += num_clusters) {
        const Unit w = unit_of(u, p);
        total += w.kb1 - w.kb0;
      }
      LoadCursor<PairWalk> ld;
      ld.seek(p, walk, cluster, ct);
      PrefetchCursor<PairWalk> pf;
      pf.seek(p, walk, cluster);
      for (int d = 0; d < g; ++d) ld.advance(p, walk, num_clusters, ct);
      for (int d = 0; d < g + 2 + SPLIT_PREFETCH; ++d) {
        if (d >= g + 2 && ((d - g) & 1) == 0) split_prefetch_l2(p, ct, pf);
        pf.advance(p, walk, num_clusters);
      }
      BRegs r;
      if (g < total) load_b<VB>(r, p, ld, ct);
      for (int it = g; it < total; it += 2) {
        const uint32_t s = it % Cf::STAGES, ph = (it / Cf::STAGES) & 1u;
        if (!warp_wait(empty_bar(s), ph ^ 1u, limit, abort_flag) ||
            !warp_wait(a_full_bar(s), ph, limit, abort_flag)) {
          give_up_pair(kErrTimeoutProducer);
          break;
        }
        split_store_tma_a(r, sbase + s * Cf::STAGE_BYTES, so, SPLIT_BOX_BYTES, true);
        fence_proxy_async_smem();  // the stores, visible to the pair's MMA reads
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(full_bar(s), 0));
        // the group's next K-block: its loads, and a prefetch two blocks further
        ld.advance(p, walk, num_clusters, ct);
        ld.advance(p, walk, num_clusters, ct);
        if (it + 2 < total) load_b<VB>(r, p, ld, ct);
        split_prefetch_l2(p, ct, pf);
        pf.advance(p, walk, num_clusters);
        pf.advance(p, walk, num_clusters);
      }
    };
    if (p.vec_b)
      convert(std::true_type{});
    else
      convert(std::false_type{});
  } else if constexpr (KIND == KIND_3XTF32_SPLIT) {
    // ------------------------------------------------------------ converters (both CTAs)
    const int ct = threadIdx.x - NUM_THREADS;
    const StoreOffsets so(ct);
    const PairWalk walk{rank};
    auto convert = [&](auto vec_a, auto vec_b) {
      constexpr bool VA = decltype(vec_a)::value, VB = decltype(vec_b)::value;
      // how many K-blocks this cluster stores
      int left = 0;
      for (int u = cluster; u < p.num_units; u += num_clusters) {
        const Unit w = unit_of(u, p);
        left += w.kb1 - w.kb0;
      }
      if (left == 0) return;
      LoadCursor<PairWalk> ld;
      ld.seek(p, walk, cluster, ct);
      PrefetchCursor<PairWalk> pf;
      pf.seek(p, walk, cluster);
      for (int d = 0; d < 2 + SPLIT_PREFETCH; ++d) {
        if (d >= 2) split_prefetch_l2(p, ct, pf);
        pf.advance(p, walk, num_clusters);
      }
      SplitRegs r0, r1;
      split_load<VA, VB>(r0, p, ld, ct);
      ld.advance(p, walk, num_clusters, ct);
      if (ld.valid) split_load<VA, VB>(r1, p, ld, ct);
      ld.advance(p, walk, num_clusters, ct);
      uint32_t it = 0;
      // Store the K-block held in r, then reuse r for the loads two blocks on.
      auto step = [&](SplitRegs& r) -> bool {
        const uint32_t s = it % Cf::STAGES, ph = (it / Cf::STAGES) & 1u;
        if (!warp_wait(empty_bar(s), ph ^ 1u, limit, abort_flag)) {
          give_up_pair(kErrTimeoutProducer);
          return false;
        }
        split_store(r, sbase + s * Cf::STAGE_BYTES, so);
        fence_proxy_async_smem();  // the stores, visible to the pair's MMA reads
        __syncwarp();
        // test hook: block 0 never completes its first stage
        const bool stall = p.inject_stall && blockIdx.x == 0 && it == 0;
        if (lane == 0 && !stall) mbar_arrive_cluster(mapa_shared(full_bar(s), 0));
        ++it;
        if (--left == 0) return false;
        if (ld.valid) split_load<VA, VB>(r, p, ld, ct);
        ld.advance(p, walk, num_clusters, ct);
        split_prefetch_l2(p, ct, pf);
        pf.advance(p, walk, num_clusters);
        return true;
      };
      while (step(r0) && step(r1)) {
      }
    };
    if (p.vec_a && p.vec_b)
      convert(std::true_type{}, std::true_type{});
    else if (p.vec_a)
      convert(std::true_type{}, std::false_type{});
    else if (p.vec_b)
      convert(std::false_type{}, std::true_type{});
    else
      convert(std::false_type{}, std::false_type{});
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // neither CTA leaves while the pair's MMAs or arrivals may touch it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, Cf::TMEM_COLS);
  }
}

// Zero the C tiles of the split work units (pair tiles [full_units,
// num_tiles)), which both K halves then add into.  Block (x, y) clears rows
// y * blockDim.y + threadIdx.y + k * gridDim.y * blockDim.y of split tile x,
// with 16-byte stores when `vec` (C 16-byte aligned, ldc % 4 == 0).
//
// Launched either in plain stream order (nothing of the call before it) or as
// a programmatic dependent of the call's pre-pass, which was itself launched
// in plain stream order, so everything before the call has finished in both
// cases and C may be written at once: the zeroing runs alongside the
// pre-pass.  Each block waits for its predecessor only before exiting, so
// that this kernel's completion, which the GEMM kernel waits for, implies the
// pre-pass's.
__global__ void zero_split_tiles_kernel(TcParams p, int tile_rows, int tile_cols, bool vec) {
  grid_launch_dependents();
  const int tile = p.full_units + blockIdx.x;
  int tm, tn;
  tile_coords(tile, p, tm, tn);
  const int64_t r0 = static_cast<int64_t>(tm) * tile_rows;
  const int64_t r_end = r0 + tile_rows < p.M ? r0 + tile_rows : p.M;
  const int64_t c0 = static_cast<int64_t>(tn) * tile_cols;
  const int cols = static_cast<int>(c0 + tile_cols < p.N ? tile_cols : p.N - c0);
  const int64_t r_step = static_cast<int64_t>(gridDim.y) * blockDim.y;
  for (int64_t r = r0 + blockIdx.y * blockDim.y + threadIdx.y; r < r_end; r += r_step) {
    float* crow = p.C + r * p.ldc + c0;
    if (vec) {
      for (int c = 4 * threadIdx.x; c < cols; c += 4 * blockDim.x) {
        if (c + 4 <= cols) {
          *reinterpret_cast<float4*>(crow + c) = make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
          for (int j = c; j < cols; ++j) crow[j] = 0.f;
        }
      }
    } else {
      for (int c = threadIdx.x; c < cols; c += blockDim.x) crow[c] = 0.f;
    }
  }
  grid_dependency_wait();
}

// Pair kernel launch: clusters of 2 CTAs, persistent over 256 x BN pair
// tiles, as many clusters as can be co-resident (at most one per pair tile).
template <int KIND, bool TMA_STORE>
cudaError_t launch_pair_t(const TcMaps& mp, const TcParams& p, bool after_prepass,
                          const DeviceCtl& ctl, cudaStream_t s) {
  auto kern = tc_gemm_pair_kernel<KIND, TMA_STORE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       PairLayout<KIND>::ALLOC);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(pair_threads<KIND>());
  cfg.dynamicSmemBytes = PairLayout<KIND>::ALLOC;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(2 * (ctl.sm_count / 2));
  int max_clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg);
  if (e != cudaSuccess) return e;
  if (max_clusters < 1) return cudaErrorInvalidConfiguration;
  int clusters = p.num_tiles < max_clusters ? p.num_tiles : max_clusters;
  // A last round that would leave more than half of the clusters idle is
  // split along K: its tiles become two half-K units each, reduce-added into
  // C (zeroed first).  Two addends onto zero give the same sum in either
  // order, so results stay bit-reproducible.
  TcParams q = p;
  q.c_even = !TMA_STORE && mp.c_even;
  q.c_odd_shift = q.c_even && !has_converters<KIND>() ? mp.c_odd_shift : -1;
  const int rem = p.num_tiles % clusters;
  if (KIND != KIND_BF16 && 2 * p.num_tiles <= max_clusters && p.num_kb >= 32) {
    // Few tiles (3xTF32): every tile becomes two half-K units, reduce-added
    // into C (zeroed first), so that twice as many clusters work.  GB300,
    // 1536^3: 60.0 -> 43.6 us per call with 256-column tiles; with fewer
    // K-blocks the zeroing and the second add cost more than they save
    // (1536 x 1536 x 512, 16 K-blocks: 25.2 against 23.2 us unsplit).
    q.full_units = 0;
    q.num_units = 2 * p.num_tiles;
    q.kb_mid = p.num_kb / 2;
    clusters = q.num_units;
    if ((e = launch_zero_split_tiles(q, 2 * PairCfg<KIND>::BM, q.bn, after_prepass, s)) !=
        cudaSuccess)
      return e;
  } else if (p.num_tiles > clusters && rem > 0 && 2 * rem <= clusters && p.num_kb >= 2) {
    q.full_units = p.num_tiles - rem;
    q.num_units = q.full_units + 2 * rem;
    q.kb_mid = p.num_kb / 2;
    if ((e = launch_zero_split_tiles(q, 2 * PairCfg<KIND>::BM, q.bn, after_prepass, s)) !=
        cudaSuccess)
      return e;
  }
  cfg.gridDim = dim3(2 * clusters);
  cfg.numAttrs = 2;  // and programmatic serialisation behind the kernel before
  char name[64];
  if (KIND == KIND_3XTF32 && p.bn != PairCfg<KIND>::BN)
    snprintf(name, sizeof(name), "tc_gemm_pair_kernel<3xtf32,n%d>", p.bn);
  else
    snprintf(name, sizeof(name), "%s",
             KIND == KIND_BF16                 ? "tc_gemm_pair_kernel<bf16>"
             : KIND == KIND_3XTF32             ? "tc_gemm_pair_kernel<3xtf32>"
             : KIND == KIND_3XTF32_SPLIT_TMA_A ? "tc_gemm_pair_kernel<3xtf32,split,tma-a>"
                                               : "tc_gemm_pair_kernel<3xtf32,split>");
  note_main_kernel(name, 2 * clusters, p.num_tiles);
  e = cudaLaunchKernelEx(&cfg, kern, mp.a0, mp.a1, mp.b0, mp.b1, mp.c, mp.c1, q);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_zero_split_tiles(const TcParams& q, int tile_rows, int tile_cols,
                                    bool after_prepass, cudaStream_t s) {
  const int split = q.num_tiles - q.full_units;
  if (split <= 0) return cudaSuccess;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(split, 8);
  cfg.blockDim = dim3(64, 4);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = after_prepass ? 1 : 0;  // see zero_split_tiles_kernel
  const bool vec = (reinterpret_cast<uintptr_t>(q.C) & 15u) == 0 && q.ldc % 4 == 0;
  note_launch();
  return cudaLaunchKernelEx(&cfg, zero_split_tiles_kernel, q, tile_rows, tile_cols, vec);
}

cudaError_t launch_cta_pair_split(bool tma_a, const float* A, const float* B, const TcMaps& maps,
                                  float* C, int64_t M, int64_t N, int64_t K, int64_t lda,
                                  int64_t ldb, int64_t ldc, bool c_tma, const DeviceCtl& ctl,
                                  cudaStream_t s) {
  TcParams p = make_params(M, N, K, PAIR_TILE_M, PAIR_TILE_N, PairCfg<KIND_3XTF32_SPLIT>::BK, C,
                           ldc, ctl);
  p.A = A;
  p.B = B;
  p.lda = lda;
  p.ldb = ldb;
  p.vec_a = (reinterpret_cast<uintptr_t>(A) % 16 == 0) && (lda % 4 == 0);
  p.vec_b = (reinterpret_cast<uintptr_t>(B) % 16 == 0) && (ldb % 4 == 0);
  if (tma_a)
    return c_tma ? launch_pair_t<KIND_3XTF32_SPLIT_TMA_A, true>(maps, p, false, ctl, s)
                 : launch_pair_t<KIND_3XTF32_SPLIT_TMA_A, false>(maps, p, false, ctl, s);
  return c_tma ? launch_pair_t<KIND_3XTF32_SPLIT, true>(maps, p, false, ctl, s)
               : launch_pair_t<KIND_3XTF32_SPLIT, false>(maps, p, false, ctl, s);
}

cudaError_t launch_cta_pair(int kind, const TcMaps& maps, float* C, int64_t M, int64_t N,
                            int64_t K, int64_t ldc, bool c_tma, bool after_prepass, int bn,
                            const DeviceCtl& ctl, cudaStream_t s) {
  if (kind == KIND_BF16) {
    const TcParams p = make_params(M, N, K, PAIR_TILE_M, PAIR_TILE_N, PairCfg<KIND_BF16>::BK, C,
                                   ldc, ctl);
    return c_tma ? launch_pair_t<KIND_BF16, true>(maps, p, after_prepass, ctl, s)
                 : launch_pair_t<KIND_BF16, false>(maps, p, after_prepass, ctl, s);
  }
  const TcParams p = make_params(M, N, K, PAIR_TILE_M, bn, PairCfg<KIND_3XTF32>::BK, C, ldc, ctl);
  return c_tma ? launch_pair_t<KIND_3XTF32, true>(maps, p, after_prepass, ctl, s)
               : launch_pair_t<KIND_3XTF32, false>(maps, p, after_prepass, ctl, s);
}

}  // namespace tc
}  // namespace mhr
