// Entry of the tensor-core paths: tensor-map encoding and the choice between
// the single-CTA kernel (tc_gemm_1cta.cu) and the CTA-pair kernel
// (tc_gemm_pair.cu).
#include "tc_common.cuh"

namespace mhr {

bool tc_pair_chosen(int kind, int64_t M, int64_t N, int64_t K, const DeviceCtl& ctl) {
  if (ctl.pair_mode == 1) return false;
  if (ctl.pair_mode == 2) return true;
  const int64_t pair_tiles = ((M + tc::PAIR_TILE_M - 1) / tc::PAIR_TILE_M) *
                             ((N + tc::PAIR_TILE_N - 1) / tc::PAIR_TILE_N);
  const int64_t clusters = ctl.sm_count / 2;
  if (2 * pair_tiles < clusters)  // 3xTF32: unless few_tile_pair_width finds a width
    return kind == tc::KIND_3XTF32 && ctl.pair_tile_n == 0 &&
           tc::few_tile_pair_width(M, N, K, static_cast<int>(clusters)) > 0;
  return kind != tc::KIND_BF16 || K >= 1536 || pair_tiles >= 2 * clusters;
}

// Small 3xTF32 problems run as one launch with the split inside the
// single-CTA kernel (no pre-pass, no zeroing, no workspace), on tiles of 128
// rows x 128, 64 or 32 columns with a cluster per tile splitting K.  GB300,
// whole calls, L2 flushed, against the split pre-pass path: 256^3 13.0
// against 13.9 us, 512^3 15.1 / 16.8, 300 x 520 x 1000 19.1 / 22.1,
// 256 x 512 x 1000 17.1 / 21.9, 128 x 128 x 1024 14.9 / 20.2, 256 x 256 x 2048
// 19.1 / 23.3, 512 x 512 x 2048 25.3 / 25.3; the pre-pass path wins from 768^3
// (20.4 against 21.2) and at 1024^3 (25.7 / 33.4), where each CTA's converter
// warps would walk too many K-blocks.
bool small_one_launch_chosen(const float* A, int64_t lda, int64_t M, int64_t N, int64_t K,
                             const DeviceCtl& ctl) {
  if (!a_serves_as_big(A, lda) || ctl.pair_mode == 2) return false;
  if (ctl.split_mode == 2) return ctl.pair_mode == 1;
  return ctl.split_mode == 0 && M * N <= (int64_t{1} << 18) && K <= 2048;
}

namespace tc {

// Pair tile width for 3xTF32.  Each CTA of a pair computes 128 rows x bn
// columns, so a tile's MMA time is proportional to bn and to its K-blocks;
// what varies with bn is how many tiles the problem needs (ceil(N / bn) per
// row of tiles), how the tiles fall into rounds over the co-resident
// clusters, whether the last round is split along K (then C is zeroed and
// both halves add into it), and how many shared-memory bytes each tensor
// cycle needs.  Per instruction-K step a CTA's MMAs read its 128 x 8 A part
// (4 KB) and bn / 2 x 8 of B (16 bn bytes) while the tensor pipe works bn / 2
// cycles, and TMA writes 32 KB of A and 128 bn bytes of B per K-block of 12
// MMAs: 13653 / bn + 53.3 bytes per cycle in all, 107 at bn = 256.  Shared
// memory delivers about 125 bytes per cycle (the bf16 kernels' measured
// ceiling), so narrower tiles run below the full tensor rate.  The estimate
// below is the busiest cluster's MMA cycles plus the last epilogue, which
// nothing overlaps (TMA stores or, when C is not TMA-aligned, register stores
// at about a third of their rate; atomic adds after a K split).  bn = 256
// unless a narrower width is at least 5 % faster by this estimate.
double pair_cycles_estimate(int64_t M, int64_t N, int64_t K, int clusters_max, bool c_tma,
                            int bn) {
  const int64_t tiles = ((M + PAIR_TILE_M - 1) / PAIR_TILE_M) * ((N + bn - 1) / bn);
  const int64_t clusters = tiles < clusters_max ? tiles : clusters_max;
  const int64_t kb = (K + 31) / 32;
  const double demand = 13653.3 / bn + 53.3;
  const double eff = demand > 125.0 ? 125.0 / demand : 1.0;
  const double tile = static_cast<double>(kb) * 6.0 * bn / eff;
  const int64_t full = tiles / clusters, rem = tiles % clusters;
  double rounds;
  bool split = false;
  if (rem == 0) {
    rounds = static_cast<double>(full);
  } else if (tiles > clusters && 2 * rem <= clusters && kb >= 2) {
    rounds = full + 0.5;
    split = true;
  } else {
    rounds = static_cast<double>(full + 1);
  }
  const double epi_per_col = split ? (c_tma ? 20.0 : 58.0) : (c_tma ? 25.0 : 61.0);
  return rounds * tile + epi_per_col * bn;
}

// A 3xTF32 problem with too few 256 x 256 tiles for half of the clusters:
// the widest CTA-pair tile (256, 192 or 128 columns) whose work units keep at
// least 80 % of the clusters busy -- every tile split into two K halves when
// twice the tiles fit on the clusters (the pair kernel does so from 32
// K-blocks on) -- or 0, leaving the problem to the single-CTA kernel.  GB300,
// whole calls against the single-CTA kernel: 1536^3 43.6 / 47.7 us and
// 1024 x 2048 x 2048 52.8 / 60.0 (256 columns, 72 and 64 half-K units),
// 1024 x 1024 x 4096 61.1 / 64.1 and 1024^3 26.2 / 26.2 (128 columns, 64
// units); 768^3 (36 units of 128 columns) and 512 x 512 x 8192 (16) stay on
// the single-CTA kernel.
int few_tile_pair_width(int64_t M, int64_t N, int64_t K, int clusters) {
  const int64_t kb = (K + 31) / 32;
  const int64_t rows = (M + PAIR_TILE_M - 1) / PAIR_TILE_M;
  for (const int bn : {256, 192, 128}) {
    const int64_t tiles = rows * ((N + bn - 1) / bn);
    const int64_t units = 2 * tiles <= clusters && kb >= 32 ? 2 * tiles : tiles;
    if (units <= clusters && 5 * units >= 4 * static_cast<int64_t>(clusters)) return bn;
  }
  return 0;
}

int plan_pair_tile_n(int64_t M, int64_t N, int64_t K, int clusters, bool c_tma) {
  if (clusters < 1) return PAIR_TILE_N;
  const double full_width = pair_cycles_estimate(M, N, K, clusters, c_tma, PAIR_TILE_N);
  int best = PAIR_TILE_N;
  double best_t = full_width;
  // TMA stores write C in chunks of 32 columns, so their tiles are whole chunks
  for (int bn = PAIR_TILE_N - (c_tma ? 32 : 16); bn >= 128; bn -= c_tma ? 32 : 16) {
    const double t = pair_cycles_estimate(M, N, K, clusters, c_tma, bn);
    if (t < best_t) {
      best_t = t;
      best = bn;
    }
  }
  return best_t <= 0.95 * full_width ? best : PAIR_TILE_N;
}

// Tile width of the single-CTA 3xTF32 kernel (128 rows x bn, bn = 128, 96,
// 64 or 32; it runs problems with too few 256 x 256 tiles to fill the CTA
// pairs).  Narrower tiles put more SMs on a small problem: with every tile in
// one round (or split into K halves when twice the tiles fit), a unit's time
// is its K-blocks times the slower of two rates -- TMA filling the stage
// (A's 32 KB plus 256 bn bytes of B at some 64 bytes per SM cycle, measured
// on the 256^3 main loop) and the 12 MMAs of N = bn (6 bn cycles) -- plus
// its last epilogue (about 20 cycles per column with TMA stores, 60 with
// register stores).  The cluster split keeps whole tiles; bn = 128 unless a
// narrower width is at least 5 % faster by this estimate.
double single_cycles_estimate(int64_t M, int64_t N, int64_t K, int sms, bool c_tma, int bn) {
  const int64_t tiles = ((M + 127) / 128) * ((N + bn - 1) / bn);
  const int64_t kb = (K + 31) / 32;
  const bool split = 2 * tiles <= sms && kb >= 4;
  const int64_t units = split ? 2 * tiles : tiles;
  const int64_t kb_unit = split ? kb - kb / 2 : kb;
  const int64_t rounds = (units + sms - 1) / sms;
  const double fill = (32768.0 + 256.0 * bn) / 64.0, mma = 6.0 * bn;
  return static_cast<double>(rounds * kb_unit) * (fill > mma ? fill : mma) +
         (c_tma ? 20.0 : 60.0) * bn;
}

int plan_single_tile_n(int64_t M, int64_t N, int64_t K, int sms, bool c_tma) {
  if (sms < 1) return 128;
  const int64_t tiles = ((M + 127) / 128) * ((N + 127) / 128);
  if (2 * tiles <= sms && (K + 31) / 32 >= 64) return 128;  // the cluster split's domain
  const double full_width = single_cycles_estimate(M, N, K, sms, c_tma, 128);
  int best = 128;
  double best_t = full_width;
  for (int bn = 96; bn >= 32; bn -= 32) {
    const double t = single_cycles_estimate(M, N, K, sms, c_tma, bn);
    if (t < best_t) {
      best_t = t;
      best = bn;
    }
  }
  return best_t <= 0.95 * full_width ? best : 128;
}

}  // namespace tc

namespace {

using namespace tc;

// 1-CTA or CTA-pair kernel.  The pair kernel moves half the shared-memory
// bytes per FLOP; it is chosen once its 256 x 256 tiles occupy at least half
// of the clusters, and for bf16 only when there is also enough work per tile
// to amortise its prologue and epilogue (K >= 1536, or at least two rounds of
// tiles).  3xTF32 needs no such margin: its 1-CTA tile, 128 x 128, reads as
// many shared-memory bytes per clock as the MMAs consume and runs the tensor
// pipe near 57 % busy.  GB300 measurements, 3xTF32 calls: pair faster at
// 2048^3 (1.2x), 2048 x 2048 x 1024 (1.13x), 3000 x 2048 x 1000 (1.12x),
// 8192 x 1024 x 1024 (1.18x); 1-CTA faster at 1536^3 with 256-column pair
// tiles (36 of them; with the planner's 128-column ones, 72, the pair kernel
// wins: tc_pair_chosen) and 1024 x 1024 x 4096 (16).  bf16, against the 1-CTA kernel's
// 128 x 256 tiles: pair faster at 2560 x 2560 x 1536 (27.3 / 29.3 us), 3000 x 2050 x 1536
// (46.7 / 51.8) and 2304 x 2560 x 2000 (31.4 / 35.5), equal at 2048 x 2048 x 1536; 1-CTA
// faster at 2048 x 2048 x 1280 (17.0 / 19.1) and 2560 x 2048 x 256 (15.0 / 19.1).
// DeviceCtl::pair_mode forces one of them (tests).
cudaError_t launch_tc_any(int kind, const TcMaps& maps, float* C, int64_t M, int64_t N, int64_t K,
                          int64_t ldc, bool c_tma, bool after_prepass, const DeviceCtl& ctl,
                          cudaStream_t s) {
  return tc_pair_chosen(kind, M, N, K, ctl)
             ? launch_cta_pair(kind, maps, C, M, N, K, ldc, c_tma, after_prepass, PAIR_TILE_N,
                               ctl, s)
             : launch_single_cta(kind, maps, C, M, N, K, ldc, c_tma, after_prepass, 0, ctl, s);
}

// C's map: the whole of C in boxes of 32 x 32 when TMA can store C.
// Otherwise, when C is 16-byte aligned and ldc even (so that every other row
// starts on a 16-byte boundary: the case of an ldc that is 2 mod 4, or of N
// not a multiple of 4), a map over C's even rows (pitch 2 ldc, boxes of 32
// columns x 16 rows) with which the register-store kernels write half of
// each chunk by TMA (TcMaps::c_even), and a map over the odd rows: row
// 2 y + 1 starts ldc floats after row 2 y, so its base moves ldc % 4 columns
// left, to the 16-byte boundary below (TcMaps::c_odd_shift; its first
// columns then belong to the row above and are never written).
CUresult encode_c_map(TcMaps* mp, float* C, int64_t M, int64_t N, int64_t ldc, bool c_tma) {
  const auto f32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  mp->c_even = false;
  mp->c_odd_shift = -1;
  if (c_tma) return encode_tmap_2d(&mp->c, f32, C, N, M, ldc * 4, 32, 32, sw);
  if ((reinterpret_cast<uintptr_t>(C) & 15u) == 0 && ldc % 2 == 0 &&
      encode_tmap_2d(&mp->c, f32, C, N, (M + 1) / 2, ldc * 8, 32, 16, sw) == CUDA_SUCCESS) {
    mp->c_even = true;
    const int64_t shift = ldc % 4;  // 0 or 2
    if (M >= 2 && encode_tmap_2d(&mp->c1, f32, C + ldc - shift, N + shift, M / 2, ldc * 8, 32,
                                 16, sw) == CUDA_SUCCESS)
      mp->c_odd_shift = static_cast<int>(shift);
  }
  return CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_tc_bf16(const uint16_t* A, const uint16_t* B, float* C, int64_t M, int64_t N,
                           int64_t K, int64_t lda, int64_t ldb, int64_t ldc, bool c_tma,
                           bool after_prepass, const DeviceCtl& ctl, cudaStream_t s) {
  TcMaps mp;
  if (encode_tmap_2d(&mp.a0, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A, K, M, lda * 2, 64, 128,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
      encode_tmap_2d(&mp.b0, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, B, N, K, ldb * 2, 64, 64,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
      encode_c_map(&mp, C, M, N, ldc, c_tma) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  mp.a1 = mp.a0;  // unused by the bf16 kernels
  mp.b1 = mp.b0;
  if (!c_tma && !mp.c_even) mp.c = mp.a0;  // unused without TMA stores
  if (mp.c_odd_shift < 0) mp.c1 = mp.c;
  return launch_tc_any(KIND_BF16, mp, C, M, N, K, ldc, c_tma, after_prepass, ctl, s);
}

cudaError_t launch_tc_3xtf32(const float* a_big, int64_t a_big_ld, const float* a_small,
                             const float* bt_big, const float* bt_small, float* C, int64_t M,
                             int64_t N, int64_t K, int64_t Kp, int64_t ldc, bool c_tma,
                             const DeviceCtl& ctl, cudaStream_t s) {
  TcMaps mp;
  const auto f32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  // The CTA-pair kernel's tiles are 256 x bn (each CTA loads bn / 2 rows of
  // B^T per part), the single-CTA kernel's 128 x bn (bn rows).  A tile width
  // the planner would not give with TMA stores (one that is not whole
  // 32-column chunks, forced by the test hook) writes C with register stores.
  const bool pair = tc_pair_chosen(KIND_3XTF32, M, N, K, ctl);
  const int clusters = ctl.sm_count / 2;
  const int few = few_tile_pair_width(M, N, K, clusters);
  const int64_t tiles256 = ((M + PAIR_TILE_M - 1) / PAIR_TILE_M) * ((N + PAIR_TILE_N - 1) / PAIR_TILE_N);
  int bn;
  if (pair) {
    bn = ctl.pair_tile_n > 0                  ? ctl.pair_tile_n
         : 2 * tiles256 < clusters && few > 0 ? few
                                              : plan_pair_tile_n(M, N, K, clusters, c_tma);
  } else if (ctl.single_tile_n > 0 && ctl.single_tile_n <= 128) {
    bn = ctl.single_tile_n;
  } else {
    bn = plan_single_tile_n(M, N, K, ctl.sm_count, c_tma);
  }
  const bool tma_c = c_tma && bn % 32 == 0;
  const int b_box_rows = pair ? bn / 2 : bn;
  if (encode_tmap_2d(&mp.a0, f32, a_big, K, M, a_big_ld * 4, 32, 128, sw) != CUDA_SUCCESS ||
      encode_tmap_2d(&mp.a1, f32, a_small, K, M, Kp * 4, 32, 128, sw) != CUDA_SUCCESS ||
      encode_tmap_2d(&mp.b0, f32, bt_big, K, N, Kp * 4, 32, b_box_rows, sw) != CUDA_SUCCESS ||
      encode_tmap_2d(&mp.b1, f32, bt_small, K, N, Kp * 4, 32, b_box_rows, sw) != CUDA_SUCCESS ||
      encode_c_map(&mp, C, M, N, ldc, tma_c) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  if (!tma_c && !mp.c_even) mp.c = mp.a0;  // unused without TMA stores
  if (mp.c_odd_shift < 0) mp.c1 = mp.c;
  return pair ? launch_cta_pair(KIND_3XTF32, mp, C, M, N, K, ldc, tma_c, true, bn, ctl, s)
              : launch_single_cta(KIND_3XTF32, mp, C, M, N, K, ldc, tma_c, true, bn, ctl, s);
}

cudaError_t launch_tc_3xtf32_split(const float* A, const float* B, float* C, int64_t M,
                                   int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                                   bool c_tma, const DeviceCtl& ctl, cudaStream_t s) {
  TcMaps mp = {};
  if (encode_c_map(&mp, C, M, N, ldc, c_tma) != CUDA_SUCCESS) return cudaErrorInvalidValue;
  // A itself, staged by TMA as its big part, when TMA can address it.
  const bool tma_a = a_serves_as_big(A, lda);
  if (tma_a && encode_tmap_2d(&mp.a0, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, A, K, M, lda * 4, 32, 128,
                              CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  return launch_cta_pair_split(tma_a, A, B, mp, C, M, N, K, lda, ldb, ldc, c_tma, ctl, s);
}

cudaError_t launch_tc_3xtf32_small(const float* A, const float* B, float* C, int64_t M, int64_t N,
                                   int64_t K, int64_t lda, int64_t ldb, int64_t ldc, bool c_tma,
                                   const DeviceCtl& ctl, cudaStream_t s) {
  TcMaps mp = {};
  if (encode_c_map(&mp, C, M, N, ldc, c_tma) != CUDA_SUCCESS ||
      encode_tmap_2d(&mp.a0, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, A, K, M, lda * 4, 32, 128,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  return launch_single_cta_split(mp, A, B, C, M, N, K, lda, ldb, ldc, c_tma, ctl, s);
}

}  // namespace mhr
