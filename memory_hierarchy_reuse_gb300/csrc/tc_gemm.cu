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
  if (2 * pair_tiles < clusters) return false;
  return kind != tc::KIND_BF16 || K >= 2048 || pair_tiles >= 2 * clusters;
}

namespace {

using namespace tc;

// 1-CTA or CTA-pair kernel.  The pair kernel moves half the shared-memory
// bytes per FLOP; it is chosen once its 256 x 256 tiles occupy at least half
// of the clusters, and for bf16 only when there is also enough work per tile
// to amortise its prologue and epilogue (K >= 2048, or at least two rounds of
// tiles).  3xTF32 needs no such margin: its 1-CTA tile, 128 x 128, reads as
// many shared-memory bytes per clock as the MMAs consume and runs the tensor
// pipe near 57 % busy.  GB300 measurements, 3xTF32 calls: pair faster at
// 2048^3 (1.2x), 2048 x 2048 x 1024 (1.13x), 3000 x 2048 x 1000 (1.12x),
// 8192 x 1024 x 1024 (1.18x); 1-CTA faster at 1536^3 (36 pair tiles) and
// 1024 x 1024 x 4096 (16).  bf16: 1-CTA (128 x 256 tiles) faster at
// 3000 x 2050 x 1000.  DeviceCtl::pair_mode forces one of them (tests).
cudaError_t launch_tc_any(int kind, const TcMaps& maps, float* C, int64_t M, int64_t N, int64_t K,
                          int64_t ldc, bool c_tma, bool after_prepass, const DeviceCtl& ctl,
                          cudaStream_t s) {
  return tc_pair_chosen(kind, M, N, K, ctl)
             ? launch_cta_pair(kind, maps, C, M, N, K, ldc, c_tma, after_prepass, ctl, s)
             : launch_single_cta(kind, maps, C, M, N, K, ldc, c_tma, after_prepass, ctl, s);
}

CUresult encode_c_map(CUtensorMap* cm, float* C, int64_t M, int64_t N, int64_t ldc, bool c_tma) {
  if (!c_tma) return CUDA_SUCCESS;
  return encode_tmap_2d(cm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, C, N, M, ldc * 4, 32, 32,
                        CU_TENSOR_MAP_SWIZZLE_128B);
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
      encode_c_map(&mp.c, C, M, N, ldc, c_tma) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  mp.a1 = mp.a0;  // unused by the bf16 kernels
  mp.b1 = mp.b0;
  if (!c_tma) mp.c = mp.a0;  // unused without TMA stores
  return launch_tc_any(KIND_BF16, mp, C, M, N, K, ldc, c_tma, after_prepass, ctl, s);
}

cudaError_t launch_tc_3xtf32(const float* a_big, int64_t a_big_ld, const float* a_small,
                             const float* bt_big, const float* bt_small, float* C, int64_t M,
                             int64_t N, int64_t K, int64_t Kp, int64_t ldc, bool c_tma,
                             const DeviceCtl& ctl, cudaStream_t s) {
  TcMaps mp;
  const auto f32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  if (encode_tmap_2d(&mp.a0, f32, a_big, K, M, a_big_ld * 4, 32, 128, sw) != CUDA_SUCCESS ||
      encode_tmap_2d(&mp.a1, f32, a_small, K, M, Kp * 4, 32, 128, sw) != CUDA_SUCCESS ||
      encode_tmap_2d(&mp.b0, f32, bt_big, K, N, Kp * 4, 32, 128, sw) != CUDA_SUCCESS ||
      encode_tmap_2d(&mp.b1, f32, bt_small, K, N, Kp * 4, 32, 128, sw) != CUDA_SUCCESS ||
      encode_c_map(&mp.c, C, M, N, ldc, c_tma) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  if (!c_tma) mp.c = mp.a0;  // unused without TMA stores
  return launch_tc_any(KIND_3XTF32, mp, C, M, N, K, ldc, c_tma, true, ctl, s);
}

cudaError_t launch_tc_3xtf32_split(const float* A, const float* B, float* C, int64_t M,
                                   int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                                   bool c_tma, const DeviceCtl& ctl, cudaStream_t s) {
  TcMaps mp = {};
  if (encode_c_map(&mp.c, C, M, N, ldc, c_tma) != CUDA_SUCCESS) return cudaErrorInvalidValue;
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
  if (encode_c_map(&mp.c, C, M, N, ldc, c_tma) != CUDA_SUCCESS ||
      encode_tmap_2d(&mp.a0, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, A, K, M, lda * 4, 32, 128,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  return launch_single_cta_split(mp, A, B, C, M, N, K, lda, ldb, ldc, c_tma, ctl, s);
}

}  // namespace mhr
