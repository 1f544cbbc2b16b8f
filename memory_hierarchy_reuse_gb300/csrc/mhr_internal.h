// Launchers shared between the C-ABI front end (api.cu) and the kernel
// translation units.  Every launcher assumes validated arguments (sizes >= 1,
// pointers non-null) and returns the launch's cudaError_t.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>
#include <mutex>

namespace mhr {

// Knobs read by the tensor-core kernels; set by the C-ABI front end.
struct DeviceCtl {
  uint32_t* status = nullptr;          // device address of the status word
  uint64_t wait_limit_ns = 2000000000ull;
  int inject_stall = 0;                // test hook: block 0 leaves its first ring stage incomplete
  int sm_count = 0;
  int pair_mode = 0;                   // 0 auto, 1 single-CTA kernel, 2 CTA-pair kernel (test hook)
  int raster_group = 0;                // tile rows per raster group, 0 = default (tuning hook)
  int split_mode = 0;                  // 3xTF32: 0 auto, 1 split pre-pass, 2 in-kernel split (test hook)
  int pair_tile_n = 0;                 // 3xTF32 CTA-pair tile columns, 0 = planned (test hook)
  int single_tile_n = 0;               // single-CTA tile columns, 0 = planned (test hook)
};

// wide_mode: 0 automatic, 1 never the 128 x 256 kernel, 2 that kernel
// whenever the sizes allow (see simt_wide_plan).
cudaError_t launch_simt_f32(const float* A, const float* B, float* C, int64_t M, int64_t N,
                            int64_t K, int64_t lda, int64_t ldb, int64_t ldc, int wide_mode,
                            cudaStream_t s);
// The SIMT kernel an M x N x K problem with 16-byte aligned operands takes on
// `sms` SMs: 0 the 128 x 128 kernel, 1 the 128 x 256 kernel, 2 that kernel on
// two K halves (host arithmetic only).
int simt_wide_plan(int64_t M, int64_t N, int64_t K, int sms, int wide_mode);

// The pages' ladder: rung 0 = one thread per output, 1 = 16 x 16 shared tiles,
// 2 = 32 x 32 shared tiles.  Requires ceil(M / T) <= 65535.
cudaError_t launch_ladder(int rung, const float* A, const float* B, float* C, int64_t M, int64_t N,
                          int64_t K, int64_t lda, int64_t ldb, int64_t ldc, cudaStream_t s);

// C[M x N] = 0 (the K == 0 case).
cudaError_t launch_zero_fill(float* C, int64_t M, int64_t N, int64_t ldc, cudaStream_t s);

// Copy a rows x cols matrix of 2-byte elements to a buffer with leading
// dimension dst_ld (used when a bf16 operand is not TMA-aligned).
cudaError_t launch_pack_u16(const uint16_t* src, int64_t rows, int64_t cols, int64_t src_ld,
                            uint16_t* dst, int64_t dst_ld, cudaStream_t s);

// 3xTF32 split: A (M x K, lda) -> a_big, a_small (M x Kp, K-contiguous; big
// truncated to tf32, a_big may be null when A itself serves as A_big);
// B (K x N, ldb) -> bt_big, bt_small (N x Kp, K-contiguous, i.e. B transposed;
// big truncated to tf32).
cudaError_t launch_split_tf32(const float* A, const float* B, int64_t M, int64_t N, int64_t K,
                              int64_t lda, int64_t ldb, int64_t Kp, float* a_big, float* a_small,
                              float* bt_big, float* bt_small, cudaStream_t s);

// bf16 x bf16 -> fp32 on tcgen05.  A: M x K bf16 (row pitch lda, 16-byte
// aligned rows), B: K x N bf16 (pitch ldb, aligned).  C via TMA store when
// c_tma is true (C 16-byte aligned, ldc % 4 == 0), else direct stores.
// after_prepass: this call launched a pre-pass (repack) just before, in plain
// stream order (see launch_cta_pair).
cudaError_t launch_tc_bf16(const uint16_t* A, const uint16_t* B, float* C, int64_t M, int64_t N,
                           int64_t K, int64_t lda, int64_t ldb, int64_t ldc, bool c_tma,
                           bool after_prepass, const DeviceCtl& ctl, cudaStream_t s);

// 3xTF32 main loop over the split operands (pitch Kp floats; a_big with
// pitch a_big_ld, which is A itself when a_big_ld = lda), launched right after
// the split pre-pass that writes them.
cudaError_t launch_tc_3xtf32(const float* a_big, int64_t a_big_ld, const float* a_small,
                             const float* bt_big, const float* bt_small, float* C, int64_t M,
                             int64_t N, int64_t K, int64_t Kp, int64_t ldc, bool c_tma,
                             const DeviceCtl& ctl, cudaStream_t s);

// Whether the 3xTF32 path may read A itself as its big part: TMA needs a
// 16-byte aligned base and a row pitch that is a multiple of 16 bytes.
inline bool a_serves_as_big(const float* A, int64_t lda) {
  return (reinterpret_cast<uintptr_t>(A) & 15u) == 0 && lda % 4 == 0;
}

// 3xTF32 with the split done inside the CTA-pair kernel: A (M x K, lda) and
// B (K x N, ldb) row-major fp32, read directly; no workspace.
cudaError_t launch_tc_3xtf32_split(const float* A, const float* B, float* C, int64_t M,
                                   int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                                   bool c_tma, const DeviceCtl& ctl, cudaStream_t s);

// 3xTF32 in one launch of the single-CTA kernel, split inside it (A staged by
// TMA as its own big part, so a_serves_as_big(A, lda) must hold); for
// problems small enough that a pre-pass launch would dominate.
cudaError_t launch_tc_3xtf32_small(const float* A, const float* B, float* C, int64_t M, int64_t N,
                                   int64_t K, int64_t lda, int64_t ldb, int64_t ldc, bool c_tma,
                                   const DeviceCtl& ctl, cudaStream_t s);

// Whether the tensor-core path of `kind` (KIND_BF16 or KIND_3XTF32, in
// tc_common.cuh) runs the CTA-pair kernel for this shape (else the
// single-CTA kernel); for 3xTF32 this may be at a narrower planned width.
bool tc_pair_chosen(int kind, int64_t M, int64_t N, int64_t K, const DeviceCtl& ctl);
// Whether a 3xTF32 call runs as one launch of the single-CTA kernel with the
// split inside (launch_tc_3xtf32_small): forced by the test hooks (split mode
// 2 with the single-CTA kernel), or chosen for small problems (M N <= 2^18,
// K <= 2048) in the automatic mode; A must be its own big part.
bool small_one_launch_chosen(const float* A, int64_t lda, int64_t M, int64_t N, int64_t K,
                             const DeviceCtl& ctl);
namespace tc {
// Columns of the CTA-pair kernel's 3xTF32 tiles (256, or a narrower multiple
// of 16 -- of 32 when C is written by TMA -- down to 128) for an M x N x K
// problem with up to `clusters` co-resident clusters; tc_gemm.cu gives the
// cost model.
int plan_pair_tile_n(int64_t M, int64_t N, int64_t K, int clusters, bool c_tma);
// For 3xTF32 problems with too few 256 x 256 tiles for half of the clusters:
// the CTA-pair tile columns (256, 192 or 128) that keep at least 80 % of the
// clusters busy, counting K halves, or 0 (the single-CTA kernel runs).
int few_tile_pair_width(int64_t M, int64_t N, int64_t K, int clusters);
// Columns of the single-CTA kernel's 3xTF32 tiles (128, 96, 64 or 32) on
// `sms` SMs; tc_gemm.cu gives the cost model.
int plan_single_tile_n(int64_t M, int64_t N, int64_t K, int sms, bool c_tma);
}  // namespace tc

// Whether C can be written with TMA stores: 16-byte aligned base and pitch,
// and N a multiple of 4.  A TMA store clips a box at the tensor's inner extent
// only in 16-byte units, so with N % 4 != 0 it would also write the columns
// of C's padding up to the next multiple of 4 (measured on GB300).
inline bool c_tma_eligible(const float* C, int64_t N, int64_t ldc) {
  return (reinterpret_cast<uintptr_t>(C) & 15u) == 0 && ldc % 4 == 0 && N % 4 == 0;
}

// Tensor-map encoding through the driver entry point (no libcuda link).
CUresult encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                        uint64_t inner, uint64_t outer, uint64_t row_pitch_bytes,
                        uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle);

// Name of the main kernel the last tensor-core or SIMT launch used, with its
// grid (for profiling labels; static storage).  Called right before that
// kernel's launch: counts as a launch, and records the caller's main-kernel
// start event there when one is set.
void note_main_kernel(const char* name, int grid, int tiles);
// Kernel-launch count of the current gemm_* call: reset by begin_call() at
// the start of every entry point, incremented by each launcher.
void begin_call();
void note_launch();
const char* last_main_kernel();

// The C-ABI front end's argument checks (api.cu), for entry points defined in
// other translation units.  Returns an mhr_status; *noop is set when M or N is 0.
int check_gemm_args(const void* A, const void* B, const void* C, int64_t M, int64_t N, int64_t K,
                    int64_t lda, int64_t ldb, int64_t ldc, int64_t esz_ab, bool* noop);

// The library lock (api.cu).  Every entry point holds it while it reads the
// settings, looks up device state and scratch, and enqueues its kernels.
std::mutex& library_mutex();

// The current device's kernel controls (status word, wait limit, SM count);
// MHR_ERR_UNSUPPORTED unless the device is sm_103.  The caller holds
// library_mutex().
int device_ctl_locked(DeviceCtl* ctl, int* dev);

// The caller's profiling events around the main kernel of a call
// (gemm_testing_set_main_kernel_events): while armed, note_main_kernel()
// records the start event on the call's stream right before the main kernel
// launch; disarming records the stop event.  The caller holds
// library_mutex().
void main_events_arm(cudaStream_t s);
void main_events_disarm();
struct MainKernelEvents {
  explicit MainKernelEvents(cudaStream_t s) { main_events_arm(s); }
  ~MainKernelEvents() { main_events_disarm(); }
  MainKernelEvents(const MainKernelEvents&) = delete;
  MainKernelEvents& operator=(const MainKernelEvents&) = delete;
};

}  // namespace mhr
