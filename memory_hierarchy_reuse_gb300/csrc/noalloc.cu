// gemm_f32_3xtf32_noalloc: the 3xTF32 GEMM with its scratch in static device
// memory, for callers that must not allocate device memory.
//
// gemm_f32_3xtf32 splits A and B into tf32 "big" and "small" parts in a
// workspace that the library allocates with cudaMalloc on first use (and
// grows later).  Some callers cannot have that happen inside a GEMM call: an
// application whose device memory is owned by its own pool allocator, which
// may have reserved nearly all of HBM so that an outside cudaMalloc fails or
// fragments it; latency-critical loops, where cudaMalloc/cudaFree
// synchronise the device and stall every stream; and programs in which only
// one owner thread may allocate.  This entry point computes the same product
// with the same kernels, but its split operands live in the fixed array below,
// so a call performs no allocation at all.
//
// Limits and sharing:
//   * the scratch holds 8 * Kp * (M + N) bytes, Kp = K rounded up to a
//     multiple of 4, at most kScratchBytes (64 MiB; e.g. M = N = K = 2048);
//     larger problems are rejected with MHR_ERR_INVALID_ARG before any work;
//   * every GPU on which the library is loaded keeps this 64 MiB until the
//     process exits;
//   * all calls on a device share the one array, and it keeps the last
//     call's contents.  Nothing in it needs to start at zero: every element a
//     call reads was written by that call's split pass.  Calls whose work
//     overlaps on the GPU (different streams, no ordering between them) race
//     on the array and give wrong results; order them on one stream or with
//     events;
//   * the first call on each device looks up the array's device address
//     (cudaGetSymbolAddress, with that device current).  Make that first call
//     before any stream capture begins.
#include <cuda_runtime.h>

#include <cstdint>
#include <map>
#include <mutex>

#include "mhr_gemm.h"
#include "mhr_internal.h"

#define MHR_API extern "C" __attribute__((visibility("default")))

// The scratch array: file scope, 64 MiB, 256-byte aligned.
static constexpr size_t kScratchBytes = size_t{64} << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

namespace mhr {
namespace {

std::mutex g_scratch_mu;
std::map<int, float*> g_scratch_addr;  // device -> device address of g_noalloc_scratch

// Device address of the scratch array on `dev` (the current device); looked
// up once per device.  In host code the array's name is only a host-side
// stand-in, so it must never be passed to a kernel directly.
int scratch_address(int dev, float** out) {
  std::lock_guard<std::mutex> g(g_scratch_mu);
  auto it = g_scratch_addr.find(dev);
  if (it == g_scratch_addr.end()) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return MHR_ERR_CUDA;
    }
    it = g_scratch_addr.emplace(dev, static_cast<float*>(p)).first;
  }
  *out = it->second;
  return MHR_OK;
}

}  // namespace
}  // namespace mhr

using namespace mhr;

MHR_API int gemm_f32_3xtf32_noalloc(const float* A, const float* B, float* C, int64_t M,
                                    int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                                    void* stream) {
  bool noop;
  int rc = check_gemm_args(A, B, C, M, N, K, lda, ldb, ldc, 4, &noop);
  if (rc != MHR_OK || noop) return rc;
  begin_call();
  const int64_t Kp = (K + 3) / 4 * 4;
  // 8 * Kp * (M + N) bytes must fit; M, N, K are below 2^31, so no overflow.
  if (K > 0 && static_cast<uint64_t>(Kp) * static_cast<uint64_t>(M + N) * 8u > kScratchBytes)
    return MHR_ERR_INVALID_ARG;
  // The same lock as every other entry point: the settings, the profiling
  // events and the launch counters are shared library state.
  std::lock_guard<std::mutex> lock(library_mutex());
  DeviceCtl ctl;
  int dev = 0;
  if ((rc = device_ctl_locked(&ctl, &dev)) != MHR_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (K == 0) {
    e = launch_zero_fill(C, M, N, ldc, s);
  } else if (small_one_launch_chosen(A, lda, M, N, K, ctl)) {  // as in gemm_f32_3xtf32
    MainKernelEvents ev(s);
    e = launch_tc_3xtf32_small(A, B, C, M, N, K, lda, ldb, ldc, c_tma_eligible(C, N, ldc), ctl,
                               s);
  } else {
    float* scratch;
    if ((rc = scratch_address(dev, &scratch)) != MHR_OK) return rc;
    float* a_big = scratch;
    float* a_small = a_big + M * Kp;
    float* bt_big = a_small + M * Kp;
    float* bt_small = bt_big + N * Kp;
    const bool a_raw = a_serves_as_big(A, lda);  // as in gemm_f32_3xtf32
    e = launch_split_tf32(A, B, M, N, K, lda, ldb, Kp, a_raw ? nullptr : a_big, a_small, bt_big,
                          bt_small, s);
    if (e == cudaSuccess) {
      const bool c_tma = c_tma_eligible(C, N, ldc);
      MainKernelEvents ev(s);
      e = launch_tc_3xtf32(a_raw ? A : a_big, a_raw ? lda : Kp, a_small, bt_big, bt_small, C, M,
                           N, K, Kp, ldc, c_tma, ctl, s);
    }
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MHR_ERR_CUDA;
  }
  return MHR_OK;
}
