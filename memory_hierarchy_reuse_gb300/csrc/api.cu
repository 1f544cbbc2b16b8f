// C-ABI front end of libmhr_gemm.so: argument validation, degenerate cases,
// workspace management, tensor-map encoding and kernel dispatch.  The
// operation and its contract are documented in include/mhr_gemm.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "mhr_gemm.h"
#include "mhr_gemm_testing.h"
#include "mhr_internal.h"

#define MHR_API extern "C" __attribute__((visibility("default")))

namespace mhr {
namespace {

constexpr int kVersion = 1 * 10000 + 0 * 100 + 0;
constexpr int64_t kMaxDim = (int64_t{1} << 31) - 512;  // tile/TMA coordinates are int32

// Per-device status word: tensor-core kernels OR their timeout bits into it.
__device__ uint32_t g_status_word;
// gemm_check's copy of the status word, taken and cleared in one atomic step
// on the caller's stream.
__device__ uint32_t g_status_taken;

__global__ void take_status_kernel(uint32_t* status, uint32_t* out) {
  *out = atomicExch(status, 0u);
}

struct DeviceState {
  int checked = 0;  // 0 = not yet, 1 = sm_103, 2 = unsupported
  uint32_t* status = nullptr;
  uint32_t* taken = nullptr;
  int sm_count = 0;
};

// A workspace belongs to one (device, stream).  `last_use` is recorded on the
// stream after every call that used the buffer; a call waits for it on its
// own stream before touching the buffer, so a stream handle reused after
// cudaStreamDestroy (whose last kernels may still be running) cannot overwrite
// data they read, and the host waits for it before freeing the buffer.
struct Workspace {
  void* ptr = nullptr;
  size_t bytes = 0;
  cudaEvent_t last_use = nullptr;
  uint64_t stamp = 0;  // least recently used workspaces are freed first
};
// Workspaces kept per device; a call on a further stream frees the least
// recently used one first.
constexpr int kMaxWorkspacesPerDevice = 4;

std::mutex g_mu;
std::map<int, DeviceState> g_devices;
std::map<std::pair<int, cudaStream_t>, Workspace> g_workspaces;
uint64_t g_workspace_clock = 0;
uint64_t g_wait_limit_ns = 2000000000ull;
int g_inject_stall = 0;
int g_pair_mode = 0;
int g_raster_group = 0;
int g_split_mode = 0;
int g_pair_tile_n = 0;
int g_single_tile_n = 0;
int g_simt_wide_mode = 0;
uint64_t g_workspace_limit = UINT64_MAX;
int g_zero_a_small = 0;
cudaEvent_t g_main_start = nullptr, g_main_stop = nullptr;

// The caller's profiling events around the main kernel launch, if set (see
// MainKernelEvents in mhr_internal.h).  Entry points hold g_mu meanwhile.
cudaStream_t g_events_stream = nullptr;
bool g_events_armed = false;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// Current device: check it is sm_103 and find its status word (once).
int device_state(DeviceState** out, int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MHR_ERR_CUDA;
  DeviceState& st = g_devices[dev];
  if (st.checked == 0) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MHR_ERR_CUDA;
    if (major != 10 || minor != 3) {
      st.checked = 2;
    } else {
      void* p = nullptr;
      void* q = nullptr;
      if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess ||
          cudaGetSymbolAddress(&q, g_status_taken) != cudaSuccess) {
        cudaGetLastError();
        return MHR_ERR_CUDA;
      }
      st.status = static_cast<uint32_t*>(p);
      st.taken = static_cast<uint32_t*>(q);
      st.sm_count = sms;
      st.checked = 1;
    }
  }
  if (st.checked != 1) return MHR_ERR_UNSUPPORTED;
  *out = &st;
  if (dev_out) *dev_out = dev;
  return MHR_OK;
}

bool mul_ok(int64_t a, int64_t b, int64_t* r) { return !__builtin_mul_overflow(a, b, r); }

// Byte extent [lo, hi) of a rows x cols row-major matrix with pitch ld.
bool extent(const void* p, int64_t rows, int64_t cols, int64_t ld, int64_t esz, uintptr_t* lo,
            uintptr_t* hi) {
  int64_t span, bytes;
  if (!mul_ok(rows - 1, ld, &span) || __builtin_add_overflow(span, cols, &span) ||
      !mul_ok(span, esz, &bytes))
    return false;
  *lo = reinterpret_cast<uintptr_t>(p);
  if (__builtin_add_overflow(*lo, static_cast<uintptr_t>(bytes), hi)) return false;
  return true;
}

bool overlaps(uintptr_t a0, uintptr_t a1, uintptr_t b0, uintptr_t b1) { return a0 < b1 && b0 < a1; }

// Shared validation.  Returns MHR_OK with *noop set when there is nothing to do.
int validate(const void* A, const void* B, const void* C, int64_t M, int64_t N, int64_t K,
             int64_t lda, int64_t ldb, int64_t ldc, int64_t esz_ab, bool* noop) {
  *noop = false;
  if (M < 0 || N < 0 || K < 0) return MHR_ERR_INVALID_ARG;
  if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return MHR_ERR_INVALID_ARG;
  if (M == 0 || N == 0) {
    *noop = true;
    return MHR_OK;
  }
  if (C == nullptr || ldc < N) return MHR_ERR_INVALID_ARG;
  uintptr_t c0, c1;
  if (!extent(C, M, N, ldc, 4, &c0, &c1)) return MHR_ERR_INVALID_ARG;
  if (K == 0) return MHR_OK;
  if (A == nullptr || B == nullptr || lda < K || ldb < N) return MHR_ERR_INVALID_ARG;
  uintptr_t a0, a1, b0, b1;
  if (!extent(A, M, K, lda, esz_ab, &a0, &a1) || !extent(B, K, N, ldb, esz_ab, &b0, &b1))
    return MHR_ERR_INVALID_ARG;
  if (overlaps(c0, c1, a0, a1) || overlaps(c0, c1, b0, b1)) return MHR_ERR_INVALID_ARG;
  return MHR_OK;
}

// Frees a workspace once the last call that used it has finished.
void free_workspace(int dev, Workspace& w) {
  int cur = 0;
  cudaGetDevice(&cur);
  if (cur != dev) cudaSetDevice(dev);
  if (w.last_use) {
    cudaEventSynchronize(w.last_use);
    cudaEventDestroy(w.last_use);
  }
  if (w.ptr) cudaFree(w.ptr);
  cudaGetLastError();
  if (cur != dev) cudaSetDevice(cur);
  w = Workspace{};
}

// Workspace of at least `bytes` for (device, stream), ready for use on `s`:
// the stream has been made to wait for the buffer's previous use.  The caller
// records that use with workspace_used() after its launches.  At most
// kMaxWorkspacesPerDevice are kept per device.
int workspace(int dev, cudaStream_t s, size_t bytes, void** out, Workspace** ws_out) {
  constexpr size_t kGrain = size_t{2} << 20;
  if (bytes > SIZE_MAX - kGrain) return MHR_ERR_CUDA;  // no such allocation exists
  if (bytes > g_workspace_limit) return MHR_ERR_CUDA;  // test hook: as if cudaMalloc failed
  const auto key = std::make_pair(dev, s);
  if (g_workspaces.find(key) == g_workspaces.end()) {
    int kept = 0;
    auto lru = g_workspaces.end();
    for (auto it = g_workspaces.begin(); it != g_workspaces.end(); ++it) {
      if (it->first.first != dev) continue;
      ++kept;
      if (lru == g_workspaces.end() || it->second.stamp < lru->second.stamp) lru = it;
    }
    if (kept >= kMaxWorkspacesPerDevice && lru != g_workspaces.end()) {
      free_workspace(dev, lru->second);
      g_workspaces.erase(lru);
    }
  }
  Workspace& w = g_workspaces[key];
  if (!w.last_use && cudaEventCreateWithFlags(&w.last_use, cudaEventDisableTiming) != cudaSuccess) {
    cudaGetLastError();
    w.last_use = nullptr;
    return MHR_ERR_CUDA;
  }
  if (w.bytes < bytes) {
    if (w.ptr) {
      cudaEventSynchronize(w.last_use);  // the previous calls' kernels have read it
      cudaFree(w.ptr);
      w.ptr = nullptr;
      w.bytes = 0;
    }
    const size_t rounded = (bytes + kGrain - 1) & ~(kGrain - 1);
    if (cudaMalloc(&w.ptr, rounded) != cudaSuccess) {
      cudaGetLastError();
      w.ptr = nullptr;
      return MHR_ERR_CUDA;
    }
    w.bytes = rounded;
  } else if (cudaStreamWaitEvent(s, w.last_use, 0) != cudaSuccess) {
    cudaGetLastError();
    return MHR_ERR_CUDA;
  }
  w.stamp = ++g_workspace_clock;
  *out = w.ptr;
  *ws_out = &w;
  return MHR_OK;
}

// Records the end of this call's use of the workspace on its stream.
void workspace_used(Workspace* w, cudaStream_t s) {
  if (w && w->last_use) cudaEventRecord(w->last_use, s);
}

DeviceCtl make_ctl(const DeviceState& st) {
  DeviceCtl c;
  c.status = st.status;
  c.wait_limit_ns = g_wait_limit_ns;
  c.inject_stall = g_inject_stall;
  c.sm_count = st.sm_count;
  c.pair_mode = g_pair_mode;
  c.raster_group = g_raster_group;
  c.split_mode = g_split_mode;
  c.pair_tile_n = g_pair_tile_n;
  c.single_tile_n = g_single_tile_n;
  return c;
}

int from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return MHR_OK;
  cudaGetLastError();  // clear the sticky-free launch error so later calls start clean
  return MHR_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

}  // namespace

CUresult encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                        uint64_t inner, uint64_t outer, uint64_t row_pitch_bytes,
                        uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return CUDA_ERROR_NOT_FOUND;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_pitch_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

namespace {
char g_last_kernel[160] = "none";
std::mutex g_last_kernel_mu;
std::atomic<int> g_call_launches{0};
}  // namespace

void begin_call() { g_call_launches.store(0); }

void note_launch() { g_call_launches.fetch_add(1); }

void note_main_kernel(const char* name, int grid, int tiles) {
  note_launch();
  if (g_events_armed) cudaEventRecord(g_main_start, g_events_stream);
  std::lock_guard<std::mutex> g(g_last_kernel_mu);
  snprintf(g_last_kernel, sizeof(g_last_kernel), "%s grid=%d tiles=%d", name, grid, tiles);
}

const char* last_main_kernel() { return g_last_kernel; }

int check_gemm_args(const void* A, const void* B, const void* C, int64_t M, int64_t N, int64_t K,
                    int64_t lda, int64_t ldb, int64_t ldc, int64_t esz_ab, bool* noop) {
  return validate(A, B, C, M, N, K, lda, ldb, ldc, esz_ab, noop);
}

std::mutex& library_mutex() { return g_mu; }

int device_ctl_locked(DeviceCtl* ctl, int* dev) {
  DeviceState* st;
  const int rc = device_state(&st, dev);
  if (rc == MHR_OK) *ctl = make_ctl(*st);
  return rc;
}

void main_events_arm(cudaStream_t s) {
  if (g_main_start && g_main_stop) {
    g_events_stream = s;
    g_events_armed = true;
  }
}

void main_events_disarm() {
  if (g_events_armed) cudaEventRecord(g_main_stop, g_events_stream);
  g_events_armed = false;
}

}  // namespace mhr

using namespace mhr;

MHR_API int gemm_f32(const float* A, const float* B, float* C, int64_t M, int64_t N, int64_t K,
                     int64_t lda, int64_t ldb, int64_t ldc, void* stream) {
  bool noop;
  int rc = validate(A, B, C, M, N, K, lda, ldb, ldc, 4, &noop);
  if (rc != MHR_OK || noop) return rc;
  begin_call();
  std::lock_guard<std::mutex> g(g_mu);
  DeviceState* st;
  if ((rc = device_state(&st, nullptr)) != MHR_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K == 0) return from_cuda(launch_zero_fill(C, M, N, ldc, s));
  MainKernelEvents ev(s);
  return from_cuda(launch_simt_f32(A, B, C, M, N, K, lda, ldb, ldc, g_simt_wide_mode, s));
}

MHR_API int gemm_f32_ladder(int rung, const float* A, const float* B, float* C, int64_t M,
                            int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                            void* stream) {
  if (rung < 0 || rung > 2) return MHR_ERR_INVALID_ARG;
  bool noop;
  int rc = validate(A, B, C, M, N, K, lda, ldb, ldc, 4, &noop);
  if (rc != MHR_OK || noop) return rc;
  begin_call();
  const int64_t T = rung == 2 ? 32 : 16;
  if ((M + T - 1) / T > 65535) return MHR_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> g(g_mu);
  DeviceState* st;
  if ((rc = device_state(&st, nullptr)) != MHR_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K == 0) return from_cuda(launch_zero_fill(C, M, N, ldc, s));
  MainKernelEvents ev(s);
  return from_cuda(launch_ladder(rung, A, B, C, M, N, K, lda, ldb, ldc, s));
}

MHR_API int gemm_f32_3xtf32(const float* A, const float* B, float* C, int64_t M, int64_t N,
                            int64_t K, int64_t lda, int64_t ldb, int64_t ldc, void* stream) {
  bool noop;
  int rc = validate(A, B, C, M, N, K, lda, ldb, ldc, 4, &noop);
  if (rc != MHR_OK || noop) return rc;
  begin_call();
  std::lock_guard<std::mutex> g(g_mu);
  DeviceState* st;
  int dev;
  if ((rc = device_state(&st, &dev)) != MHR_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K == 0) return from_cuda(launch_zero_fill(C, M, N, ldc, s));
  const bool c_tma = c_tma_eligible(C, N, ldc);
  const DeviceCtl ctl = make_ctl(*st);
  // Split operands: a_big, a_small (M x Kp), bt_big, bt_small (N x Kp), in
  // the workspace.  Without one (split mode 2, or no memory for it) the
  // CTA-pair kernel splits on chip.
  const int64_t Kp = round_up(K, 4);
  size_t a_bytes, b_bytes, ws_bytes;
  const bool fits = !__builtin_mul_overflow(static_cast<size_t>(M), static_cast<size_t>(Kp) * 4,
                                            &a_bytes) &&
                    !__builtin_mul_overflow(static_cast<size_t>(N), static_cast<size_t>(Kp) * 4,
                                            &b_bytes) &&
                    !__builtin_add_overflow(a_bytes, b_bytes, &ws_bytes) &&
                    !__builtin_mul_overflow(ws_bytes, size_t{2}, &ws_bytes);
  // Small problems (or the test hooks' choice): one launch of the single-CTA
  // kernel with the split inside.
  if (small_one_launch_chosen(A, lda, M, N, K, ctl)) {
    MainKernelEvents ev(s);
    return from_cuda(launch_tc_3xtf32_small(A, B, C, M, N, K, lda, ldb, ldc, c_tma, ctl, s));
  }
  void* ws = nullptr;
  Workspace* wsd = nullptr;
  if (ctl.split_mode == 2 ||
      (ctl.split_mode == 0 && (!fits || workspace(dev, s, ws_bytes, &ws, &wsd) != MHR_OK))) {
    MainKernelEvents ev(s);
    return from_cuda(launch_tc_3xtf32_split(A, B, C, M, N, K, lda, ldb, ldc, c_tma, ctl, s));
  }
  if (!fits) return MHR_ERR_CUDA;
  if (!ws && (rc = workspace(dev, s, ws_bytes, &ws, &wsd)) != MHR_OK) return rc;
  float* a_big = static_cast<float*>(ws);
  float* a_small = a_big + M * Kp;
  float* bt_big = a_small + M * Kp;
  float* bt_small = bt_big + N * Kp;
  // A itself serves as A_big when TMA can read it (the tensor core truncates
  // it to tf32, which is the split's big part); then only A_small is written.
  const bool a_raw = a_serves_as_big(A, lda);
  cudaError_t e = launch_split_tf32(A, B, M, N, K, lda, ldb, Kp, a_raw ? nullptr : a_big, a_small,
                                    bt_big, bt_small, s);
  if (e == cudaSuccess && g_zero_a_small)  // test hook: the tensor core sees A alone
    e = cudaMemsetAsync(a_small, 0, static_cast<size_t>(M) * Kp * 4, s);
  if (e == cudaSuccess) {
    MainKernelEvents ev(s);
    e = launch_tc_3xtf32(a_raw ? A : a_big, a_raw ? lda : Kp, a_small, bt_big, bt_small, C, M, N,
                         K, Kp, ldc, c_tma, ctl, s);
  }
  workspace_used(wsd, s);
  return from_cuda(e);
}

MHR_API int gemm_bf16_f32acc(const uint16_t* A, const uint16_t* B, float* C, int64_t M, int64_t N,
                             int64_t K, int64_t lda, int64_t ldb, int64_t ldc, void* stream) {
  bool noop;
  int rc = validate(A, B, C, M, N, K, lda, ldb, ldc, 2, &noop);
  if (rc != MHR_OK || noop) return rc;
  begin_call();
  std::lock_guard<std::mutex> g(g_mu);
  DeviceState* st;
  int dev;
  if ((rc = device_state(&st, &dev)) != MHR_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K == 0) return from_cuda(launch_zero_fill(C, M, N, ldc, s));
  Workspace* wsd = nullptr;
  const bool a_ok = aligned16(A) && (lda % 8) == 0;
  const bool b_ok = aligned16(B) && (ldb % 8) == 0;
  if (!a_ok || !b_ok) {
    // TMA needs 16-byte aligned rows: repack the offending operand(s).
    const int64_t lda_p = round_up(K, 8), ldb_p = round_up(N, 8);
    const size_t a_bytes = a_ok ? 0 : static_cast<size_t>(M) * lda_p * 2;
    const size_t b_bytes = b_ok ? 0 : static_cast<size_t>(K) * ldb_p * 2;
    size_t ws_bytes;  // each part is below 2^63 (validated extents); their sum may not be
    if (__builtin_add_overflow(static_cast<size_t>(round_up(a_bytes, 256)), b_bytes, &ws_bytes))
      return MHR_ERR_CUDA;
    void* ws;
    if ((rc = workspace(dev, s, ws_bytes, &ws, &wsd)) != MHR_OK) return rc;
    uint16_t* pa = static_cast<uint16_t*>(ws);
    uint16_t* pb = reinterpret_cast<uint16_t*>(static_cast<char*>(ws) + round_up(a_bytes, 256));
    cudaError_t e;
    if (!a_ok) {
      if ((e = launch_pack_u16(A, M, K, lda, pa, lda_p, s)) != cudaSuccess) {
        workspace_used(wsd, s);
        return from_cuda(e);
      }
      A = pa;
      lda = lda_p;
    }
    if (!b_ok) {
      if ((e = launch_pack_u16(B, K, N, ldb, pb, ldb_p, s)) != cudaSuccess) {
        workspace_used(wsd, s);
        return from_cuda(e);
      }
      B = pb;
      ldb = ldb_p;
    }
  }
  const bool c_tma = c_tma_eligible(C, N, ldc);
  cudaError_t e;
  {
    MainKernelEvents ev(s);
    e = launch_tc_bf16(A, B, C, M, N, K, lda, ldb, ldc, c_tma, !a_ok || !b_ok, make_ctl(*st), s);
  }
  workspace_used(wsd, s);
  return from_cuda(e);
}

MHR_API int gemm_check(void* stream) {
  std::lock_guard<std::mutex> g(g_mu);
  DeviceState* st;
  int rc;
  if ((rc = device_state(&st, nullptr)) != MHR_OK) return rc;
  // Take and clear the status word in one atomic step, in stream order, then
  // wait for this stream alone.
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t bits = 0;
  take_status_kernel<<<1, 1, 0, s>>>(st->status, st->taken);
  if (cudaGetLastError() != cudaSuccess ||
      cudaMemcpyAsync(&bits, st->taken, sizeof(bits), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return MHR_ERR_CUDA;
  }
  return bits ? MHR_ERR_TIMEOUT : MHR_OK;
}

MHR_API const char* gemm_status_string(int status) {
  switch (status) {
    case MHR_OK: return "MHR_OK";
    case MHR_ERR_INVALID_ARG: return "MHR_ERR_INVALID_ARG: invalid argument";
    case MHR_ERR_UNSUPPORTED: return "MHR_ERR_UNSUPPORTED: device is not sm_103 (GB300)";
    case MHR_ERR_CUDA: return "MHR_ERR_CUDA: a CUDA call failed";
    case MHR_ERR_TIMEOUT: return "MHR_ERR_TIMEOUT: a device-side bounded wait ran out";
    default: return "unknown mhr_status";
  }
}

MHR_API void gemm_release(void) {
  std::lock_guard<std::mutex> g(g_mu);
  for (auto& kv : g_workspaces) free_workspace(kv.first.first, kv.second);
  g_workspaces.clear();
}

MHR_API int gemm_version(void) { return kVersion; }

MHR_API uint64_t gemm_testing_set_wait_limit_ns(uint64_t limit_ns) {
  std::lock_guard<std::mutex> g(g_mu);
  const uint64_t old = g_wait_limit_ns;
  g_wait_limit_ns = limit_ns < 1000000ull ? 1000000ull : limit_ns;
  return old;
}

MHR_API int gemm_testing_set_inject_stall(int enable) {
  std::lock_guard<std::mutex> g(g_mu);
  const int old = g_inject_stall;
  g_inject_stall = enable ? 1 : 0;
  return old;
}

MHR_API const char* gemm_testing_last_main_kernel(void) {
  std::lock_guard<std::mutex> g(g_last_kernel_mu);
  return last_main_kernel();
}

MHR_API int gemm_testing_set_raster_group(int tile_rows) {
  std::lock_guard<std::mutex> g(g_mu);
  const int old = g_raster_group;
  g_raster_group = tile_rows > 0 ? tile_rows : 0;
  return old;
}

MHR_API int gemm_testing_set_cta_pair_mode(int mode) {
  std::lock_guard<std::mutex> g(g_mu);
  const int old = g_pair_mode;
  g_pair_mode = (mode == 1 || mode == 2) ? mode : 0;
  return old;
}

MHR_API int gemm_testing_last_launches(void) { return g_call_launches.load(); }

MHR_API uint64_t gemm_testing_set_workspace_limit(uint64_t bytes) {
  std::lock_guard<std::mutex> g(g_mu);
  const uint64_t old = g_workspace_limit;
  g_workspace_limit = bytes;
  return old;
}

MHR_API int gemm_testing_set_pair_tile_n(int columns) {
  std::lock_guard<std::mutex> g(g_mu);
  const int old = g_pair_tile_n;
  g_pair_tile_n = (columns >= 128 && columns <= 256 && columns % 16 == 0) ? columns : 0;
  return old;
}

MHR_API int gemm_testing_set_single_tile_n(int columns) {
  std::lock_guard<std::mutex> g(g_mu);
  const int old = g_single_tile_n;
  g_single_tile_n =
      (columns == 32 || columns == 64 || columns == 96 || columns == 128 || columns == 256)
          ? columns
          : 0;
  return old;
}

MHR_API int gemm_testing_set_simt_wide_mode(int mode) {
  std::lock_guard<std::mutex> g(g_mu);
  const int old = g_simt_wide_mode;
  g_simt_wide_mode = (mode == 1 || mode == 2) ? mode : 0;
  return old;
}

MHR_API int gemm_testing_plan_simt_wide(int64_t M, int64_t N, int64_t K, int sms) {
  return simt_wide_plan(M, N, K, sms, 0);
}

MHR_API int gemm_testing_plan_single_tile_n(int64_t M, int64_t N, int64_t K, int sms, int c_tma) {
  return tc::plan_single_tile_n(M, N, K, sms, c_tma != 0);
}

MHR_API int gemm_testing_plan_pair_tile_n(int64_t M, int64_t N, int64_t K, int clusters,
                                          int c_tma) {
  return tc::plan_pair_tile_n(M, N, K, clusters, c_tma != 0);
}

MHR_API int gemm_testing_set_zero_a_small(int enable) {
  std::lock_guard<std::mutex> g(g_mu);
  const int old = g_zero_a_small;
  g_zero_a_small = enable ? 1 : 0;
  return old;
}

MHR_API int gemm_testing_set_split_mode(int mode) {
  std::lock_guard<std::mutex> g(g_mu);
  const int old = g_split_mode;
  g_split_mode = (mode == 1 || mode == 2) ? mode : 0;
  return old;
}

MHR_API void gemm_testing_set_main_kernel_events(void* start, void* stop) {
  std::lock_guard<std::mutex> g(g_mu);
  g_main_start = static_cast<cudaEvent_t>(start);
  g_main_stop = static_cast<cudaEvent_t>(stop);
}

MHR_API int64_t gemm_testing_peek_status(void* stream) {
  std::lock_guard<std::mutex> g(g_mu);
  DeviceState* st;
  if (device_state(&st, nullptr) != MHR_OK) return -1;
  uint32_t bits = 0;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess ||
      cudaMemcpy(&bits, st->status, sizeof(bits), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  return bits;
}
