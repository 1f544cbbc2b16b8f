"""Python binding of libmhr_gemm.so, the sm_103a dense GEMM library.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI (``include/mhr_gemm.h``). PyTorch is used for device
memory and streams. There is no CPU fallback: if the library is not built or
the device is not a GB300, calls raise.

Raw entry points (same names and arguments as the C ABI; pointers are ints,
``stream`` a ``cudaStream_t`` as int or None):

    gemm_f32(A, B, C, M, N, K, lda, ldb, ldc, stream) -> status
    gemm_f32_3xtf32(...)                               -> status
    gemm_bf16_f32acc(...)                              -> status
    gemm_f32_3xtf32_noalloc(...)                       -> status
    gemm_f32_ladder(rung, A, B, C, ...)                -> status
    gemm_check(stream) -> status
    gemm_status_string(status) -> str
    gemm_release()
    gemm_version() -> int

Tensor-level helper: ``matmul(a, b, path, out=None)`` for row-major CUDA
tensors (the last dimension contiguous; the leading dimension is the row
stride).
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmhr_gemm.so")

MHR_OK = 0
MHR_ERR_INVALID_ARG = 1
MHR_ERR_UNSUPPORTED = 2
MHR_ERR_CUDA = 3
MHR_ERR_TIMEOUT = 4

PATHS = ("f32", "3xtf32", "bf16")

#: every symbol the public headers declare
EXPORTS = ("gemm_f32", "gemm_f32_3xtf32", "gemm_bf16_f32acc", "gemm_f32_3xtf32_noalloc",
           "gemm_f32_ladder",
           "gemm_check",
           "gemm_status_string", "gemm_release", "gemm_version",
           "gemm_testing_set_wait_limit_ns", "gemm_testing_set_inject_stall",
           "gemm_testing_peek_status", "gemm_testing_set_main_kernel_events",
           "gemm_testing_set_cta_pair_mode", "gemm_testing_last_main_kernel",
           "gemm_testing_set_raster_group", "gemm_testing_set_split_mode",
           "gemm_testing_last_launches", "gemm_testing_set_workspace_limit",
           "gemm_testing_set_zero_a_small", "gemm_testing_set_pair_tile_n",
           "gemm_testing_plan_pair_tile_n", "gemm_testing_set_single_tile_n",
           "gemm_testing_plan_single_tile_n", "gemm_testing_set_simt_wide_mode",
           "gemm_testing_plan_simt_wide")

_lib = None


class GemmError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {gemm_status_string(status)} (status {status})")
        self.status = status


def load(path: str | None = None):
    """Load the shared library (once). Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with memory_hierarchy_reuse_gb300.build.build() "
            "(there is no fallback implementation)")
    lib = ctypes.CDLL(path)
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    for name in ("gemm_f32", "gemm_f32_3xtf32", "gemm_bf16_f32acc", "gemm_f32_3xtf32_noalloc"):
        f = getattr(lib, name)
        f.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, vp]
        f.restype = ctypes.c_int
    lib.gemm_f32_ladder.argtypes = [ctypes.c_int, vp, vp, vp, i64, i64, i64, i64, i64, i64, vp]
    lib.gemm_f32_ladder.restype = ctypes.c_int
    lib.gemm_check.argtypes = [vp]
    lib.gemm_check.restype = ctypes.c_int
    lib.gemm_status_string.argtypes = [ctypes.c_int]
    lib.gemm_status_string.restype = ctypes.c_char_p
    lib.gemm_release.argtypes = []
    lib.gemm_release.restype = None
    lib.gemm_version.argtypes = []
    lib.gemm_version.restype = ctypes.c_int
    lib.gemm_testing_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.gemm_testing_set_wait_limit_ns.restype = ctypes.c_uint64
    lib.gemm_testing_set_inject_stall.argtypes = [ctypes.c_int]
    lib.gemm_testing_set_inject_stall.restype = ctypes.c_int
    lib.gemm_testing_peek_status.argtypes = [vp]
    lib.gemm_testing_peek_status.restype = ctypes.c_int64
    lib.gemm_testing_set_raster_group.argtypes = [ctypes.c_int]
    lib.gemm_testing_set_raster_group.restype = ctypes.c_int
    lib.gemm_testing_last_main_kernel.argtypes = []
    lib.gemm_testing_last_main_kernel.restype = ctypes.c_char_p
    lib.gemm_testing_set_cta_pair_mode.argtypes = [ctypes.c_int]
    lib.gemm_testing_set_cta_pair_mode.restype = ctypes.c_int
    lib.gemm_testing_set_zero_a_small.argtypes = [ctypes.c_int]
    lib.gemm_testing_set_zero_a_small.restype = ctypes.c_int
    lib.gemm_testing_set_pair_tile_n.argtypes = [ctypes.c_int]
    lib.gemm_testing_set_pair_tile_n.restype = ctypes.c_int
    lib.gemm_testing_plan_pair_tile_n.argtypes = [i64, i64, i64, ctypes.c_int, ctypes.c_int]
    lib.gemm_testing_plan_pair_tile_n.restype = ctypes.c_int
    lib.gemm_testing_set_single_tile_n.argtypes = [ctypes.c_int]
    lib.gemm_testing_set_single_tile_n.restype = ctypes.c_int
    lib.gemm_testing_plan_single_tile_n.argtypes = [i64, i64, i64, ctypes.c_int, ctypes.c_int]
    lib.gemm_testing_plan_single_tile_n.restype = ctypes.c_int
    lib.gemm_testing_set_simt_wide_mode.argtypes = [ctypes.c_int]
    lib.gemm_testing_set_simt_wide_mode.restype = ctypes.c_int
    lib.gemm_testing_plan_simt_wide.argtypes = [i64, i64, i64, ctypes.c_int]
    lib.gemm_testing_plan_simt_wide.restype = ctypes.c_int
    lib.gemm_testing_set_split_mode.argtypes = [ctypes.c_int]
    lib.gemm_testing_set_split_mode.restype = ctypes.c_int
    lib.gemm_testing_set_workspace_limit.argtypes = [ctypes.c_uint64]
    lib.gemm_testing_set_workspace_limit.restype = ctypes.c_uint64
    lib.gemm_testing_last_launches.argtypes = []
    lib.gemm_testing_last_launches.restype = ctypes.c_int
    lib.gemm_testing_set_main_kernel_events.argtypes = [vp, vp]
    lib.gemm_testing_set_main_kernel_events.restype = None
    _lib = lib
    return lib


def gemm_f32(A, B, C, M, N, K, lda, ldb, ldc, stream=None) -> int:
    return load().gemm_f32(A, B, C, M, N, K, lda, ldb, ldc, stream)


def gemm_f32_3xtf32(A, B, C, M, N, K, lda, ldb, ldc, stream=None) -> int:
    return load().gemm_f32_3xtf32(A, B, C, M, N, K, lda, ldb, ldc, stream)


def gemm_bf16_f32acc(A, B, C, M, N, K, lda, ldb, ldc, stream=None) -> int:
    return load().gemm_bf16_f32acc(A, B, C, M, N, K, lda, ldb, ldc, stream)


def gemm_f32_3xtf32_noalloc(A, B, C, M, N, K, lda, ldb, ldc, stream=None) -> int:
    """gemm_f32_3xtf32 with its scratch in a 64 MiB static device array: no
    device allocation in the call (for callers that must not allocate)."""
    return load().gemm_f32_3xtf32_noalloc(A, B, C, M, N, K, lda, ldb, ldc, stream)


def gemm_f32_ladder(rung, A, B, C, M, N, K, lda, ldb, ldc, stream=None) -> int:
    """The pages' kernels: rung 0 naive, 1 tiled 16x16, 2 tiled 32x32."""
    return load().gemm_f32_ladder(int(rung), A, B, C, M, N, K, lda, ldb, ldc, stream)


def gemm_check(stream=None) -> int:
    return load().gemm_check(stream)


def gemm_status_string(status: int) -> str:
    return load().gemm_status_string(int(status)).decode()


def gemm_release() -> None:
    load().gemm_release()


def gemm_version() -> int:
    return load().gemm_version()


def gemm_testing_set_wait_limit_ns(limit_ns: int) -> int:
    return load().gemm_testing_set_wait_limit_ns(int(limit_ns))


def gemm_testing_set_inject_stall(enable: int) -> int:
    return load().gemm_testing_set_inject_stall(int(enable))


def gemm_testing_peek_status(stream=None) -> int:
    return load().gemm_testing_peek_status(stream)


def gemm_testing_set_raster_group(tile_rows: int) -> int:
    return load().gemm_testing_set_raster_group(int(tile_rows))


def gemm_testing_last_main_kernel() -> str:
    return load().gemm_testing_last_main_kernel().decode()


def gemm_testing_set_cta_pair_mode(mode: int) -> int:
    """0 = automatic, 1 = single-CTA tensor-core kernel, 2 = CTA-pair kernel."""
    return load().gemm_testing_set_cta_pair_mode(int(mode))


def gemm_testing_last_launches() -> int:
    """Kernels launched by the most recent gemm_* call."""
    return load().gemm_testing_last_launches()


def gemm_testing_set_workspace_limit(nbytes: int) -> int:
    """Cap the workspace (2**64 - 1 = no cap); a larger request fails like an allocation."""
    return load().gemm_testing_set_workspace_limit(int(nbytes))


def gemm_testing_set_split_mode(mode: int) -> int:
    """3xTF32 split: 0 = automatic (pre-pass; on chip without workspace), 1 = pre-pass,
    2 = inside the CTA-pair kernel."""
    return load().gemm_testing_set_split_mode(int(mode))


def gemm_testing_set_zero_a_small(enable: int) -> int:
    """Clear A's small part after the 3xTF32 split pre-pass (test hook)."""
    return load().gemm_testing_set_zero_a_small(int(enable))


def gemm_testing_set_pair_tile_n(columns: int) -> int:
    """Force the 3xTF32 CTA-pair tiles' columns (a multiple of 16 in
    [128, 256]); 0 restores the planner (test hook)."""
    return load().gemm_testing_set_pair_tile_n(int(columns))


def gemm_testing_plan_pair_tile_n(M: int, N: int, K: int, clusters: int, c_tma: bool) -> int:
    """The 3xTF32 CTA-pair tile columns the planner picks (host logic only)."""
    return load().gemm_testing_plan_pair_tile_n(M, N, K, int(clusters), int(bool(c_tma)))


def gemm_testing_set_main_kernel_events(start=None, stop=None) -> None:
    """start/stop: cudaEvent_t handles as ints (torch.cuda.Event().cuda_event) or None."""
    load().gemm_testing_set_main_kernel_events(start, stop)


_ENTRY = {"f32": "gemm_f32", "3xtf32": "gemm_f32_3xtf32", "bf16": "gemm_bf16_f32acc"}


def _rowmajor(t, name):
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D")
    if t.shape[0] > 0 and t.shape[1] > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} must be row-major (last dimension contiguous)")
    return max(t.stride(0), t.shape[1]) if t.shape[0] > 1 else t.shape[1]


def matmul(a, b, path: str = "f32", out=None, stream=None, lda=None, ldb=None, ldc=None):
    """C = a @ b through the C ABI.

    ``path``: "f32" (SIMT fp32), "3xtf32" (tensor cores, fp32-accurate) or
    "bf16" (a and b torch.bfloat16; fp32 accumulate and output). ``a``, ``b``
    and ``out`` are row-major CUDA tensors; ``out`` (fp32, M x N) is allocated
    when omitted. ``lda``/``ldb``/``ldc`` override the leading dimensions
    (e.g. for views into padded buffers). Launches on ``stream`` (default: the
    current torch stream) and returns ``out`` without synchronising.
    """
    import torch

    if path not in _ENTRY:
        raise ValueError(f"path must be one of {PATHS}")
    want = torch.bfloat16 if path == "bf16" else torch.float32
    if a.dtype != want or b.dtype != want:
        raise TypeError(f"path {path!r} takes {want} operands")
    M, K = a.shape
    K2, N = b.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=a.device)
    if out.dtype != torch.float32 or tuple(out.shape) != (M, N):
        raise TypeError("out must be float32 of shape (M, N)")
    lda = _rowmajor(a, "a") if lda is None else lda
    ldb = _rowmajor(b, "b") if ldb is None else ldb
    ldc = _rowmajor(out, "out") if ldc is None else ldc
    if stream is None:
        stream = torch.cuda.current_stream(a.device).cuda_stream
    with torch.cuda.device(a.device):
        rc = getattr(load(), _ENTRY[path])(a.data_ptr(), b.data_ptr(), out.data_ptr(),
                                           M, N, K, lda, ldb, ldc, stream)
    if rc != MHR_OK:
        raise GemmError(rc, _ENTRY[path])
    return out


# The same call under the name the C ABI's family uses: gemm(a, b, path).
gemm = matmul


def gemm_testing_set_single_tile_n(columns: int) -> int:
    """Force the single-CTA tiles' columns (3xTF32: 128, 96, 64 or 32; bf16:
    256 or 128); 0 restores the planners (test hook)."""
    return load().gemm_testing_set_single_tile_n(int(columns))


def gemm_testing_plan_single_tile_n(M: int, N: int, K: int, sms: int, c_tma: bool) -> int:
    """The 3xTF32 single-CTA tile columns the planner picks (host logic only)."""
    return load().gemm_testing_plan_single_tile_n(M, N, K, int(sms), int(bool(c_tma)))


def gemm_testing_set_simt_wide_mode(mode: int) -> int:
    """Choose gemm_f32's SIMT kernel for aligned 128 x 256 x 8 multiples: 0
    automatic, 1 the 128 x 128 kernel, 2 the 128 x 256 kernel (test hook)."""
    return load().gemm_testing_set_simt_wide_mode(int(mode))


def gemm_testing_plan_simt_wide(M: int, N: int, K: int, sms: int) -> int:
    """The automatic SIMT kernel choice: 0 128 x 128, 1 128 x 256, 2 128 x 256
    on K halves (host logic only)."""
    return load().gemm_testing_plan_simt_wide(M, N, K, int(sms))
