"""Cache-blocked CPU GEMM (fp32), the pages' tiling applied to CPU caches.

A host comparator for the benchmark, beside the plain oracle: same seeded
inputs, blocked for L1/L2 instead of shared memory, OpenMP over output
blocks. Built with gcc -O3 (portable flags only). It shares no code with the
oracle or with the CUDA library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cpu_tiled_gemm.c")
_LIB = os.path.join(_HERE, "libcpu_tiled_gemm.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            tmp = _LIB + f".tmp{os.getpid()}"
            subprocess.check_call(["gcc", "-O3", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                                   _SRC, "-o", tmp])
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        i64, vp = ctypes.c_int64, ctypes.c_void_p
        lib.cpu_tiled_gemm.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, ctypes.c_int]
        lib.cpu_tiled_gemm.restype = ctypes.c_int
        lib.cpu_tiled_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().cpu_tiled_max_threads())


def gemm(A: np.ndarray, B: np.ndarray, nthreads: int = 0) -> np.ndarray:
    """C = A @ B for C-contiguous float32 matrices."""
    A = np.ascontiguousarray(A, dtype=np.float32)
    B = np.ascontiguousarray(B, dtype=np.float32)
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    C = np.empty((M, N), dtype=np.float32)
    p = lambda x: x.ctypes.data_as(ctypes.c_void_p)  # noqa: E731
    rc = _load().cpu_tiled_gemm(p(A), p(B), p(C), M, N, K, K, N, N, int(nthreads))
    if rc != 0:
        raise ValueError("cpu_tiled_gemm rejected its arguments")
    return C
