"""CPU oracle for C = A * B (fp64 accumulation, one rounding to fp32).

TEST INFRASTRUCTURE ONLY. The tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use it; the CUDA library and its Python binding
never import it. It shares no code with the CUDA path: its arithmetic lives in
``oracle_gemm.c`` (plain C, built with gcc, no CUDA headers).

Every function here follows the plain definition
``C[i][j] = sum_k A[i][k] * B[k][j]`` (row-major, ascending k, fp64 sum) -- the
naive dot product that the pages start from ("矩阵乘法 tiling", section 一;
"CUDA 深入浅出（二）", section "naive kernel 怎么读数据"; "CUDA 编程系列之三",
section 6). All functions are pinned by tests that do not go through this code
(``tests/test_oracle_pins.py``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle_gemm.c")
_LIB = os.path.join(_HERE, "liboracle_gemm.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle_gemm.c`` into ``liboracle_gemm.so`` (gcc, OpenMP,
    strict IEEE: no fast-math, no contraction)."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            tmp = _LIB + f".tmp{os.getpid()}"
            subprocess.check_call([
                "gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm",
            ])
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        i64, ptr = ctypes.c_int64, ctypes.c_void_p
        lib.oracle_gemm.argtypes = [ptr, ptr, ptr, i64, i64, i64, i64, i64, i64, ptr, ctypes.c_int]
        lib.oracle_gemm.restype = ctypes.c_int
        lib.oracle_gemm_entries.argtypes = [ptr, ptr, i64, i64, i64, i64, i64, ptr, ptr, i64,
                                            ptr, ptr, ctypes.c_int]
        lib.oracle_gemm_entries.restype = ctypes.c_int
        lib.oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _operand(x, rows, cols, ld):
    """A float32 row-major buffer holding a rows x cols matrix with leading
    dimension ld (ld defaults to the buffer's row length)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim != 2:
        raise ValueError("operands are 2-D buffers (rows x ld)")
    if ld is None:
        ld = x.shape[1]
    if x.shape[1] != ld or ld < cols or x.shape[0] < rows:
        raise ValueError("operand buffer does not hold (rows, cols, ld)")
    return x, ld


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def gemm(A, B, M=None, N=None, K=None, lda=None, ldb=None, with_abs=False, nthreads=0):
    """Full product of row-major fp32 operands.

    ``A`` holds an M x K matrix (leading dimension ``lda``), ``B`` a K x N
    matrix (``ldb``); omitted sizes come from the buffers' shapes. Returns C
    (M x N float32) and, with ``with_abs``, also S[i, j] = sum_k |A_ik| |B_kj|
    (float64).
    """
    M = A.shape[0] if M is None else M
    K = (A.shape[1] if lda is None else lda) if K is None else K
    N = (B.shape[1] if ldb is None else ldb) if N is None else N
    A, lda = _operand(A, M, K, lda)
    B, ldb = _operand(B, K, N, ldb)
    C = np.zeros((M, N), dtype=np.float32)
    S = np.zeros((M, N), dtype=np.float64) if with_abs else None
    rc = _load().oracle_gemm(_ptr(A), _ptr(B), _ptr(C), M, N, K, lda, ldb, max(N, 1),
                             _ptr(S), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_gemm rejected its arguments (rc={rc})")
    return (C, S) if with_abs else C


def gemm_entries(A, B, rows, cols, M, N, K, lda=None, ldb=None, nthreads=0):
    """Entries (rows[t], cols[t]) of A * B: returns (values fp32, abs-sums fp64)."""
    A, lda = _operand(A, M, K, lda)
    B, ldb = _operand(B, K, N, ldb)
    r = np.ascontiguousarray(rows, dtype=np.int64)
    c = np.ascontiguousarray(cols, dtype=np.int64)
    if r.shape != c.shape:
        raise ValueError("rows and cols differ in length")
    out = np.zeros(r.size, dtype=np.float32)
    ab = np.zeros(r.size, dtype=np.float64)
    rc = _load().oracle_gemm_entries(_ptr(A), _ptr(B), M, N, K, lda, ldb, _ptr(r), _ptr(c),
                                     r.size, _ptr(out), _ptr(ab), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_gemm_entries rejected its arguments (rc={rc})")
    return out, ab
