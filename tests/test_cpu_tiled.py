"""The cache-blocked CPU comparator against the oracle (CPU only)."""
import numpy as np
import pytest

import cpu_tiled
import oracle
import seeded_inputs as si


@pytest.mark.parametrize("shape", [(1, 1, 1), (7, 5, 3), (64, 256, 256), (65, 257, 513),
                                   (130, 300, 1000)], ids=lambda s: "x".join(map(str, s)))
def test_matches_oracle(shape):
    M, N, K = shape
    A = si.matrix(M, K, 71, "normal")
    B = si.matrix(K, N, 72, "normal")
    C = cpu_tiled.gemm(A, B)
    ref, S = oracle.gemm(A, B, with_abs=True)
    assert np.max(np.abs(C.astype(np.float64) - ref) / S) <= 1e-5
    Ai = si.matrix(M, K, 73, "int")
    Bi = si.matrix(K, N, 74, "int")
    assert np.array_equal(cpu_tiled.gemm(Ai, Bi), oracle.gemm(Ai, Bi))


def test_k_zero_and_threads():
    C = cpu_tiled.gemm(np.zeros((3, 0), np.float32), np.zeros((0, 4), np.float32))
    assert C.shape == (3, 4) and np.all(C == 0)
    A = si.matrix(100, 300, 75, "normal")
    B = si.matrix(300, 90, 76, "normal")
    assert np.array_equal(cpu_tiled.gemm(A, B, nthreads=1), cpu_tiled.gemm(A, B, nthreads=3))
