"""Pins of the CPU oracle to facts fixed outside it (CPU only).

The oracle computes C[i][j] = sum_k A[i][k] B[k][j] in fp64 and rounds once to
fp32. Each test below checks it against something that does not go through
its code: the pages' block decomposition, closed forms, special cases, and
brute force in exact rational arithmetic. Together they catch a dropped term,
a wrong sign or index, a transposed operand, a wrong leading dimension,
accumulation in fp32 instead of fp64, and a missing final rounding.
"""
from fractions import Fraction
import struct

import numpy as np
import pytest

import seeded_inputs as si


def f32_rne(q: Fraction) -> float:
    """Exact rational -> nearest fp32 (ties to even), as a Python float."""
    if q == 0:
        return 0.0
    sign = -1.0 if q < 0 else 1.0
    q = abs(q)
    e = q.numerator.bit_length() - q.denominator.bit_length()
    if Fraction(2) ** e > q:
        e -= 1
    ulp_e = max(e - 23, -149)
    scaled = q / (Fraction(2) ** ulp_e)
    n = scaled.numerator // scaled.denominator
    rem = scaled - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    val = sign * n * 2.0 ** ulp_e
    assert abs(val) < 3.5e38
    return val


def exact_product(A, B):
    M, K = A.shape
    _, N = B.shape
    C = np.zeros((M, N), dtype=np.float32)
    for i in range(M):
        for j in range(N):
            s = sum((Fraction(float(A[i, k])) * Fraction(float(B[k, j])) for k in range(K)),
                    Fraction(0))
            C[i, j] = f32_rne(s)
    return C


def bits(x):
    return np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)


def test_f32_rne_helper():
    # the helper itself: exact values, a tie to even, subnormals
    assert f32_rne(Fraction(1, 3)) == struct.unpack("f", struct.pack("f", 1 / 3))[0]
    one_plus_half_ulp = Fraction(1) + Fraction(1, 2 ** 24)
    assert f32_rne(one_plus_half_ulp) == 1.0  # tie -> even
    assert f32_rne(Fraction(1) + Fraction(3, 2 ** 25)) == 1.0 + 2.0 ** -23
    assert f32_rne(Fraction(1, 2 ** 149)) == 2.0 ** -149


def test_block_decomposition_n8_tile4(oracle_lib):
    """ijyty.com page, step ③ and its diagram: with N=8 and TILE=4, each 4x4
    block of C is the sum over the two K tiles, C00 = A00*B00 + A01*B10, and
    likewise for C01, C10, C11. Integer inputs make every sum exact."""
    A = si.matrix(8, 8, 11, "int")
    B = si.matrix(8, 8, 12, "int")
    C = oracle_lib.gemm(A, B)
    T = 4
    for bi in range(2):
        for bj in range(2):
            parts = [oracle_lib.gemm(np.ascontiguousarray(A[bi * T:(bi + 1) * T, t * T:(t + 1) * T]),
                                     np.ascontiguousarray(B[t * T:(t + 1) * T, bj * T:(bj + 1) * T]))
                     for t in range(2)]
            assert np.array_equal(C[bi * T:(bi + 1) * T, bj * T:(bj + 1) * T], parts[0] + parts[1])
    # and the blocks really depend on both K tiles (not a vacuous identity)
    assert not np.array_equal(C[:4, :4], parts[0] * 0 + oracle_lib.gemm(
        np.ascontiguousarray(A[:4, :4]), np.ascontiguousarray(B[:4, :4])))


def test_identity_left_and_right(oracle_lib):
    for M, N in [(1, 1), (5, 3), (17, 40)]:
        B = si.matrix(M, N, 21, "normal")
        assert np.array_equal(bits(oracle_lib.gemm(np.eye(M, dtype=np.float32), B)), bits(B))
        A = si.matrix(M, N, 22, "uniform")
        assert np.array_equal(bits(oracle_lib.gemm(A, np.eye(N, dtype=np.float32))), bits(A))


def test_all_ones_gives_k(oracle_lib):
    for M, N, K in [(1, 1, 1), (3, 5, 7), (2, 3, 1000), (2, 2, 8192)]:
        C = oracle_lib.gemm(np.ones((M, K), np.float32), np.ones((K, N), np.float32))
        assert np.all(C == K)


def test_k_zero_is_zero(oracle_lib):
    C = oracle_lib.gemm(np.zeros((4, 1), np.float32), np.zeros((1, 3), np.float32), M=4, N=3, K=0)
    assert np.all(C == 0) and C.shape == (4, 3)


@pytest.mark.parametrize("dist", ["uniform", "normal"])
def test_brute_force_tiny(oracle_lib, dist):
    """Exact rational sum of the products, rounded once to fp32."""
    rng = np.random.default_rng(5)
    seed = 100
    for _ in range(12):
        M, N, K = (int(v) for v in rng.integers(1, 7, size=3))
        A = si.matrix(M, K, seed, dist)
        B = si.matrix(K, N, seed + 1, dist)
        seed += 2
        assert np.array_equal(bits(oracle_lib.gemm(A, B)), bits(exact_product(A, B)))


def test_brute_force_padded_leading_dims(oracle_lib):
    """Leading dimensions larger than the logical width, pads full of NaN: a
    stride mistake reads a NaN or a wrong element and fails the exact match."""
    A = si.matrix(5, 6, 31, "normal")
    B = si.matrix(6, 4, 32, "normal")
    C = oracle_lib.gemm(si.padded(A, 9), si.padded(B, 7), M=5, N=4, K=6, lda=9, ldb=7)
    assert np.array_equal(bits(C), bits(exact_product(A, B)))


def test_not_transposed(oracle_lib):
    """A non-symmetric case whose transposed variants differ."""
    A = np.array([[1, 2], [3, 4]], np.float32)
    B = np.array([[5, 6], [7, 8]], np.float32)
    assert np.array_equal(oracle_lib.gemm(A, B), np.array([[19, 22], [43, 50]], np.float32))


def test_fp64_accumulation(oracle_lib):
    """2^24 + 1 - 2^24: an fp32 running sum loses the 1, the fp64 sum keeps it."""
    A = np.array([[2.0 ** 24, 1.0, -(2.0 ** 24)]], np.float32)
    B = np.ones((3, 1), np.float32)
    assert oracle_lib.gemm(A, B)[0, 0] == 1.0
    # ... and the single final rounding: 1 + 2^-24 + 2^-24 is exactly 1 + 2^-23
    A = np.array([[1.0, 2.0 ** -24, 2.0 ** -24]], np.float32)
    assert oracle_lib.gemm(A, B)[0, 0] == np.float32(1.0 + 2.0 ** -23)


def test_entries_match_full(oracle_lib):
    A = si.matrix(37, 300, 41, "normal")
    B = si.matrix(300, 29, 42, "normal")
    C, S = oracle_lib.gemm(A, B, with_abs=True)
    rows = np.array([0, 5, 36, 17, 36], np.int64)
    cols = np.array([0, 28, 0, 13, 28], np.int64)
    v, s = oracle_lib.gemm_entries(A, B, rows, cols, 37, 29, 300)
    assert np.array_equal(bits(v), bits(C[rows, cols]))
    assert np.array_equal(s, S[rows, cols])
    # the scale sum_k |a||b| against exact arithmetic (one fp64 rounding per step)
    exact = sum(abs(Fraction(float(A[5, k])) * Fraction(float(B[k, 28]))) for k in range(300))
    assert s[1] == pytest.approx(float(exact), rel=1e-13)


def test_entries_brute_force(oracle_lib):
    A = si.matrix(9, 64, 51, "uniform")
    B = si.matrix(64, 11, 52, "uniform")
    rows = np.arange(9, dtype=np.int64).repeat(11)
    cols = np.tile(np.arange(11, dtype=np.int64), 9)
    v, _ = oracle_lib.gemm_entries(A, B, rows, cols, 9, 11, 64)
    assert np.array_equal(bits(v.reshape(9, 11)), bits(exact_product(A, B)))


def test_rejects_bad_arguments(oracle_lib):
    with pytest.raises(ValueError):
        oracle_lib.gemm(np.zeros((2, 3), np.float32), np.zeros((3, 2), np.float32), lda=2)
    with pytest.raises(ValueError):
        oracle_lib.gemm_entries(np.zeros((2, 3), np.float32), np.zeros((3, 2), np.float32),
                                [2], [0], 2, 2, 3)


def test_threads_do_not_change_results(oracle_lib):
    A = si.matrix(64, 200, 61, "normal")
    B = si.matrix(200, 48, 62, "normal")
    assert np.array_equal(bits(oracle_lib.gemm(A, B, nthreads=1)),
                          bits(oracle_lib.gemm(A, B, nthreads=4)))


# ---------------------------------------------------------------- invariants
# Identities of the exact product that hold bit for bit for the oracle's
# definition (each product exact in fp64, summed in ascending k, rounded once),
# checked on seeded real-valued inputs that are larger than the brute-force
# cases above. Each one fails on a plausible mistake elsewhere in the code:
# an index swap, a stride, a dropped or duplicated term, a rounding.

def test_transpose_identity(oracle_lib):
    """(A B)^T = B^T A^T: the same products summed in the same k order."""
    A = si.matrix(37, 53, 8101, "normal")
    B = si.matrix(53, 29, 8102, "normal")
    C = oracle_lib.gemm(A, B)
    Ct = oracle_lib.gemm(np.ascontiguousarray(B.T), np.ascontiguousarray(A.T))
    assert np.array_equal(bits(C.T), bits(Ct))


def test_row_and_column_permutations(oracle_lib):
    """Permuting the rows of A permutes the rows of C; permuting the columns
    of B permutes the columns of C."""
    A = si.matrix(31, 40, 8103, "uniform")
    B = si.matrix(40, 23, 8104, "uniform")
    C = oracle_lib.gemm(A, B)
    p = np.random.default_rng(1).permutation(31)
    q = np.random.default_rng(2).permutation(23)
    assert np.array_equal(bits(oracle_lib.gemm(np.ascontiguousarray(A[p]), B)), bits(C[p]))
    assert np.array_equal(bits(oracle_lib.gemm(A, np.ascontiguousarray(B[:, q]))), bits(C[:, q]))


def test_power_of_two_scaling(oracle_lib):
    """Scaling A by 2^5 and B by 2^-3 scales every product, every partial sum
    and the rounded result by exactly 2^2."""
    A = si.matrix(19, 33, 8105, "normal")
    B = si.matrix(33, 17, 8106, "normal")
    C = oracle_lib.gemm(A, B)
    C2 = oracle_lib.gemm(A * np.float32(32.0), B * np.float32(0.125))
    assert np.array_equal(bits(C2), bits(C * np.float32(4.0)))


def test_integer_linearity_and_k_split(oracle_lib):
    """On small integers every sum is exact: C(A1 + A2, B) = C(A1, B) +
    C(A2, B), and C(A, B) equals the sum of the products of any split of K
    (the block decomposition of the pages, for every cut)."""
    A1 = si.matrix(24, 50, 8107, "int")
    A2 = si.matrix(24, 50, 8108, "int")
    B = si.matrix(50, 18, 8109, "int")
    C = oracle_lib.gemm(A1 + A2, B)
    assert np.array_equal(C, oracle_lib.gemm(A1, B) + oracle_lib.gemm(A2, B))
    for cut in (1, 17, 32, 49):
        left = oracle_lib.gemm(np.ascontiguousarray(A1[:, :cut]), np.ascontiguousarray(B[:cut]))
        right = oracle_lib.gemm(np.ascontiguousarray(A1[:, cut:]), np.ascontiguousarray(B[cut:]))
        assert np.array_equal(oracle_lib.gemm(A1, B), left + right)
