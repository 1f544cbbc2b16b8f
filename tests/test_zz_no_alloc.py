"""gemm_f32_3xtf32_noalloc: the 3xTF32 product without device allocation.

Some callers cannot let a library call allocate device memory: programs whose
HBM belongs to their own pool allocator (an outside cudaMalloc may fail or
fragment the pool), latency-critical loops (cudaMalloc and cudaFree
synchronise the whole device), and programs in which only one owner thread may
allocate. This entry point keeps its split operands in a 64 MiB static device
array instead of a cudaMalloc'd workspace.

The tests call it through the C ABI and compare it with the allocating entry
point, gemm_f32_3xtf32, which runs the same kernels in the same order -- so
the two must agree bit for bit -- and with the CPU oracle. Two calls run back
to back: a small problem that both entry points run as one launch with the
split inside (no scratch at all), then one that splits into the scratch.
The limit is exercised at its exact edge (M = N = K = 2048 fills the array to
its last byte), with an unaligned A (which makes the split write A's big part
too), and one row beyond it on real buffers of that size, where the call must
be rejected before any kernel is enqueued.

This file is collected last and passes both alone in a fresh process and after
the rest of the suite.
"""
import numpy as np
import pytest

import oracle
import seeded_inputs as si
from parity_util import TOL, normalised_error, sample_indices

pytestmark = pytest.mark.gpu

# 8 * Kp * (M + N) bytes of split operands must fit in the 64 MiB array.
SCRATCH_BYTES = 64 << 20


def _call(mhr, name, a, b, c, M, N, K, lda, ldb, ldc):
    return getattr(mhr, name)(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K, lda, ldb, ldc,
                              None)


def _both(mhr, a, b, M, N, K, lda, ldb):
    """C from the allocating entry point and from the no-alloc one, in that
    order, on the same device operands (C starts as NaN in both)."""
    import torch

    out = []
    for name in ("gemm_f32_3xtf32", "gemm_f32_3xtf32_noalloc"):
        c = torch.full((M, N), float("nan"), device="cuda")
        rc = _call(mhr, name, a, b, c, M, N, K, lda, ldb, N)
        assert rc == mhr.MHR_OK, (name, mhr.gemm_status_string(rc))
        assert mhr.gemm_check(None) == mhr.MHR_OK
        out.append(c.cpu().numpy())
    return out


def _assert_bitwise(new, ref):
    assert np.all(np.isfinite(new)), "an entry of C was not written"
    mismatch = np.count_nonzero(new.view(np.uint32) != ref.view(np.uint32))
    assert mismatch == 0, f"{mismatch} entries differ from gemm_f32_3xtf32 (same kernels)"


def test_noalloc_two_calls_match_allocating_entry_point_and_oracle(mhr):
    import torch

    # two different problems back to back, the second larger than the first
    for M, N, K, seed in [(300, 520, 200, 7101), (1000, 1200, 700, 7103)]:
        A = si.matrix(M, K, seed, "normal")
        B = si.matrix(K, N, seed + 1, "normal")
        a, b = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
        ref, new = _both(mhr, a, b, M, N, K, K, N)
        _assert_bitwise(new, ref)
        Cref, S = oracle.gemm(A, B, with_abs=True)
        assert normalised_error(new, Cref, S) <= TOL["3xtf32"]


def _sampled_error(C, A, B, M, N, K, lda, seed):
    r, c = sample_indices(M, N, seed, n_random=4096, rows=(0, M - 1), cols=(0, N - 1))
    ref, S = oracle.gemm_entries(A, B, r, c, M, N, K, lda=lda)
    return normalised_error(C[r, c], ref, S)


def test_noalloc_at_the_limit_and_one_row_beyond(mhr):
    """M = N = K = 2048 uses the scratch to its last byte and must run; the
    same problem with one more row of A and C, on real buffers that hold it,
    must be rejected with MHR_ERR_INVALID_ARG before any kernel is enqueued."""
    import torch

    M = N = K = 2048
    assert 8 * K * (M + N) == SCRATCH_BYTES
    A = si.matrix(M + 1, K, 7201, "uniform")  # one spare row for the call beyond the limit
    B = si.matrix(K, N, 7202, "uniform")
    a, b = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    ref, new = _both(mhr, a, b, M, N, K, K, N)
    _assert_bitwise(new, ref)
    assert _sampled_error(new, A, B, M, N, K, K, 7203) <= TOL["3xtf32"]

    c = torch.full((M + 1, N), float("nan"), device="cuda")
    rc = _call(mhr, "gemm_f32_3xtf32_noalloc", a, b, c, M + 1, N, K, K, N, N)
    assert rc == mhr.MHR_ERR_INVALID_ARG
    assert mhr.gemm_testing_last_launches() == 0, "a rejected call enqueued kernels"
    torch.cuda.synchronize()
    assert torch.isnan(c).all().item(), "a rejected call wrote C"
    # the same buffers are valid arguments: the allocating entry point takes them
    rc = _call(mhr, "gemm_f32_3xtf32", a, b, c, M + 1, N, K, K, N, N)
    assert rc == mhr.MHR_OK
    assert mhr.gemm_check(None) == mhr.MHR_OK


def test_noalloc_unaligned_a_near_the_limit(mhr):
    """A one float off 16-byte alignment cannot serve as its own big part, so
    the split writes A_big into the scratch as well: with K = 2047 (pitch 2048)
    the four parts again fill the array exactly."""
    import torch

    M = N = 2048
    K = 2047
    Kp = 2048
    assert 8 * Kp * (M + N) == SCRATCH_BYTES
    A = si.matrix(M, K, 7301, "normal")
    B = si.matrix(K, N, 7302, "normal")
    buf = torch.empty(M * K + 1, device="cuda")
    buf[1:].copy_(torch.from_numpy(A).reshape(-1).cuda())
    a = buf[1:]
    assert a.data_ptr() % 16 != 0
    b = torch.from_numpy(B).cuda()
    ref, new = _both(mhr, a, b, M, N, K, K, N)
    _assert_bitwise(new, ref)
    assert _sampled_error(new, A, B, M, N, K, K, 7303) <= TOL["3xtf32"]
