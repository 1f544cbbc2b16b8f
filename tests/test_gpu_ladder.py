"""The pages' ladder kernels (naive, 16x16 tiled, 32x32 tiled) against the
oracle through the C ABI (GB300 only)."""
import numpy as np
import pytest

import oracle
from parity_util import TOL, normalised_error, sample_indices, operands

pytestmark = pytest.mark.gpu


def run_ladder(mhr, rung, A, B, ldc=None):
    import torch

    M, K = A.shape
    N = B.shape[1]
    ldc = ldc or N
    a, b = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    c = torch.full((M, ldc), -7.25, device="cuda")
    c[:, :N] = float("nan")
    rc = mhr.gemm_f32_ladder(rung, a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K, K, N, ldc,
                             None)
    assert rc == mhr.MHR_OK
    assert mhr.gemm_check(None) == mhr.MHR_OK
    out = c.cpu().numpy()
    assert np.all(out[:, N:] == np.float32(-7.25))  # padding untouched
    return np.ascontiguousarray(out[:, :N])


@pytest.mark.parametrize("rung", [0, 1, 2], ids=["naive", "tile16", "tile32"])
@pytest.mark.parametrize("shape", [(1, 1, 1), (8, 8, 8), (33, 17, 45), (100, 130, 77),
                                   (256, 256, 256), (300, 520, 200)],
                         ids=lambda s: "x".join(map(str, s)))
def test_ladder_matches_oracle(mhr, rung, shape):
    M, N, K = shape
    A, B, _, _ = operands(M, N, K, 8000 + sum(shape), "normal", "f32")
    C = run_ladder(mhr, rung, A, B, ldc=N + 3)
    Cref, S = oracle.gemm(A, B, with_abs=True)
    assert normalised_error(C, Cref, S) <= TOL["f32"]
    # integer inputs: exact
    A, B, _, _ = operands(M, N, K, 8100 + sum(shape), "int", "f32")
    assert np.array_equal(run_ladder(mhr, rung, A, B), oracle.gemm(A, B))


@pytest.mark.parametrize("rung", [0, 1, 2], ids=["naive", "tile16", "tile32"])
def test_ladder_4096_sampled(mhr, rung):
    """The pages' worked size, 4096^3 uniform[-1, 1), seeds (2001, 2002)."""
    M = N = K = 4096
    A, B, _, _ = operands(M, N, K, 2001, "uniform", "f32")
    C = run_ladder(mhr, rung, A, B)
    rows, cols = sample_indices(M, N, 2001, n_random=2048, rows=(0, M - 1), cols=(N - 1,))
    ref, S = oracle.gemm_entries(A, B, rows, cols, M, N, K)
    assert normalised_error(C[rows, cols], ref, S) <= TOL["f32"]
