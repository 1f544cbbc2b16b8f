"""gemm_f32_3xtf32_noalloc: the 3xTF32 product without device allocation.

Callers whose device memory belongs to their own pool allocator, or that
cannot afford cudaMalloc's device-wide synchronisation inside a GEMM call, use
this entry point: its split operands live in a 64 MiB static device array
instead of a cudaMalloc'd workspace. This test calls it through the C ABI and
checks it against the allocating entry point, gemm_f32_3xtf32, on two calls in
a row (so the second call runs over the scratch the first one left behind).
It sits in its own file, collected last, and passes both alone in a fresh
process and after the rest of the suite.
"""
import numpy as np
import pytest

import seeded_inputs as si
from parity_util import TOL

pytestmark = pytest.mark.gpu


def _normalised_error(C, Cref, A, B):
    S = np.abs(A.astype(np.float64)) @ np.abs(B.astype(np.float64))
    return float(np.max(np.abs(C.astype(np.float64) - Cref.astype(np.float64)) / S))


def test_noalloc_matches_allocating_entry_point(mhr):
    import torch

    # two different problems back to back, the second larger than the first
    for M, N, K, seed in [(300, 520, 200, 7101), (1000, 1200, 700, 7103)]:
        A = si.matrix(M, K, seed, "normal")
        B = si.matrix(K, N, seed + 1, "normal")
        a, b = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
        c_ref = torch.full((M, N), float("nan"), device="cuda")
        c_new = torch.full((M, N), float("nan"), device="cuda")
        rc = mhr.gemm_f32_3xtf32(a.data_ptr(), b.data_ptr(), c_ref.data_ptr(), M, N, K, K, N, N,
                                 None)
        assert rc == mhr.MHR_OK
        rc = mhr.gemm_f32_3xtf32_noalloc(a.data_ptr(), b.data_ptr(), c_new.data_ptr(), M, N, K,
                                         K, N, N, None)
        assert rc == mhr.MHR_OK, mhr.gemm_status_string(rc)
        assert mhr.gemm_check(None) == mhr.MHR_OK
        ref, new = c_ref.cpu().numpy(), c_new.cpu().numpy()
        assert np.all(np.isfinite(new))
        assert _normalised_error(new, ref, A, B) <= TOL["3xtf32"]


def test_noalloc_rejects_problems_beyond_its_scratch(mhr):
    import torch

    c = torch.zeros((2, 2), device="cuda")
    # 8 * 2048 * (2048 + 2048) bytes = 64 MiB fits exactly; one more row does not
    dummy = torch.zeros(16, device="cuda")
    rc = mhr.gemm_f32_3xtf32_noalloc(dummy.data_ptr(), dummy.data_ptr() + 4096, c.data_ptr(),
                                     2049, 2048, 2048, 2048, 2048, 2048, None)
    assert rc == mhr.MHR_ERR_INVALID_ARG
