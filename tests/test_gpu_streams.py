"""Workspace ownership through the C ABI (GB300 only): calls on different
streams use separate workspaces and may overlap; gemm_release() frees them and
the next call allocates afresh."""
import numpy as np
import pytest

import oracle
from parity_util import TOL, normalised_error, operands

pytestmark = pytest.mark.gpu


def _run(mhr, torch, A, B, stream):
    M, K = A.shape
    N = B.shape[1]
    a, b = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    c = torch.full((M, N), float("nan"), device="cuda")
    torch.cuda.synchronize()
    rc = mhr.gemm_f32_3xtf32(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K, K, N, N,
                             stream.cuda_stream)
    assert rc == mhr.MHR_OK
    return a, b, c


def test_concurrent_streams_have_separate_workspaces(mhr):
    import torch

    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    probs = [operands(700, 900, 1500, 7301, "normal", "f32"),
             operands(1100, 600, 2000, 7303, "normal", "f32")]
    live = []
    for (A, B, _, _), s in zip(probs, (s1, s2)):
        live.append(_run(mhr, torch, A, B, s))  # both enqueued before either is checked
    assert mhr.gemm_check(s1.cuda_stream) == mhr.MHR_OK
    assert mhr.gemm_check(s2.cuda_stream) == mhr.MHR_OK
    for (A, B, _, _), (_, _, c) in zip(probs, live):
        Cref, S = oracle.gemm(A, B, with_abs=True)
        assert normalised_error(c.cpu().numpy(), Cref, S) <= TOL["3xtf32"]


def test_release_then_reuse(mhr):
    import torch

    A, B, _, _ = operands(300, 400, 500, 7305, "normal", "f32")
    s = torch.cuda.current_stream()
    _, _, c1 = _run(mhr, torch, A, B, s)
    assert mhr.gemm_check(s.cuda_stream) == mhr.MHR_OK
    first = c1.cpu().numpy()
    mhr.gemm_release()
    _, _, c2 = _run(mhr, torch, A, B, s)
    assert mhr.gemm_check(s.cuda_stream) == mhr.MHR_OK
    assert np.array_equal(c2.cpu().numpy(), first)
