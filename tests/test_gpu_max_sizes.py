"""The largest dimensions the C ABI accepts (2^31 - 512) on the GPU.

Each case puts one dimension -- M (rows of A and C) or N (columns of B and C)
-- at the maximum and the other two at 1, so the buffers stay at 8 GiB each
(plus the 3xTF32 split workspace of 64 GiB where it is used). Every 32-bit
tile, row and column coordinate of the kernels then reaches its largest value.
Inputs are small integers generated on the device, so every product is exact;
sampled outputs are compared bit for bit with the oracle on copies of the same
rows, and a NaN guard band past the end of C must stay untouched.
"""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu

KMAX = (1 << 31) - 512
GUARD = 64


def _int_vector(torch, n, seed):
    """Integers in {-2..2} from the element index, built on the device in chunks."""
    out = torch.empty(n, dtype=torch.float32, device="cuda")
    chunk = 1 << 27
    for s in range(0, n, chunk):
        i = torch.arange(s, min(s + chunk, n), dtype=torch.int64, device="cuda")
        out[s:s + i.numel()] = (((i * 2654435761 + seed) >> 7) % 5 - 2).float()
    return out


def _samples(n):
    picks = [0, 1, 127, 128, 255, 256, n // 2, n - 513, n - 257, n - 256, n - 2, n - 1]
    rng = np.random.default_rng(7)
    return np.unique(np.concatenate([picks, rng.integers(0, n, 20)]))


@pytest.mark.parametrize("case", ["f32", "3xtf32", "3xtf32-onchip"])
@pytest.mark.parametrize("dim", ["M", "N"])
def test_maximum_dimension(mhr, case, dim):
    import torch

    torch.cuda.empty_cache()
    n = KMAX
    entry = mhr.gemm_f32 if case == "f32" else mhr.gemm_f32_3xtf32
    old_limit = mhr.gemm_testing_set_workspace_limit(0 if case == "3xtf32-onchip" else 2**64 - 1)
    try:
        long_vec = _int_vector(torch, n, 11)               # A's column (dim M) or B's row (dim N)
        short = torch.tensor([[3.0]], device="cuda")       # the other operand, 1 x 1
        c = torch.full((n + GUARD,), float("nan"), device="cuda")
        if dim == "M":   # A: n x 1, B: 1 x 1, C: n x 1
            args = (long_vec.data_ptr(), short.data_ptr(), c.data_ptr(), n, 1, 1, 1, 1, 1)
        else:            # A: 1 x 1, B: 1 x n, C: 1 x n
            args = (short.data_ptr(), long_vec.data_ptr(), c.data_ptr(), 1, n, 1, 1, n, n)
        assert entry(*args, None) == mhr.MHR_OK
        assert mhr.gemm_check(None) == mhr.MHR_OK
        label = mhr.gemm_testing_last_main_kernel()
        if case == "3xtf32-onchip":
            assert label.startswith("tc_gemm_pair_kernel<3xtf32,split> "), label
        rows = _samples(n)
        idx = torch.from_numpy(rows).cuda()
        got = c[idx].cpu().numpy()
        vals = long_vec[idx].cpu().numpy().astype(np.float32)
        if dim == "M":
            ref = oracle.gemm(vals.reshape(-1, 1), np.array([[3.0]], np.float32)).reshape(-1)
        else:
            ref = oracle.gemm(np.array([[3.0]], np.float32), vals.reshape(1, -1)).reshape(-1)
        assert np.array_equal(got, ref), (case, dim, label)
        assert torch.isnan(c[n:]).all()
    finally:
        mhr.gemm_testing_set_workspace_limit(old_limit)
        mhr.gemm_release()
        del c
        torch.cuda.empty_cache()


def _int_bf16(torch, n, seed):
    """The same integers as _int_vector, stored as bf16 (exact)."""
    out = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    chunk = 1 << 27
    for s in range(0, n, chunk):
        i = torch.arange(s, min(s + chunk, n), dtype=torch.int64, device="cuda")
        out[s:s + i.numel()] = (((i * 2654435761 + seed) >> 7) % 5 - 2).to(torch.bfloat16)
    return out


@pytest.mark.parametrize("dim", ["M", "N"])
def test_maximum_dimension_bf16(mhr, dim):
    """bf16 on the tensor cores at the largest M (A: M x 8, 32 GiB) or N
    (B: 8 x N, 32 GiB), K = 8 so that the long operand's rows are 16-byte
    aligned for TMA; C in fp32 with a guard band."""
    import torch

    torch.cuda.empty_cache()
    n, k = KMAX, 8
    try:
        long_mat = _int_bf16(torch, n * k, 13)                  # A (n x 8) or B (8 x n)
        short = _int_bf16(torch, k, 17)                          # B (8 x 1) or A (1 x 8)
        c = torch.full((n + GUARD,), float("nan"), device="cuda")
        if dim == "M":
            args = (long_mat.data_ptr(), short.data_ptr(), c.data_ptr(), n, 1, k, k, 1, 1)
        else:
            args = (short.data_ptr(), long_mat.data_ptr(), c.data_ptr(), 1, n, k, k, n, n)
        assert mhr.gemm_bf16_f32acc(*args, None) == mhr.MHR_OK
        assert mhr.gemm_check(None) == mhr.MHR_OK
        label = mhr.gemm_testing_last_main_kernel()
        rows = _samples(n)
        idx = torch.from_numpy(rows).cuda()
        got = c[idx].cpu().numpy()
        s = short.float().cpu().numpy()
        if dim == "M":
            a = long_mat.view(n, k)[idx].float().cpu().numpy()
            ref = oracle.gemm(a, s.reshape(k, 1)).reshape(-1)
        else:
            b = long_mat.view(k, n)[:, idx].float().cpu().numpy()
            ref = oracle.gemm(s.reshape(1, k), np.ascontiguousarray(b)).reshape(-1)
        assert np.array_equal(got, ref), (dim, label)
        assert torch.isnan(c[n:]).all()
    finally:
        mhr.gemm_release()
        torch.cuda.empty_cache()
