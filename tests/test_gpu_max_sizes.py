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
