"""What the tensor core reads from an fp32 operand under tcgen05.mma kind::tf32.

gemm_f32_3xtf32 splits A as A = A_big + A_small with A_big = A with the low 13
bits of every value cleared, and lets A itself stand in for A_big: the split
pre-pass writes only A_small. That is exact only if the tensor core, given a
raw fp32 operand, keeps the top 19 bits of each value and drops the rest
(truncation, not rounding to nearest). This pins that behaviour on the GPU:
with B the identity and A_small cleared by a test hook, the main kernel
computes C = A_big * (B_big + B_small) = A_big * I, one exact product per
output, so C must equal A & ~0x1FFF bit for bit. About half of the values
below round to a different tf32 value, so rounding would fail the test.
Without the hook, the same call must come within 2^-20 of A and differ from
the truncated values, which shows that the hook is what removed A_small.
"""
import numpy as np
import pytest

import seeded_inputs as si

pytestmark = pytest.mark.gpu


def _operand_with_low_bits(M, K, seed):
    """Normal fp32 values (magnitudes far from subnormal) whose low 13 bits are
    all nonzero."""
    x = si.matrix(M, K, seed, "normal")
    u = x.view(np.uint32).copy()
    low = (si.splitmix64(seed + 7, 0, M * K).reshape(M, K) & np.uint64(0x1FFF)).astype(np.uint32)
    u = (u & np.uint32(0xFFFFE000)) | np.maximum(low, np.uint32(1))
    out = u.view(np.float32)
    assert np.all(np.abs(out[out != 0]) > 2.0 ** -60)
    return out


@pytest.mark.parametrize("pair_mode", [1, 2], ids=["1cta", "pair"])
def test_tensor_core_truncates_fp32_operand_to_tf32(mhr, pair_mode):
    import torch

    M, K = 384, 256
    A = _operand_with_low_bits(M, K, 7401)
    eye = np.eye(K, dtype=np.float32)
    expected = (A.view(np.uint32) & np.uint32(0xFFFFE000)).view(np.float32)
    rounded_differs = np.count_nonzero(
        expected != ((A.view(np.uint32) + np.uint32(0x1000)) & np.uint32(0xFFFFE000)).view(np.float32))
    assert rounded_differs > M * K // 4  # the check can tell truncation from rounding
    a = torch.from_numpy(A).cuda()
    b = torch.from_numpy(eye).cuda()
    assert a.data_ptr() % 16 == 0  # A serves as its own big part
    c = torch.full((M, K), float("nan"), device="cuda")
    old_mode = mhr.gemm_testing_set_cta_pair_mode(pair_mode)
    old_split = mhr.gemm_testing_set_split_mode(1)
    old_zero = mhr.gemm_testing_set_zero_a_small(1)
    try:
        rc = mhr.gemm_f32_3xtf32(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, K, K, K, K, K, None)
        assert rc == mhr.MHR_OK
        assert mhr.gemm_check(None) == mhr.MHR_OK
    finally:
        mhr.gemm_testing_set_zero_a_small(old_zero)
        mhr.gemm_testing_set_split_mode(old_split)
        mhr.gemm_testing_set_cta_pair_mode(old_mode)
    got = c.cpu().numpy()
    bad = np.count_nonzero(got.view(np.uint32) != expected.view(np.uint32))
    assert bad == 0, (
        f"{bad} of {M * K} outputs differ from A & ~0x1FFF: the tensor core no longer truncates "
        "fp32 operands to tf32, so A cannot serve as its own big part in the 3xTF32 split "
        "(a_serves_as_big in the C ABI must then be turned off)")
    # Control: without the hook the same call is the full 3xTF32 product A * I,
    # which keeps about 22 of A's 24 significant bits -- within 2^-20 of A,
    # and (A_small being nonzero) not the truncated value.
    c2 = torch.full((M, K), float("nan"), device="cuda")
    old_mode = mhr.gemm_testing_set_cta_pair_mode(pair_mode)
    try:
        assert mhr.gemm_f32_3xtf32(a.data_ptr(), b.data_ptr(), c2.data_ptr(), M, K, K, K, K, K,
                                   None) == mhr.MHR_OK
        assert mhr.gemm_check(None) == mhr.MHR_OK
    finally:
        mhr.gemm_testing_set_cta_pair_mode(old_mode)
    full = c2.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(full - A) <= 2.0 ** -20 * np.abs(A))
    assert np.count_nonzero(full != expected) > M * K // 2
