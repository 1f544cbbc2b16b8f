"""Failure detection on the GPU without a fault (GB300 only).

A test hook makes block 0 of a tensor-core kernel leave its first ring stage
incomplete (a TMA producer arms it without loading it; the in-kernel split's
converter warps, where they fill it alone, fill it without arriving), so its
consumers' bounded waits run out. The kernel must record
the timeout, free its TMEM and exit; gemm_check() must report
MHR_ERR_TIMEOUT; and the context must stay usable (a following call is
correct). Nothing traps, faults or hangs.
"""
import numpy as np
import pytest

import oracle
from parity_util import TOL, DeviceCall, normalised_error, operands

pytestmark = pytest.mark.gpu


# Every producer kind: TMA loads in both kernels, the TMA loads of A beside
# the converter warps of the in-kernel split (aligned operands), and the
# converter warps alone (operands one element off alignment)
# (path, CTA-pair mode, 3xTF32 split mode, operand offset)
VARIANTS = [("3xtf32", 1, 1, 0), ("3xtf32", 1, 2, 0), ("3xtf32", 2, 1, 0), ("3xtf32", 2, 2, 0),
            ("3xtf32", 2, 2, 1), ("bf16", 1, 0, 0), ("bf16", 2, 0, 0)]
IDS = ["3xtf32-1cta", "3xtf32-1cta-insplit", "3xtf32-pair-prepass", "3xtf32-pair-insplit-tma-a",
       "3xtf32-pair-insplit-registers", "bf16-1cta", "bf16-pair"]


@pytest.mark.parametrize("variant", VARIANTS, ids=IDS)
def test_injected_stall_reports_timeout(mhr, variant):
    path, mode, split, offset = variant
    A, B, Ab, Bb = operands(300, 520, 700, 6001, "normal", path)
    call = DeviceCall(path, A, B, Ab, Bb, offset=offset)
    old_split = mhr.gemm_testing_set_split_mode(split)
    old_mode = mhr.gemm_testing_set_cta_pair_mode(mode)
    old_limit = mhr.gemm_testing_set_wait_limit_ns(50_000_000)  # 50 ms
    mhr.gemm_testing_set_inject_stall(1)
    try:
        call.run(mhr, check=False)
        bits = mhr.gemm_testing_peek_status(None)
        assert bits > 0 and (bits & 0x8) == 0, bits  # a timeout, and nothing left in flight
        assert mhr.gemm_check(None) == mhr.MHR_ERR_TIMEOUT
        assert mhr.gemm_check(None) == mhr.MHR_OK  # the check clears the word
    finally:
        mhr.gemm_testing_set_inject_stall(0)
        mhr.gemm_testing_set_wait_limit_ns(old_limit)
    # the context is still healthy: the same call now succeeds
    try:
        C = call.run(mhr).result()
    finally:
        mhr.gemm_testing_set_cta_pair_mode(old_mode)
        mhr.gemm_testing_set_split_mode(old_split)
    Cref, S = oracle.gemm(A, B, with_abs=True)
    assert normalised_error(C, Cref, S) <= TOL[path]


@pytest.mark.parametrize("path,K", [("3xtf32", 32 * 128 + 40), ("bf16", 64 * 128 + 40)],
                         ids=["3xtf32", "bf16"])
def test_injected_stall_in_cluster_split(mhr, path, K):
    """The single-CTA kernel's cluster split (few tiles, long K runs): block 0,
    rank 0 of the first cluster, times out on its first stage while its peers
    finish and wait for it at the cluster barrier; the timeout is reported, the
    kernel exits, and the next call on the context is correct."""
    A, B, Ab, Bb = operands(300, 520, K, 6002, "normal", path)
    call = DeviceCall(path, A, B, Ab, Bb)
    old_mode = mhr.gemm_testing_set_cta_pair_mode(1)
    old_limit = mhr.gemm_testing_set_wait_limit_ns(50_000_000)  # 50 ms
    mhr.gemm_testing_set_inject_stall(1)
    try:
        call.run(mhr, check=False)
        assert ",cluster-K> " in mhr.gemm_testing_last_main_kernel()
        bits = mhr.gemm_testing_peek_status(None)
        assert bits > 0 and (bits & 0x8) == 0, bits
        assert mhr.gemm_check(None) == mhr.MHR_ERR_TIMEOUT
        assert mhr.gemm_check(None) == mhr.MHR_OK
    finally:
        mhr.gemm_testing_set_inject_stall(0)
        mhr.gemm_testing_set_wait_limit_ns(old_limit)
    try:
        C = call.run(mhr).result()
    finally:
        mhr.gemm_testing_set_cta_pair_mode(old_mode)
    Cref, S = oracle.gemm(A, B, with_abs=True)
    assert normalised_error(C, Cref, S) <= TOL[path]
