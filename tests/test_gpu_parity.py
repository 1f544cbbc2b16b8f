"""Parity of every CUDA path with the CPU oracle, through the C ABI (GB300 only).

Small and ragged shapes are compared element by element with the full oracle;
the full-size workloads (4096^3, 8192^3, 3000 x 2050 x 1000) in the exact
launch configuration the benchmark times are compared on sampled outputs that
the oracle computes one by one. Integer-valued inputs must match bit for bit;
real-valued inputs must meet the normalised-error tolerance of each path.
"""
import numpy as np
import pytest

import oracle
from parity_util import (TOL, DeviceCall, normalised_error, operands, pair_tile_n,
                         sample_indices)

pytestmark = pytest.mark.gpu

PATHS = ["f32", "3xtf32", "bf16"]
# Each tensor-core path has two kernels: the single-CTA kernel (128-row tiles)
# and the CTA-pair kernel (256-row tiles over a cluster of 2); 3xTF32 splits
# its operands either in a pre-pass or inside the kernel (the single-CTA
# kernel's in-kernel split needs A 16-byte aligned with lda a multiple of 4,
# and hands other operands to the CTA-pair kernel's). Every combination is
# forced in turn on every small shape; full-size checks use the automatic
# choice, as the benchmark does.
# (path, CTA-pair mode, split mode)
VARIANTS = [("f32", 0, 0), ("3xtf32", 1, 1), ("3xtf32", 1, 2), ("3xtf32", 2, 1), ("3xtf32", 2, 2),
            ("bf16", 1, 0), ("bf16", 2, 0)]
VARIANT_IDS = ["f32", "3xtf32-1cta", "3xtf32-1cta-insplit", "3xtf32-pair-prepass",
               "3xtf32-pair-insplit", "bf16-1cta", "bf16-pair"]


@pytest.fixture(params=VARIANTS, ids=VARIANT_IDS)
def path(request, mhr):
    name, mode, split = request.param
    old = mhr.gemm_testing_set_cta_pair_mode(mode)
    old_split = mhr.gemm_testing_set_split_mode(split)
    yield name
    mhr.gemm_testing_set_split_mode(old_split)
    mhr.gemm_testing_set_cta_pair_mode(old)

# (M, N, K): single elements, thin shapes, several tiles with ragged tails in
# every dimension, and K long enough to wrap every ring several times
# (bf16: 64-wide K steps x 4 stages, 1-CTA, or 128-wide x 3, pair; tf32: 32-wide x 3;
# SIMT: 8-wide x 2). N = 130 and 1026 (2 mod 4) take the 3xTF32 split's
# 8-byte loads of B and the epilogue's 8-byte stores of C.
SMALL_SHAPES = [
    (1, 1, 1), (1, 300, 7), (7, 1, 300), (2, 3, 5), (127, 129, 65), (129, 257, 127),
    (256, 256, 256), (300, 520, 200), (255, 513, 1000), (130, 260, 769), (200, 200, 289),
    (64, 1100, 33), (200, 130, 300), (70, 1026, 65),
]


def check_full(mhr, path, M, N, K, seed, dist="normal", **kw):
    A, B, Ab, Bb = operands(M, N, K, seed, dist, path)
    C = DeviceCall(path, A, B, Ab, Bb, **kw).run(mhr).result()
    Cref, S = oracle.gemm(A, B, with_abs=True)
    err = normalised_error(C, Cref, S)
    assert err <= TOL[path], (path, M, N, K, err)
    return err


@pytest.mark.parametrize("shape", SMALL_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_small_shapes(mhr, path, shape):
    check_full(mhr, path, *shape, seed=1000 + sum(shape))


def test_config1_uniform_256(mhr, path):
    """256^3, uniform[-1, 1), seeds (1001, 1002)."""
    check_full(mhr, path, 256, 256, 256, seed=1001, dist="uniform")


@pytest.mark.parametrize("shape", [(256, 256, 256), (300, 520, 1000), (8, 8, 8)],
                         ids=lambda s: "x".join(map(str, s)))
def test_integer_twin_bit_exact(mhr, path, shape):
    """Integers in {-2..2}: every product and partial sum is exact in fp32, tf32
    and bf16, so every path must reproduce the oracle bit for bit."""
    M, N, K = shape
    A, B, Ab, Bb = operands(M, N, K, 1011, "int", path)
    C = DeviceCall(path, A, B, Ab, Bb).run(mhr).result()
    assert np.array_equal(C, oracle.gemm(A, B))


def test_block_decomposition_n8_tile4(mhr, path):
    """The pages' N=8, TILE=4 example on the GPU: C00 = A00*B00 + A01*B10 on
    integer inputs, each product computed by the same entry point."""
    A, B, Ab, Bb = operands(8, 8, 8, 11, "int", path)
    C = DeviceCall(path, A, B, Ab, Bb).run(mhr).result()
    T = 4
    for bi in range(2):
        for bj in range(2):
            acc = np.zeros((T, T), np.float32)
            for t in range(2):
                a = np.ascontiguousarray(A[bi * T:(bi + 1) * T, t * T:(t + 1) * T])
                b = np.ascontiguousarray(B[t * T:(t + 1) * T, bj * T:(bj + 1) * T])
                ab = bb = None
                if path == "bf16":
                    ab = np.ascontiguousarray(Ab[bi * T:(bi + 1) * T, t * T:(t + 1) * T])
                    bb = np.ascontiguousarray(Bb[t * T:(t + 1) * T, bj * T:(bj + 1) * T])
                acc += DeviceCall(path, a, b, ab, bb).run(mhr).result()
            assert np.array_equal(C[bi * T:(bi + 1) * T, bj * T:(bj + 1) * T], acc)


def test_identity_and_ones(mhr, path):
    import seeded_inputs as si

    M, N = 200, 300
    B = si.matrix(M, N, 77, "int")
    eye = np.eye(M, dtype=np.float32)
    ab = bb = None
    if path == "bf16":
        ab, _ = si.bf16_rne(eye)
        bb, _ = si.bf16_rne(B)
    assert np.array_equal(DeviceCall(path, eye, B, ab, bb).run(mhr).result(), B)
    K = 1000
    ones_a, ones_b = np.ones((64, K), np.float32), np.ones((K, 96), np.float32)
    if path == "bf16":
        ab, _ = si.bf16_rne(ones_a)
        bb, _ = si.bf16_rne(ones_b)
    assert np.all(DeviceCall(path, ones_a, ones_b, ab, bb).run(mhr).result() == K)


def test_padded_leading_dims_nan_poison(mhr, path):
    """ld > width with NaN in every pad: a read outside the logical matrix
    poisons C; a write outside it breaks the guard band (checked in result())."""
    check_full(mhr, path, 131, 250, 77, seed=2201, lda=77 + 5, ldb=250 + 3, ldc=250 + 7)
    check_full(mhr, path, 131, 256, 128, seed=2202, lda=136, ldb=264, ldc=260)


def test_misaligned_pointers(mhr, path):
    """Operands and output shifted one element off 16-byte alignment: the SIMT
    path falls back to scalar accesses, the tensor-core paths repack/split the
    operands and store C without TMA."""
    check_full(mhr, path, 150, 270, 90, seed=2301, offset=1)
    check_full(mhr, path, 150, 270, 90, seed=2302, offset=1, lda=91, ldb=271, ldc=271)


def test_deterministic(mhr, path):
    """Fixed MMA order: repeated calls give bit-identical results (a missing
    ring barrier would show up here as run-to-run differences)."""
    A, B, Ab, Bb = operands(384, 640, 1217, 2401, "normal", path)
    call = DeviceCall(path, A, B, Ab, Bb)
    first = call.run(mhr).result()
    for _ in range(5):
        assert np.array_equal(call.run(mhr).result(), first)


def test_degenerate_sizes(mhr, path):
    import torch

    ent = {"f32": mhr.gemm_f32, "3xtf32": mhr.gemm_f32_3xtf32, "bf16": mhr.gemm_bf16_f32acc}[path]
    C = torch.full((5, 7), float("nan"), device="cuda")
    # K == 0: C becomes the empty sum, zero
    assert ent(None, None, C.data_ptr(), 5, 7, 0, 0, 0, 7, None) == mhr.MHR_OK
    assert mhr.gemm_check(None) == mhr.MHR_OK
    assert torch.all(C == 0)
    # M == 0 / N == 0: nothing written
    C.fill_(3.0)
    assert ent(None, None, C.data_ptr(), 0, 7, 4, 4, 7, 7, None) == mhr.MHR_OK
    assert ent(None, None, C.data_ptr(), 5, 0, 4, 4, 0, 7, None) == mhr.MHR_OK
    assert torch.all(C == 3.0)


def test_config3_rectangular_full(mhr):
    """3000 x 2050 x 1000, normal(0,1), seeds (3001, 3002): none of the sizes is
    a tile multiple and B's row pitch (2050 floats) is not 16-byte aligned.
    Full comparison for both fp32 paths."""
    M, N, K = 3000, 2050, 1000
    A, B, _, _ = operands(M, N, K, 3001, "normal", "f32")
    Cref, S = oracle.gemm(A, B, with_abs=True)
    for path in ("f32", "3xtf32"):
        C = DeviceCall(path, A, B).run(mhr).result()
        err = normalised_error(C, Cref, S)
        assert err <= TOL[path], (path, err)
        if path == "3xtf32":
            # C's pitch rules out TMA stores; the pair tiles are as wide as the
            # planner says for this GPU (176 columns on 76 clusters)
            label = mhr.gemm_testing_last_main_kernel()
            if label.startswith("tc_gemm_pair_kernel<3xtf32"):
                import re

                clusters = int(re.search(r"grid=(\d+)", label).group(1)) // 2
                bn = mhr.gemm_testing_plan_pair_tile_n(M, N, K, clusters, False)
                want = "tc_gemm_pair_kernel<3xtf32" + ("> " if bn == 256 else f",n{bn}> ")
                assert label.startswith(want), (label, want)


def sampled_check(mhr, path, M, N, K, seed, dist):
    A, B, Ab, Bb = operands(M, N, K, seed, dist, path)
    C = DeviceCall(path, A, B, Ab, Bb).run(mhr).result()
    rows, cols = sample_indices(M, N, seed, rows=(0, M // 2 + 1, M - 1), cols=(0, N - 1))
    ref, S = oracle.gemm_entries(A, B, rows, cols, M, N, K)
    err = normalised_error(C[rows, cols], ref, S)
    assert err <= TOL[path], (path, M, N, K, err)
    return err


@pytest.mark.parametrize("path", ["f32", "3xtf32"])
def test_config2_4096_sampled(mhr, path):
    """4096^3 fp32, uniform[-1, 1), seeds (2001, 2002)."""
    sampled_check(mhr, path, 4096, 4096, 4096, 2001, "uniform")


def test_config4_8192_3xtf32_sampled(mhr):
    """8192^3 fp32 through 3xTF32, uniform[-1, 1), seeds (4001, 4002)."""
    sampled_check(mhr, "3xtf32", 8192, 8192, 8192, 4001, "uniform")


def test_config5_8192_bf16_sampled(mhr):
    """8192^3 bf16 inputs (normal(0,1) rounded to bf16), fp32 accumulate and
    output, seeds (5001, 5002); the oracle runs on the bf16 values."""
    sampled_check(mhr, "bf16", 8192, 8192, 8192, 5001, "normal")


@pytest.fixture
def full_width_tiles(mhr):
    """The 3xTF32 CTA-pair tiles at their full 256 columns, for tests that
    count tiles or compare the pre-pass path with the in-kernel split (which
    always runs 256-column tiles) bit for bit."""
    with pair_tile_n(mhr, 256):
        yield


def pair_clusters(mhr, path):
    """The number of clusters the CTA-pair kernel runs on this GPU."""
    import re

    A, B, Ab, Bb = operands(4096, 4096, 64, 3101, "normal", path)
    DeviceCall(path, A, B, Ab, Bb).run(mhr)
    label = mhr.gemm_testing_last_main_kernel()
    clusters = int(re.search(r"grid=(\d+)", label).group(1)) // 2
    assert clusters >= 8, label
    return clusters


@pytest.mark.usefixtures("full_width_tiles")
@pytest.mark.parametrize("path", ["3xtf32", "bf16"])
def test_pair_kernel_split_last_round(mhr, path):
    """The CTA-pair kernel splits a sparse last round of tiles into two K halves
    that are reduce-added into C. Build a problem with 3 more pair tiles than
    co-resident clusters, so exactly 3 tiles are split, and compare it in full
    with the oracle, through the TMA reduce path (aligned C) and the atomic
    path (ldc odd), and for bitwise repeatability. With every buffer one
    element off 16-byte alignment, the pre-pass (the bf16 repacks, or the
    3xTF32 split with 4-byte loads) runs alongside the kernel zeroing C's
    split tiles, which then writes 4-byte stores. ldc = N + 2 (2 mod 4)
    takes the mixed path: TMA reduce-adds into C's even rows, atomic adds
    into the odd ones."""
    old = mhr.gemm_testing_set_cta_pair_mode(2)
    try:
        clusters = pair_clusters(mhr, path)
        M, N, K = 256 * (clusters + 3), 256, 320
        for ldc, offset in ((None, 0), (N + 1, 0), (N + 2, 0), (None, 1)):
            A, B, Ab, Bb = operands(M, N, K, 3103, "normal", path)
            call = DeviceCall(path, A, B, Ab, Bb, ldc=ldc, offset=offset)
            C = call.run(mhr).result()
            assert f"tiles={clusters + 3}" in mhr.gemm_testing_last_main_kernel()
            Cref, S = oracle.gemm(A, B, with_abs=True)
            assert normalised_error(C, Cref, S) <= TOL[path]
            assert np.array_equal(call.run(mhr).result(), C)
    finally:
        mhr.gemm_testing_set_cta_pair_mode(old)


@pytest.mark.usefixtures("full_width_tiles")
@pytest.mark.parametrize("path", ["3xtf32", "bf16"])
@pytest.mark.parametrize("extra", [1, -1, 5, 28], ids=["c+1", "2c-1", "2c+5", "3c+28"])
def test_pair_kernel_schedule_bit_exact(mhr, path, extra):
    """Integer inputs through tile counts around the round boundaries of the
    persistent schedule: one round plus one tile, two rounds minus one, two
    plus five, and three plus 28 (the 4096^3 case's 256 tiles on 76
    clusters). Every K-block of every tile must be computed exactly once,
    split or not; the sums are exact, so C must match the oracle bit for
    bit."""
    old = mhr.gemm_testing_set_cta_pair_mode(2)
    try:
        clusters = pair_clusters(mhr, path)
        tiles = {1: clusters + 1, -1: 2 * clusters - 1, 5: 2 * clusters + 5,
                 28: 3 * clusters + 28}[extra]
        M, N, K = 256 * tiles, 256, 320
        A, B, Ab, Bb = operands(M, N, K, 3105 + extra, "int", path)
        C = DeviceCall(path, A, B, Ab, Bb).run(mhr).result()
        assert f"tiles={tiles}" in mhr.gemm_testing_last_main_kernel()
        assert np.array_equal(C, oracle.gemm(A, B))
    finally:
        mhr.gemm_testing_set_cta_pair_mode(old)


@pytest.mark.parametrize("bn", [240, 224, 176, 144, 128])
def test_pair_kernel_narrow_tiles(mhr, bn):
    """3xTF32 CTA-pair tiles narrower than 256 columns: each CTA loads bn / 2
    rows of each B part, the MMAs run with N = bn, and the epilogue writes
    ceil(bn / 32) chunks per tile, the last one masked at the tile's edge when
    bn is not a multiple of 32. 10 tile columns (N = 10 bn - 8 or 10 bn - 7,
    a short last column) by 8 tile rows (M = 1948, ragged) are 80 tiles: one
    round plus 4 tiles split into K halves on 76 clusters. Integer inputs
    match the oracle bit for bit through TMA stores (N a multiple of 4 with C
    aligned, for widths that are whole chunks) and register stores (N odd,
    ldc = N + 1); real inputs meet the tolerance, bitwise repeatably."""
    import re

    M, K = 1948, 96 + 5
    old = mhr.gemm_testing_set_cta_pair_mode(2)
    try:
        with pair_tile_n(mhr, bn):
            for N, ldc in ((10 * bn - 8, None), (10 * bn - 7, 10 * bn - 6)):
                A, B, _, _ = operands(M, N, K, 3701 + bn, "int", "3xtf32")
                C = DeviceCall("3xtf32", A, B, ldc=ldc).run(mhr).result()
                label = mhr.gemm_testing_last_main_kernel()
                assert label.startswith(f"tc_gemm_pair_kernel<3xtf32,n{bn}> "), label
                clusters = int(re.search(r"grid=(\d+)", label).group(1)) // 2
                assert f"tiles={8 * 10}" in label, label
                assert np.array_equal(C, oracle.gemm(A, B)), (bn, ldc, clusters)
            A, B, _, _ = operands(M, N, K, 3702 + bn, "normal", "3xtf32")
            call = DeviceCall("3xtf32", A, B, ldc=ldc)
            C = call.run(mhr).result()
            Cref, S = oracle.gemm(A, B, with_abs=True)
            assert normalised_error(C, Cref, S) <= TOL["3xtf32"]
            assert np.array_equal(call.run(mhr).result(), C)
    finally:
        mhr.gemm_testing_set_cta_pair_mode(old)


# (path, CTA-pair mode, split mode, forced pair tile width)
ODD_ROW_VARIANTS = [("3xtf32", 2, 1, 256), ("3xtf32", 2, 1, 176), ("3xtf32", 1, 1, 0),
                    ("bf16", 2, 0, 0), ("bf16", 1, 0, 0)]


@pytest.mark.parametrize("variant", ODD_ROW_VARIANTS,
                         ids=["3xtf32-pair", "3xtf32-pair-n176", "3xtf32-1cta", "bf16-pair",
                              "bf16-1cta"])
def test_even_and_odd_row_maps(mhr, variant):
    """C 16-byte aligned with an even ldc but not storable by TMA as a whole
    (ldc 2 mod 4, or N not a multiple of 4): whole chunks store their even
    rows through a map over rows 0, 2, 4, ... and their odd rows through a map
    over rows 1, 3, 5, ... whose base lies ldc % 4 columns left of each odd
    row (so a box starts 2 columns into the chunk and ends 2 into the next;
    the tile's first 2 odd-row columns go out from registers). Odd and even
    M, every N mod 4, ragged tiles. Integer inputs bit-exact against the
    oracle; C's padding keeps its guard values; real inputs within the
    tolerance."""
    path, mode, split, bn = variant
    old = mhr.gemm_testing_set_cta_pair_mode(mode)
    old_split = mhr.gemm_testing_set_split_mode(split)
    try:
        with pair_tile_n(mhr, bn):
            for M, N, K, ldc in ((300, 520, 200, 522), (301, 518, 200, 520), (300, 517, 200, 518),
                                 (301, 515, 136, 516), (64, 1100, 72, 1102), (2, 298, 40, 300),
                                 (1, 298, 40, 302)):
                A, B, Ab, Bb = operands(M, N, K, 3551 + N + M, "int", path)
                C = DeviceCall(path, A, B, Ab, Bb, ldc=ldc).run(mhr).result()
                assert np.array_equal(C, oracle.gemm(A, B)), (M, N, K, ldc)
            A, B, Ab, Bb = operands(300, 520, 200, 3552, "normal", path)
            C = DeviceCall(path, A, B, Ab, Bb, ldc=522).run(mhr).result()
            Cref, S = oracle.gemm(A, B, with_abs=True)
            assert normalised_error(C, Cref, S) <= TOL[path]
    finally:
        mhr.gemm_testing_set_split_mode(old_split)
        mhr.gemm_testing_set_cta_pair_mode(old)


@pytest.mark.usefixtures("full_width_tiles")
@pytest.mark.parametrize("path", ["3xtf32", "bf16"])
def test_split_last_round_odd_row_map(mhr, path):
    """The split last round (K halves reduce-added into zeroed C) through the
    even- and odd-row maps: N = 254 with ldc = 256 (odd-row map unshifted) and
    N = 252 with ldc = 254 (shifted by 2 columns); 3 more pair tiles than
    clusters. Integer inputs: every addend is exact, so C matches the oracle
    bit for bit, and no column is added twice."""
    old = mhr.gemm_testing_set_cta_pair_mode(2)
    try:
        clusters = pair_clusters(mhr, path)
        for N, ldc in ((254, 256), (252, 254)):
            M, K = 256 * (clusters + 3), 320
            A, B, Ab, Bb = operands(M, N, K, 3553 + N, "int", path)
            C = DeviceCall(path, A, B, Ab, Bb, ldc=ldc).run(mhr).result()
            assert f"tiles={clusters + 3}" in mhr.gemm_testing_last_main_kernel()
            assert np.array_equal(C, oracle.gemm(A, B)), (N, ldc)
    finally:
        mhr.gemm_testing_set_cta_pair_mode(old)


@pytest.mark.parametrize("bn", [128, 96, 64, 32])
def test_single_cta_tile_widths(mhr, bn):
    """The single-CTA 3xTF32 kernel at each tile width it can run (128 rows x
    bn; each stage holds bn rows of each B part, the MMAs run with N = bn).
    300 x 520 x 1000 (ragged, few tiles: K halves) and 1100 x 700 x 200 (with
    32 columns, 9 x 22 tiles: more than one round). Integer inputs bit-exact
    against the oracle through TMA stores (aligned C), register stores (odd
    ldc) and the even-row mixed path (ldc 2 mod 4); real inputs within the
    tolerance, bitwise repeatably."""
    old = mhr.gemm_testing_set_cta_pair_mode(1)
    old_split = mhr.gemm_testing_set_split_mode(1)  # the split pre-pass (small problems would
    old_n = mhr.gemm_testing_set_single_tile_n(bn)  # otherwise run as one launch)
    try:
        for M, N, K in ((300, 520, 1000), (1100, 700, 200)):
            for ldc in (None, N + 1, N + 2):
                A, B, _, _ = operands(M, N, K, 3801 + bn + K, "int", "3xtf32")
                C = DeviceCall("3xtf32", A, B, ldc=ldc).run(mhr).result()
                label = mhr.gemm_testing_last_main_kernel()
                want = "tc_gemm_kernel<3xtf32" + ("> " if bn == 128 else f",n{bn}> ")
                assert label.startswith(want), (label, want)
                assert np.array_equal(C, oracle.gemm(A, B)), (M, N, K, ldc)
            A, B, _, _ = operands(M, N, K, 3802 + bn + K, "normal", "3xtf32")
            call = DeviceCall("3xtf32", A, B, ldc=N + 2)
            C = call.run(mhr).result()
            Cref, S = oracle.gemm(A, B, with_abs=True)
            assert normalised_error(C, Cref, S) <= TOL["3xtf32"]
            assert np.array_equal(call.run(mhr).result(), C)
    finally:
        mhr.gemm_testing_set_single_tile_n(old_n)
        mhr.gemm_testing_set_split_mode(old_split)
        mhr.gemm_testing_set_cta_pair_mode(old)


@pytest.mark.parametrize("path,width", [("3xtf32", 128), ("3xtf32", 64), ("bf16", 256),
                                        ("bf16", 128)],
                         ids=["3xtf32-128", "3xtf32-64", "bf16-256", "bf16-128"])
def test_single_cta_few_tiles(mhr, path, width):
    """Few tiles on the single-CTA kernel. With long K runs (at least 16
    K-blocks per rank) it runs a cluster of 4 to 8 CTAs per tile (16 for
    3xTF32 where they fit), each on one run of K-blocks, and sums the
    partial tiles through distributed shared memory in rank order. Otherwise, when the halves of all tiles fit on the
    SMs at once (and, without a pre-pass to overlap the zeroing, K has at
    least 32 steps), every tile becomes two K halves reduce-added into a
    zeroed C. Cases: 4 tiles with 129-130 K-blocks (cluster of 8; of 16 for
    3xTF32, whose ranks then run 9 K-blocks, and 10 such tiles in clusters of
    8) and 65-66 (cluster of 4, ragged runs), half the SM count in tiles (K
    halves) and one more (no split); K ragged throughout. 3xTF32 at 128 and
    64 columns, bf16 at 256 and 128 (forced). Integer inputs bit-exact
    against the oracle through vector and scalar stores (ldc odd), real inputs within
    tolerance and bitwise repeatable."""
    import torch

    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tile_n = width or 128  # single-CTA tiles: 128 x tile_n
    bk = 64 if path == "bf16" else 32
    full = 128 if path == "3xtf32" else 256
    name = f"tc_gemm_kernel<{path}" + ("" if width == full else f",n{width}")
    old = mhr.gemm_testing_set_cta_pair_mode(1)
    old_n = mhr.gemm_testing_set_single_tile_n(width)
    try:
        cases = [(4, bk * 64 + 40, f"{name},cluster-K> grid=16 "),
                 (sms // 2, bk * 32 + 40, f"{name}> grid={sms} "),
                 (sms // 2 + 1, bk * 32 + 40, f"{name}> grid={sms // 2 + 1} ")]
        if path == "3xtf32":  # clusters of 16, and of 8 where 16 would not fit
            cases += [(4, bk * 128 + 40, f"{name},cluster-K> grid=64 "),
                      (10, bk * 128 + 40, f"{name},cluster-K> grid=80 ")]
        else:
            cases += [(4, bk * 128 + 40, f"{name},cluster-K> grid=32 ")]
        for tiles, K, want in cases:
            M, N = 128 * tiles, tile_n
            for ldc in (None, N + 1, N + 2):
                A, B, Ab, Bb = operands(M, N, K, 3112 + tiles + K, "int", path)
                C = DeviceCall(path, A, B, Ab, Bb, ldc=ldc).run(mhr).result()
                label = mhr.gemm_testing_last_main_kernel()
                assert label.startswith(want), (label, want)
                assert np.array_equal(C, oracle.gemm(A, B))
        for tiles, K in ((4, bk * 128 + 40), (sms // 2, 1000)):
            A, B, Ab, Bb = operands(128 * tiles, tile_n, K, 3113 + tiles, "normal", path)
            call = DeviceCall(path, A, B, Ab, Bb)
            C = call.run(mhr).result()
            Cref, S = oracle.gemm(A, B, with_abs=True)
            assert normalised_error(C, Cref, S) <= TOL[path]
            assert np.array_equal(call.run(mhr).result(), C)
    finally:
        mhr.gemm_testing_set_single_tile_n(old_n)
        mhr.gemm_testing_set_cta_pair_mode(old)


@pytest.mark.parametrize("shape", [(300, 520, 1000), (255, 513, 1001), (130, 260, 37),
                                   (512, 512, 4096), (256 * 79, 256, 320), (300, 130, 1000)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("offset", [0, 1], ids=["aligned", "offset1"])
@pytest.mark.usefixtures("full_width_tiles")
def test_in_kernel_split_matches_prepass_bitwise(mhr, shape, offset):
    """The CTA-pair kernel with the split inside the kernel computes exactly
    what it computes on pre-split operands: the same tf32 parts, the same
    MMAs in the same order. Aligned operands take the kind that stages A by
    TMA; operands one element off 16-byte alignment the one that reads both
    through registers, element by element. Ragged K (not a multiple of 4, of
    the 32-wide K step), ragged N (not a multiple of 4), and 79 tiles (a split
    last round on 76 clusters) included."""
    M, N, K = shape
    A, B, _, _ = operands(M, N, K, 3201 + K, "normal", "3xtf32")
    old = mhr.gemm_testing_set_cta_pair_mode(2)
    try:
        outs = []
        for split in (1, 2):
            old_split = mhr.gemm_testing_set_split_mode(split)
            try:
                outs.append(DeviceCall("3xtf32", A, B, offset=offset).run(mhr).result())
                label = mhr.gemm_testing_last_main_kernel()
                tma_a = offset == 0 and K % 4 == 0  # A 16-byte aligned, lda = K a multiple of 4
                want = ">" if split == 1 else (",split,tma-a>" if tma_a else ",split>")
                assert label.startswith("tc_gemm_pair_kernel<3xtf32" + want), label
            finally:
                mhr.gemm_testing_set_split_mode(old_split)
    finally:
        mhr.gemm_testing_set_cta_pair_mode(old)
    assert np.array_equal(outs[0], outs[1])
    Cref, S = oracle.gemm(A, B, with_abs=True)
    assert normalised_error(outs[1], Cref, S) <= TOL["3xtf32"]


@pytest.mark.parametrize("shape", [(256, 256, 256), (200, 300, 520), (512, 512, 8192),
                                   (1024, 1024, 1024), (130, 1000, 64)],
                         ids=lambda s: "x".join(map(str, s)))
def test_single_cta_in_kernel_split_is_one_launch(mhr, shape):
    """The single-CTA kernel's in-kernel split does the whole 3xTF32 product
    in one launch (no pre-pass, no zeroing of C), with clusters splitting K
    when the tiles are few, and matches the oracle; on integer inputs bit for
    bit."""
    M, N, K = shape
    old = mhr.gemm_testing_set_cta_pair_mode(1)
    old_split = mhr.gemm_testing_set_split_mode(2)
    try:
        for dist in ("normal", "int"):
            A, B, _, _ = operands(M, N, K, 3401 + K, dist, "3xtf32")
            C = DeviceCall("3xtf32", A, B).run(mhr).result()
            assert mhr.gemm_testing_last_main_kernel().startswith(
                "tc_gemm_kernel<3xtf32,split,tma-a"), mhr.gemm_testing_last_main_kernel()
            assert mhr.gemm_testing_last_launches() == 1
            if dist == "int":
                assert np.array_equal(C, oracle.gemm(A, B))
            else:
                Cref, S = oracle.gemm(A, B, with_abs=True)
                assert normalised_error(C, Cref, S) <= TOL["3xtf32"]
    finally:
        mhr.gemm_testing_set_split_mode(old_split)
        mhr.gemm_testing_set_cta_pair_mode(old)


@pytest.mark.parametrize("bn", [128, 96, 64, 32])
def test_one_launch_tile_widths(mhr, bn):
    """The one-launch form (single-CTA kernel, split inside) at each tile
    width: converter warps write bn rows of B^T's parts, the MMAs run with
    N = bn, and a cluster per tile splits K when the tiles are few (its
    partial tiles bn columns wide). 256^3 (a cluster per tile), 300 x 520 x
    1000 and 64 x 1000 x 300 (ragged tiles). Integer inputs bit-exact against
    the oracle through TMA stores, register stores (odd ldc) and the even-row
    path (ldc 2 mod 4); real inputs within the tolerance."""
    old = mhr.gemm_testing_set_cta_pair_mode(1)
    old_split = mhr.gemm_testing_set_split_mode(2)
    old_n = mhr.gemm_testing_set_single_tile_n(bn)
    try:
        for M, N, K in ((256, 256, 256), (300, 520, 1000), (64, 1000, 300)):
            for ldc in (None, N + 1, N + 2):
                A, B, _, _ = operands(M, N, K, 3901 + bn + K, "int", "3xtf32")
                C = DeviceCall("3xtf32", A, B, ldc=ldc).run(mhr).result()
                label = mhr.gemm_testing_last_main_kernel()
                want = "tc_gemm_kernel<3xtf32,split,tma-a" + ("" if bn == 128 else f",n{bn}")
                assert label.startswith(want), (label, want)
                assert mhr.gemm_testing_last_launches() == 1
                assert np.array_equal(C, oracle.gemm(A, B)), (M, N, K, ldc, label)
            A, B, _, _ = operands(M, N, K, 3902 + bn + K, "normal", "3xtf32")
            C = DeviceCall("3xtf32", A, B, ldc=N + 2).run(mhr).result()
            Cref, S = oracle.gemm(A, B, with_abs=True)
            assert normalised_error(C, Cref, S) <= TOL["3xtf32"]
    finally:
        mhr.gemm_testing_set_single_tile_n(old_n)
        mhr.gemm_testing_set_split_mode(old_split)
        mhr.gemm_testing_set_cta_pair_mode(old)


@pytest.mark.parametrize("shape,one_launch", [
    ((256, 256, 256), True), ((512, 512, 512), True), ((300, 520, 1000), True),
    ((256, 256, 2048), True), ((512, 512, 2052), False), ((1024, 1024, 1024), False)],
    ids=lambda v: "x".join(map(str, v)) if isinstance(v, tuple) else str(v))
def test_automatic_mode_runs_small_problems_as_one_launch(mhr, shape, one_launch):
    """In the automatic mode, small 3xTF32 problems (M N <= 2^18, K <= 2048)
    run as one launch of the single-CTA kernel with the split inside; larger
    ones, and A one element off 16-byte alignment, take the split pre-pass.
    Either way C matches the oracle bit for bit on integer inputs."""
    M, N, K = shape
    A, B, _, _ = operands(M, N, K, 3951 + K, "int", "3xtf32")
    for offset in (0, 1):
        call = DeviceCall("3xtf32", A, B, offset=offset)
        C = call.run(mhr).result()
        label = mhr.gemm_testing_last_main_kernel()
        if one_launch and offset == 0:
            assert label.startswith("tc_gemm_kernel<3xtf32,split,tma-a"), label
            assert mhr.gemm_testing_last_launches() == 1
        else:
            assert ",split" not in label, label
            assert mhr.gemm_testing_last_launches() >= 2  # the split pre-pass and the main kernel
        assert np.array_equal(C, oracle.gemm(A, B)), (shape, offset, label)



@pytest.mark.parametrize("shape", [(1536, 1536, 1024), (1024, 2048, 640), (1024, 1024, 1024),
                                   (1280, 1280, 512), (768, 768, 768), (1024, 1024, 200)],
                         ids=lambda s: "x".join(map(str, s)))
def test_automatic_mode_narrow_pair_tiles(mhr, shape):
    """3xTF32 shapes with too few 256 x 256 pair tiles for half of the
    clusters still take the CTA-pair kernel at the widest width (256, 192 or
    128 columns) whose work units -- every tile split into two K halves when
    twice the tiles fit on the clusters -- keep at least 80 % of the clusters
    busy (1536 x 1536: 36 tiles of 256 x 256, 72 half-K units on 76
    clusters; 1024 x 1024: 128 columns); with none the single-CTA kernel
    runs. Integer inputs bit-exact against the oracle on sampled entries."""
    import torch

    M, N, K = shape
    clusters = torch.cuda.get_device_properties(0).multi_processor_count // 2
    A, B, _, _ = operands(M, N, K, 3971 + K, "int", "3xtf32")
    C = DeviceCall("3xtf32", A, B).run(mhr).result()
    label = mhr.gemm_testing_last_main_kernel()
    rows256 = -(-M // 256)
    few = 0
    for bn in (256, 192, 128):
        tiles = rows256 * -(-N // bn)
        units = 2 * tiles if 2 * tiles <= clusters and -(-K // 32) >= 32 else tiles
        if units <= clusters and 5 * units >= 4 * clusters:
            few = bn
            break
    if 2 * rows256 * -(-N // 256) >= clusters:
        want = "tc_gemm_pair_kernel<3xtf32"
    elif few:
        want = "tc_gemm_pair_kernel<3xtf32" + ("> " if few == 256 else f",n{few}> ")
    else:
        want = "tc_gemm_kernel<3xtf32"
    assert label.startswith(want), (label, want)
    rows, cols = sample_indices(M, N, 3971, rows=(0, M // 2 + 1, M - 1), cols=(0, N - 1))
    ref = oracle.gemm_entries(A, B, rows, cols, M, N, K)[0]
    assert np.array_equal(C[rows, cols], ref)


@pytest.mark.parametrize("shape", [(2304, 2304, 1536), (2048, 2048, 1280), (1024, 2048, 2048),
                                   (1024, 1024, 2048), (3000, 2050, 1000)],
                         ids=lambda s: "x".join(map(str, s)))
def test_automatic_mode_bf16(mhr, shape):
    """bf16 takes the CTA-pair kernel when its 256 x 256 tiles fill half of
    the clusters and there is enough work per tile: K >= 1536 or at least two
    tiles per cluster; otherwise the single-CTA kernel's 128 x 256 tiles.
    Integer inputs bit-exact against the oracle on sampled entries."""
    import torch

    M, N, K = shape
    clusters = torch.cuda.get_device_properties(0).multi_processor_count // 2
    A, B, Ab, Bb = operands(M, N, K, 4211 + K, "int", "bf16")
    C = DeviceCall("bf16", A, B, Ab, Bb).run(mhr).result()
    label = mhr.gemm_testing_last_main_kernel()
    tiles = -(-M // 256) * -(-N // 256)
    pair = 2 * tiles >= clusters and (K >= 1536 or tiles >= 2 * clusters)
    want = "tc_gemm_pair_kernel<bf16" if pair else "tc_gemm_kernel<bf16"
    assert label.startswith(want), (label, want)
    rows, cols = sample_indices(M, N, 4211, rows=(0, M // 2 + 1, M - 1), cols=(0, N - 1))
    ref = oracle.gemm_entries(A, B, rows, cols, M, N, K)[0]
    assert np.array_equal(C[rows, cols], ref)


@pytest.mark.parametrize("shape,want", [
    ((1024, 1024, 1024), "tc_gemm_kernel<bf16,n128> grid=64 "),
    ((256, 256, 8192), "tc_gemm_kernel<bf16,n128,cluster-K> grid=32 "),
    ((768, 768, 768), "tc_gemm_kernel<bf16,n128> grid=36 "),
    ((1536, 2560, 512), "tc_gemm_kernel<bf16> grid=120 ")],
    ids=lambda v: "x".join(map(str, v)) if isinstance(v, tuple) else "")
def test_automatic_bf16_tile_width(mhr, shape, want):
    """The single-CTA bf16 kernel takes 128-column tiles when they put more
    CTAs to work in one round than 256-column ones: 1024^3 (64 tiles against
    32), 256 x 256 x 8192 (4 tiles in clusters of 8 against 2), 768^3 (36
    against 18); 1536 x 2560 x 512 keeps 256 columns (120 tiles; 240 narrow
    ones would need two rounds on 152 SMs). Integer inputs bit-exact against
    the oracle on sampled entries."""
    import torch

    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("tile counts stated for 152 SMs")
    M, N, K = shape
    A, B, Ab, Bb = operands(M, N, K, 4311 + K, "int", "bf16")
    C = DeviceCall("bf16", A, B, Ab, Bb).run(mhr).result()
    label = mhr.gemm_testing_last_main_kernel()
    assert label.startswith(want), (label, want)
    rows, cols = sample_indices(M, N, 4311, rows=(0, M // 2 + 1, M - 1), cols=(0, N - 1))
    ref = oracle.gemm_entries(A, B, rows, cols, M, N, K)[0]
    assert np.array_equal(C[rows, cols], ref)


def test_automatic_3xtf32_cluster_sizes(mhr):
    """After a pre-pass, 3xTF32 problems in the cluster split's domain run
    128-column tiles in the largest clusters that fit: 512 x 512 x 8192 has
    16 tiles, for which sixteen clusters of 8 do not fit at once, so it takes
    clusters of 6 (96 CTAs), whose ranks each sum a sixth of the tile's
    float4s rather than whole rows; 256 x 512 x 4096 (8 tiles) takes clusters
    of 8. Integer inputs bit-exact against the oracle on sampled entries."""
    import torch

    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("tile counts stated for 152 SMs")
    old = mhr.gemm_testing_set_cta_pair_mode(1)
    old_split = mhr.gemm_testing_set_split_mode(1)  # the pre-pass
    try:
        for (M, N, K), want in (((512, 512, 8192), "tc_gemm_kernel<3xtf32,cluster-K> grid=96 "),
                                ((256, 512, 4096), "tc_gemm_kernel<3xtf32,cluster-K> grid=64 ")):
            A, B, _, _ = operands(M, N, K, 4411 + K, "int", "3xtf32")
            C = DeviceCall("3xtf32", A, B).run(mhr).result()
            label = mhr.gemm_testing_last_main_kernel()
            assert label.startswith(want), (label, want)
            rows, cols = sample_indices(M, N, 4411, rows=(0, M // 2 + 1, M - 1), cols=(0, N - 1))
            ref = oracle.gemm_entries(A, B, rows, cols, M, N, K)[0]
            assert np.array_equal(C[rows, cols], ref)
    finally:
        mhr.gemm_testing_set_split_mode(old_split)
        mhr.gemm_testing_set_cta_pair_mode(old)


@pytest.mark.usefixtures("full_width_tiles")
def test_workspace_fallback_splits_in_kernel(mhr):
    """Operands one element off 16-byte alignment cannot be their own big
    parts, so the split runs in a pre-pass into the workspace. When that
    workspace cannot be allocated (a cap set by a test hook stands in for an
    allocation failure), gemm_f32_3xtf32 splits inside the CTA-pair kernel
    instead and returns the same C bit for bit."""
    A, B, _, _ = operands(300, 520, 1000, 3301, "normal", "3xtf32")
    old = mhr.gemm_testing_set_cta_pair_mode(2)
    try:
        ref = DeviceCall("3xtf32", A, B, offset=1).run(mhr).result()
        assert mhr.gemm_testing_last_main_kernel().startswith("tc_gemm_pair_kernel<3xtf32> ")
        with_prepass = mhr.gemm_testing_last_launches()  # split pre-pass, zeroing, main kernel
        old_limit = mhr.gemm_testing_set_workspace_limit(0)
        try:
            C = DeviceCall("3xtf32", A, B, offset=1).run(mhr).result()
            assert mhr.gemm_testing_last_main_kernel().startswith(
                "tc_gemm_pair_kernel<3xtf32,split> ")
            assert mhr.gemm_testing_last_launches() == with_prepass - 1  # no pre-pass
        finally:
            mhr.gemm_testing_set_workspace_limit(old_limit)
    finally:
        mhr.gemm_testing_set_cta_pair_mode(old)
    assert np.array_equal(C, ref)


def test_simt_split_k(mhr):
    """The SIMT kernel splits every tile along K when a partial last round of
    blocks would waste more than the split costs; both halves add into a
    zeroed C. 2560 x 2048 is 320 tiles of 128 x 128 (more than two blocks on
    each of the SMs); K = 1030 is ragged. Integer inputs must match the
    oracle bit for bit, real ones within tolerance and bitwise repeatably."""
    M, N, K = 2560, 2048, 1030
    A, B, _, _ = operands(M, N, K, 3401, "int", "f32")
    call = DeviceCall("f32", A, B)
    C = call.run(mhr).result()
    assert mhr.gemm_testing_last_main_kernel().startswith("simt_f32_kernel<split-K> grid=640 ")
    assert np.array_equal(C, oracle.gemm(A, B))
    A, B, _, _ = operands(M, N, K, 3402, "normal", "f32")
    call = DeviceCall("f32", A, B, ldc=N + 1)  # scalar atomic adds
    C = call.run(mhr).result()
    Cref, S = oracle.gemm(A, B, with_abs=True)
    assert normalised_error(C, Cref, S) <= TOL["f32"]
    assert np.array_equal(call.run(mhr).result(), C)


@pytest.mark.parametrize("shape,mode,label", [
    ((2048, 2560, 1032), 2, "simt_f32_kernel<wide,split-K> grid=320 "),
    ((2048, 2560, 1032), 0, "simt_f32_kernel<split-K> grid=640 "),
    ((2048, 4864, 64), 0, "simt_f32_kernel<wide> grid=304 "),
    ((2048, 4864 + 4, 64), 2, "simt_f32_kernel grid="),
    ((2048, 2560, 1032), 2, "simt_f32_kernel<wide,split-K> grid=320 "),
    ((2048, 2048, 512), 0, "simt_f32_kernel<wide> grid=128 "),
    ((512, 4864, 1024), 0, "simt_f32_kernel<wide,split-K> grid=152 "),
    ((2048, 2560, 1000), 0, "simt_f32_kernel grid=320 "),
    ((2048, 2560, 1000), 2, "simt_f32_kernel<wide> grid=160 "),
    ((1024, 2048, 512), 0, "simt_f32_kernel grid=")],
    ids=["160-tiles-split-forced", "160-tiles-auto", "304-tiles", "ragged-n-standard",
         "160-tiles-padded-ld", "128-tiles", "76-tiles-split", "k1000-auto", "k1000-forced",
         "64-tiles-standard"])
def test_simt_wide_tiles(mhr, shape, mode, label, request):
    """Aligned problems whose sizes are multiples of 128 x 256 x 8 can take
    the wide-tile SIMT kernel (8 x 16 outputs per thread, no masks), alone or
    on K halves added into a zeroed C. The automatic choice takes it when its
    queue of blocks per SM, at 11/6 of a 128 x 128 block's time per block, is
    the shorter: 128 and 304 tiles unsplit, 76 tiles on K halves; 160 tiles
    (two rounds) stay on the 128 x 128 kernel, split along K at K = 1032 and
    whole at K = 1000. Mode 2 forces the wide kernel; N one vector wider, or
    64 tiles, leave the shape to the masked kernel.
    The padded case pads every leading dimension by a multiple of 4 with NaN
    in the pads: a read outside the logical matrices poisons C, a write outside
    C breaks its guard band. Integer inputs bit-exact against the oracle,
    real inputs within tolerance and bitwise repeatable."""
    M, N, K = shape
    lds = {}
    if request.node.callspec.id.endswith("padded-ld"):
        lds = dict(lda=K + 4, ldb=N + 8, ldc=N + 4)
    old = mhr.gemm_testing_set_simt_wide_mode(mode)
    try:
        A, B, _, _ = operands(M, N, K, 3601 + K, "int", "f32")
        C = DeviceCall("f32", A, B, **lds).run(mhr).result()
        assert mhr.gemm_testing_last_main_kernel().startswith(label)
        assert np.array_equal(C, oracle.gemm(A, B))
        A, B, _, _ = operands(M, N, K, 3602 + K, "normal", "f32")
        call = DeviceCall("f32", A, B, **lds)
        C = call.run(mhr).result()
        Cref, S = oracle.gemm(A, B, with_abs=True)
        assert normalised_error(C, Cref, S) <= TOL["f32"]
        assert np.array_equal(call.run(mhr).result(), C)
    finally:
        mhr.gemm_testing_set_simt_wide_mode(old)


@pytest.mark.parametrize("shape,ldb,ldc,offset", [
    ((300, 522, 200), 522, 522, 0),      # B and C 8 bytes wide, A 16; ragged last group
    ((300, 522, 200), 522, 522, 2),      # every operand 8-byte aligned only
    ((300, 520, 200), 522, 521, 0),      # B 8 bytes wide, C scalar
    ((300, 520, 200), 521, 522, 0),      # B scalar, C 8 bytes wide
    ((1280, 2050, 1024), 2050, 2050, 0),  # K halves: 8-byte atomic adds into C
    ((256, 258, 512), 258, 258, 0)],     # a cluster per tile, 8-byte stores of the sums
    ids=["b2c2", "all8", "b2c1", "b1c2", "b2c2-split", "b2c2-cluster"])
def test_simt_eight_byte_rows(mhr, shape, ldb, ldc, offset):
    """Leading dimensions that are even but not multiples of 4 (C3's 2050),
    or operands 8 bytes off 16-byte alignment, give the SIMT kernel 8-byte
    loads of B and stores of C; odd ones scalar. Integer inputs bit-exact
    against the oracle, real inputs within tolerance and bitwise repeatable;
    the guard band of C's padding stays untouched."""
    M, N, K = shape
    A, B, _, _ = operands(M, N, K, 3701 + K, "int", "f32")
    C = DeviceCall("f32", A, B, ldb=ldb, ldc=ldc, offset=offset).run(mhr).result()
    assert mhr.gemm_testing_last_main_kernel().startswith("simt_f32_kernel")
    assert np.array_equal(C, oracle.gemm(A, B))
    A, B, _, _ = operands(M, N, K, 3702 + K, "normal", "f32")
    call = DeviceCall("f32", A, B, ldb=ldb, ldc=ldc, offset=offset)
    C = call.run(mhr).result()
    Cref, S = oracle.gemm(A, B, with_abs=True)
    assert normalised_error(C, Cref, S) <= TOL["f32"]
    assert np.array_equal(call.run(mhr).result(), C)


@pytest.mark.parametrize("shape,grid", [((256, 256, 256), 32), ((300, 520, 200), 120),
                                        ((129, 257, 100), 24)],
                         ids=["256-c8", "300x520x200-c8-empty-rank", "129x257x100-c4"])
def test_simt_cluster_split_k(mhr, shape, grid):
    """With few tiles the SIMT kernel runs a cluster of 8, 4 or 2 CTAs per
    tile, each on its own run of K-steps, and sums the partial tiles in
    distributed shared memory in rank order. 256^3: 4 tiles x 8 ranks of 4
    K-steps. 300 x 520 x 200: 15 tiles x 8 ranks; 25 K-steps in runs of 4
    leave rank 6 one step and rank 7 none. 129 x 257 x 100: 6 tiles x 4 ranks,
    K ragged (100 = 12 x 8 + 4). Integer inputs match the oracle bit for bit;
    real inputs (and C with an odd pitch: scalar stores) meet the tolerance,
    bitwise repeatably."""
    M, N, K = shape
    A, B, _, _ = operands(M, N, K, 3501 + K, "int", "f32")
    C = DeviceCall("f32", A, B).run(mhr).result()
    assert mhr.gemm_testing_last_main_kernel().startswith(
        f"simt_f32_kernel<cluster-K> grid={grid} ")
    assert np.array_equal(C, oracle.gemm(A, B))
    A, B, _, _ = operands(M, N, K, 3502 + K, "normal", "f32")
    call = DeviceCall("f32", A, B, ldc=N + 1)
    C = call.run(mhr).result()
    Cref, S = oracle.gemm(A, B, with_abs=True)
    assert normalised_error(C, Cref, S) <= TOL["f32"]
    assert np.array_equal(call.run(mhr).result(), C)


@pytest.mark.parametrize("N", [182, 195, 1], ids=lambda n: f"N{n}")
def test_ragged_n_with_tma_aligned_c(mhr, path, N):
    """C 16-byte aligned with ldc % 4 == 0 but N % 4 != 0: C's padding columns
    must keep their guard values (a TMA store clips only in 16-byte units, so
    such C must not be written with TMA stores). Found by the random sweep."""
    ldc = (N + 3) // 4 * 4 + 4
    check_full(mhr, path, 300, N, 150, seed=3501 + N, ldc=ldc)
    check_full(mhr, path, 97, N, 1000, seed=3601 + N, dist="int", ldc=ldc)


@pytest.mark.parametrize("shape", [(130, 264, 77), (257, 90, 200), (40, 45, 13)],
                         ids=lambda s: "x".join(map(str, s)))
def test_bf16_tma_operands_with_ragged_extents(mhr, shape):
    """bf16 operands whose pitches are TMA-aligned (lda, ldb multiples of 8)
    while K or N is not a multiple of 8, with NaN in every padding element: the
    TMA loads must stop at the logical extent (a NaN read would poison C)."""
    M, N, K = shape
    for mode in (1, 2):
        old = mhr.gemm_testing_set_cta_pair_mode(mode)
        try:
            check_full(mhr, "bf16", M, N, K, seed=3701 + K, lda=(K + 7) // 8 * 8,
                       ldb=(N + 7) // 8 * 8 + 8)
        finally:
            mhr.gemm_testing_set_cta_pair_mode(old)
