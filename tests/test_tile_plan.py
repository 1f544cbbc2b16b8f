"""The tile-width planners of the 3xTF32 kernels and the choice between the
two SIMT fp32 kernels (host arithmetic in libmhr_gemm.so, no GPU needed):
which width or kernel they pick for the listed workloads and for shapes
measured on GB300 (152 SMs, 76 co-resident CTA pairs), and that every pick
is one the kernels support."""
import numpy as np
import pytest

import memory_hierarchy_reuse_gb300 as mhr

SMS = 152
CLUSTERS = SMS // 2  # CTA pairs


@pytest.fixture(scope="module")
def lib():
    try:
        return mhr.load()
    except OSError as e:  # the library is built by __graft_entry__.build()
        pytest.skip(f"libmhr_gemm.so not built: {e}")


@pytest.mark.parametrize("shape,c_tma,want", [
    ((4096, 4096, 4096), True, 256),   # 256 tiles: 3 rounds + a split one, whole-width best
    ((8192, 8192, 8192), True, 256),   # 1024 tiles: 13 rounds + a split one
    ((3000, 2048, 1000), True, 256),
    # 3000 x 2050 x 1000 with C's odd pitch (register stores): 108 tiles of 256
    # columns need a K-split last round ending in atomic adds; 144 tiles of 176
    # columns fill two whole rounds
    ((3000, 2050, 1000), False, 176),
])
def test_planned_width_for_listed_workloads(lib, shape, c_tma, want):
    assert mhr.gemm_testing_plan_pair_tile_n(*shape, CLUSTERS, c_tma) == want


def test_planned_width_is_supported(lib):
    rng = np.random.default_rng(11)
    for _ in range(400):
        M, N = (int(x) for x in rng.integers(1, 20000, size=2))
        K = int(rng.integers(1, 9000))
        clusters = int(rng.integers(1, 80))
        for c_tma in (False, True):
            bn = mhr.gemm_testing_plan_pair_tile_n(M, N, K, clusters, c_tma)
            assert 128 <= bn <= 256 and bn % 16 == 0, (M, N, K, clusters, bn)
            if c_tma:
                assert bn % 32 == 0, (M, N, K, clusters, bn)


def test_no_clusters_keeps_full_width(lib):
    assert mhr.gemm_testing_plan_pair_tile_n(4096, 4096, 4096, 0, True) == 256


@pytest.mark.parametrize("shape,want", [
    # 256^3: 4 tiles of 128 columns in K halves keep 8 SMs busy; 16 tiles of 32
    # columns in K halves keep 32 busy, each loading less and storing a
    # quarter of the epilogue
    ((256, 256, 256), 32),
    ((300, 520, 1000), 32),
    ((1024, 1024, 1024), 128),   # 64 tiles in K halves already fill 128 SMs
    ((1536, 1536, 1536), 128),   # 144 tiles: one round
    ((512, 512, 8192), 128),     # the cluster split's domain (whole tiles only)
])
def test_single_cta_planned_width(lib, shape, want):
    for c_tma in (False, True):
        assert mhr.gemm_testing_plan_single_tile_n(*shape, SMS, c_tma) == want


def test_single_cta_planned_width_is_supported(lib):
    rng = np.random.default_rng(12)
    for _ in range(400):
        M, N = (int(x) for x in rng.integers(1, 4000, size=2))
        K = int(rng.integers(1, 9000))
        sms = int(rng.integers(1, 160))
        for c_tma in (False, True):
            bn = mhr.gemm_testing_plan_single_tile_n(M, N, K, sms, c_tma)
            assert bn in (32, 64, 96, 128), (M, N, K, sms, bn)
    assert mhr.gemm_testing_plan_single_tile_n(256, 256, 256, 0, True) == 128


@pytest.mark.parametrize("shape,want", [
    # GB300, whole calls, the 128 x 128 kernel against the 128 x 256 one:
    ((4096, 4096, 4096), 2),   # 2407 / 2195 us
    ((4096, 4096, 1024), 2),   # 613 / 578
    ((2048, 2048, 2048), 1),   # 363 / 318
    ((3072, 3072, 1000), 1),   # 347 / 314
    ((3584, 2304, 512), 1),    # 185 / 167
    ((8192, 8192, 8192), 1),
    ((3072, 2048, 1000), 0),   # 265 / 310: 192 wide tiles, two rounds, K too short for halves
    ((2560, 2560, 1000), 0),   # 265 / 314
    ((2048, 2560, 2048), 0),   # 462 / 483
    ((2048, 2560, 1032), 0),   # 245 / 254
    ((1024, 2048, 512), 0),    # 64 wide tiles: fewer than half the SMs
    ((3000, 2048, 1000), 0),   # not a multiple of 128 rows
    ((2048, 2050, 1000), 0),
    ((2048, 2048, 1001), 0),
])
def test_simt_wide_plan(lib, shape, want):
    assert mhr.gemm_testing_plan_simt_wide(*shape, SMS) == want


def test_simt_wide_plan_is_a_queue_model(lib):
    """Whatever the shape and SM count, the wide kernel is chosen only where
    its sizes allow it and its tiles fill at least half of the SMs, with K
    halves only where each half keeps at least 64 steps of 8."""
    rng = np.random.default_rng(13)
    for _ in range(2000):
        a, b = (int(x) for x in rng.integers(1, 64, size=2))
        M, N, K = 128 * a, 256 * b, 8 * int(rng.integers(1, 1200))
        sms = int(rng.integers(1, 200))
        plan = mhr.gemm_testing_plan_simt_wide(M, N, K, sms)
        assert plan in (0, 1, 2)
        if plan == 2:
            assert K >= 1024
        if plan:
            assert 2 * a * b >= sms, (M, N, K, sms)
        assert mhr.gemm_testing_plan_simt_wide(M + 1, N, K, sms) == 0
        assert mhr.gemm_testing_plan_simt_wide(M, N + 4, K, sms) == 0
    assert mhr.gemm_testing_plan_simt_wide(4096, 4096, 4096, 0) == 0
