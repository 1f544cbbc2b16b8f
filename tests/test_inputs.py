"""The seeded input generator (CPU only)."""
import numpy as np

import seeded_inputs as si


def test_splitmix64_published_sequence():
    # SplitMix64 from state 0: the first outputs of the published reference
    # generator (Steele, Lea and Flood 2014; Vigna's splitmix64.c).
    got = [int(v) for v in si.splitmix64(0, 0, 3)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_counter_access_is_consistent():
    whole = si.splitmix64(7, 0, 100)
    assert np.array_equal(whole[40:60], si.splitmix64(7, 40, 20))


def test_distributions():
    u = si.matrix(300, 300, 1, "uniform")
    assert u.dtype == np.float32 and u.min() >= -1.0 and u.max() < 1.0
    assert abs(float(u.mean())) < 0.01
    # exact in fp32: multiples of 2^-23
    assert np.all((u.astype(np.float64) * 2 ** 23) == np.round(u.astype(np.float64) * 2 ** 23))
    n = si.matrix(300, 300, 2, "normal")
    assert abs(float(n.mean())) < 0.02 and abs(float(n.std()) - 1.0) < 0.02
    i = si.matrix(300, 300, 3, "int")
    assert set(np.unique(i).tolist()) == {-2.0, -1.0, 0.0, 1.0, 2.0}


def test_reproducible_and_seed_dependent():
    assert np.array_equal(si.matrix(50, 70, 9), si.matrix(50, 70, 9))
    assert not np.array_equal(si.matrix(50, 70, 9), si.matrix(50, 70, 10))
    # chunking does not change values: element (r, c) is draw r*cols + c
    big = si.matrix(3, 2_000_000, 4)
    assert big[2, 1_999_999] == si.matrix(1, 6_000_000, 4)[0, 5_999_999]


def test_bf16_rne():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -9, -2.5, 1.0 + 2 ** -9], np.float32)
    b, w = si.bf16_rne(x)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: even -> 1.0
    assert w.tolist() == [1.0, 1.0, 1.0 + 2 ** -7, -2.5, 1.0]
    assert b.tolist() == [0x3F80, 0x3F80, 0x3F81, 0xC020, 0x3F80]
