"""Seeded random sweep of every path variant against the oracle (GB300 only).

Sixty cases with dimensions anywhere in 1..700, sixty with every dimension at
or next to a tile boundary (1, 8, 16, ..., 512, each +-1), twenty-four drawn
onto the schedules that split or widen tiles, and twenty-four small aligned
problems in the automatic mode (one launch with the split inside, at the tile
width it picks); and sixty-four larger ones on the host's tiling choices
(tiling_choice_cases), checked on sampled entries. Each draws a path variant (SIMT fp32; 3xTF32 in the automatic
mode, on the single-CTA kernel, on the CTA-pair kernel with the split
pre-pass, and with the split on chip; bf16 on either kernel), a shape,
padded leading dimensions (0 to 9 extra elements), an element offset that
breaks 16-byte alignment or not, and integer or real inputs. Integer inputs must
match the oracle bit for bit, real ones within the path's tolerance; the
padding of C must keep its guard value (checked by DeviceCall.result)."""
import numpy as np
import pytest

import oracle
from parity_util import TOL, DeviceCall, normalised_error, operands, sample_indices

pytestmark = pytest.mark.gpu

# (path, CTA-pair mode -- for f32 the SIMT kernel mode of gemm_testing_set_simt_wide_mode --,
#  split mode)
VARIANTS = [("f32", 0, 0), ("3xtf32", 0, 0), ("3xtf32", 1, 1), ("3xtf32", 1, 2), ("3xtf32", 2, 1),
            ("3xtf32", 2, 2), ("bf16", 1, 0), ("bf16", 2, 0)]


def cases(n=60, seed=20261202):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        v = VARIANTS[i % len(VARIANTS)]
        M, N, K = (int(x) for x in rng.integers(1, 701, 3))
        pads = [int(x) for x in rng.integers(0, 10, 3)]
        offset = int(rng.integers(0, 2))
        dist = "int" if rng.random() < 0.4 else ("normal" if rng.random() < 0.5 else "uniform")
        out.append((v, M, N, K, pads, offset, dist, 9000 + i))
    return out


EDGES = [1, 2, 3, 7, 8, 9, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 255, 256, 257,
         511, 512, 513]


def edge_cases(n=60, seed=20261203):
    """Shapes whose every dimension sits at or next to a tile, box or K-step
    boundary."""
    rng = np.random.default_rng(seed)
    out = []
    for v, M, N, K, pads, offset, dist, s in cases(n, seed):
        M, N, K = (EDGES[int(x)] for x in rng.integers(0, len(EDGES), 3))
        out.append((v, M, N, K, pads, offset, dist, s + 1000))
    return out


def schedule_cases(n=24, seed=20261204):
    """Shapes drawn to land on the schedules that split or widen tiles:
    aligned 128 x 256 x 8 multiples with 76-120 such tiles (the wide SIMT
    kernel, forced in every other such case, else the automatic choice
    between it and the 128 x 128 kernel), few single-CTA tiles with long K (clusters of 4 or 8 CTAs summing
    through distributed shared memory, 3xTF32 and bf16), and few SIMT tiles
    (clusters of 2-8). Alignment-preserving pads for the wide kernel; any
    pads and offsets otherwise."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        kind = i % 4
        dist = "int" if rng.random() < 0.5 else "normal"
        if kind == 0:
            while True:
                a, b = int(rng.integers(2, 17)), int(rng.integers(1, 21))
                if 76 <= a * b <= 120:
                    break
            M, N, K = 128 * a, 256 * b, 8 * int(rng.integers(1, 34))
            pads = [4 * int(x) for x in rng.integers(0, 3, 3)]
            out.append((("f32", 2 if i % 8 == 0 else 0, 0), M, N, K, pads, 0, dist, 9500 + i))
            continue
        M, N = (int(x) for x in rng.integers(1, 401, 2))
        K = {1: int(rng.integers(2048, 4501)), 2: int(rng.integers(4096, 8401)),
             3: int(rng.integers(16, 3001))}[kind]
        v = {1: ("3xtf32", 1, 1), 2: ("bf16", 1, 0), 3: ("f32", 0, 0)}[kind]
        pads = [int(x) for x in rng.integers(0, 10, 3)]
        out.append((v, M, N, K, pads, int(rng.integers(0, 2)), dist, 9500 + i))
    return out


def aligned_split_cases(n=24, seed=20261205):
    """Shapes for the in-kernel 3xTF32 split with A and B 16-byte aligned and
    leading dimensions multiples of 4, so that its converter warps read both
    operands with 16-byte loads, at random and at tile-boundary sizes, ragged
    N and K included."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        if i % 2:
            M, N, K = (EDGES[int(x)] for x in rng.integers(0, len(EDGES), 3))
        else:
            M, N, K = (int(x) for x in rng.integers(1, 1101, 3))
        # lda, ldb: the next multiple of 4, plus 0-2 more groups of 4
        pa, pb = ((-d) % 4 + 4 * int(rng.integers(0, 3)) for d in (K, N))
        dist = "int" if rng.random() < 0.4 else "normal"
        out.append((("3xtf32", 1 + (i % 3 == 0), 2), M, N, K, [pa, pb, int(rng.integers(0, 6))],
                    0, dist, 9700 + i))
    return out


def auto_small_cases(n=24, seed=20261206):
    """Small 3xTF32 problems (M N <= 2^18, K <= 2048) with A 16-byte aligned
    and lda a multiple of 4, in the automatic mode: one launch of the
    single-CTA kernel with the split inside, on 128-, 64- or 32-column tiles
    with clusters splitting K, whichever puts the most CTAs to work; B and C
    at any padding."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        while True:
            M, N = (int(x) for x in rng.integers(1, 700, 2))
            if M * N <= 1 << 18:
                break
        K = 4 * int(rng.integers(1, 513))
        pads = [4 * int(rng.integers(0, 3)), int(rng.integers(0, 10)), int(rng.integers(0, 10))]
        dist = "int" if rng.random() < 0.5 else "normal"
        out.append((("3xtf32", 0, 0), M, N, K, pads, 0, dist, 9800 + i))
    return out


@pytest.mark.parametrize("case", cases() + edge_cases() + schedule_cases() + aligned_split_cases() +
                         auto_small_cases(),
                         ids=lambda c: f"{c[0][0]}-{c[0][1]}{c[0][2]}-{c[1]}x{c[2]}x{c[3]}-{c[6]}")
def test_random_case(mhr, case):
    (path, pair_mode, split_mode), M, N, K, pads, offset, dist, seed = case
    A, B, Ab, Bb = operands(M, N, K, seed, dist, path)
    simt = path == "f32"
    old_pair = mhr.gemm_testing_set_cta_pair_mode(0 if simt else pair_mode)
    old_wide = mhr.gemm_testing_set_simt_wide_mode(pair_mode if simt else 0)
    old_split = mhr.gemm_testing_set_split_mode(split_mode)
    try:
        C = DeviceCall(path, A, B, Ab, Bb, lda=K + pads[0], ldb=N + pads[1], ldc=N + pads[2],
                       offset=offset).run(mhr).result()
        label = mhr.gemm_testing_last_main_kernel()
    finally:
        mhr.gemm_testing_set_split_mode(old_split)
        mhr.gemm_testing_set_simt_wide_mode(old_wide)
        mhr.gemm_testing_set_cta_pair_mode(old_pair)
    small_aligned = (offset == 0 and (K + pads[0]) % 4 == 0 and M * N <= 1 << 18 and K <= 2048)
    if path == "3xtf32" and (pair_mode, split_mode) == (0, 0) and small_aligned:
        assert label.startswith("tc_gemm_kernel<3xtf32,split,tma-a"), (case, label)
    if simt and pair_mode == 2 and offset == 0 and all(p % 4 == 0 for p in pads):
        assert label.startswith("simt_f32_kernel<wide"), (case, label)
    if dist == "int":
        assert np.array_equal(C, oracle.gemm(A, B)), case
    else:
        Cref, S = oracle.gemm(A, B, with_abs=True)
        assert normalised_error(C, Cref, S) <= TOL[path], case


def tiling_choice_cases(n=64, seed=20261207):
    """Shapes on the host's tiling choices, in the automatic mode of each:
    bf16 on the single-CTA kernel (256- or 128-column tiles, clusters of 4 to
    8 CTAs, K halves) or the pair kernel; 3xTF32 after the split pre-pass on
    the single-CTA kernel with long K (clusters of up to 16); SIMT fp32 with
    even pitches or 8-byte offsets (8-byte loads of B and stores of C); and
    SIMT on aligned 128 x 256 x 8 multiples, automatic or with the wide
    kernel forced."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        kind = i % 4
        pads = [int(x) for x in rng.integers(0, 10, 3)]
        offset = int(rng.choice([0, 0, 1, 2]))
        if kind == 0:
            v = ("bf16", 0, 0)
            M, N = (int(x) for x in rng.integers(64, 1600, 2))
            K = int(rng.integers(256, 9000))
        elif kind == 1:
            v = ("3xtf32", 1, 1)
            M, N = (int(x) for x in rng.integers(32, 1100, 2))
            K = int(rng.integers(1024, 9000))
        elif kind == 2:
            v = ("f32", 0, 0)
            M, N, K = (int(x) for x in rng.integers(1, 1400, 3))
            pads = [2 * int(x) for x in rng.integers(0, 4, 3)]
        else:
            v = ("f32", int(rng.choice([0, 2])), 0)
            M, N = 128 * int(rng.integers(1, 20)), 256 * int(rng.integers(1, 10))
            K = 8 * int(rng.integers(1, 200))
            pads = [4 * int(x) for x in rng.integers(0, 3, 3)]
            offset = 0
        dist = "int" if rng.random() < 0.5 else "normal"
        out.append((v, M, N, K, pads, offset, dist, 15000 + i))
    return out


@pytest.mark.parametrize("case", tiling_choice_cases(),
                         ids=lambda c: f"{c[0][0]}-{c[0][1]}{c[0][2]}-{c[1]}x{c[2]}x{c[3]}-{c[6]}")
def test_tiling_choice_case(mhr, case):
    """As test_random_case, at sizes where the oracle is taken on sampled
    entries (2048 random ones plus the first and last rows and columns):
    integer inputs bit-exact, real ones within the path's tolerance."""
    (path, mode, split_mode), M, N, K, pads, offset, dist, seed = case
    A, B, Ab, Bb = operands(M, N, K, seed, dist, path)
    simt = path == "f32"
    old_pair = mhr.gemm_testing_set_cta_pair_mode(0 if simt else mode)
    old_wide = mhr.gemm_testing_set_simt_wide_mode(mode if simt else 0)
    old_split = mhr.gemm_testing_set_split_mode(split_mode)
    try:
        C = DeviceCall(path, A, B, Ab, Bb, lda=K + pads[0], ldb=N + pads[1], ldc=N + pads[2],
                       offset=offset).run(mhr).result()
    finally:
        mhr.gemm_testing_set_split_mode(old_split)
        mhr.gemm_testing_set_simt_wide_mode(old_wide)
        mhr.gemm_testing_set_cta_pair_mode(old_pair)
    r, c = sample_indices(M, N, seed, n_random=2048, rows=(0, M - 1), cols=(0, N - 1))
    ref, S = oracle.gemm_entries(A, B, r, c, M, N, K)
    if dist == "int":
        assert np.array_equal(C[r, c], ref), case
    else:
        assert normalised_error(C[r, c], ref, S) <= TOL[path], case
