"""The counting model and index map, pinned to the figures the pages print
(tests/golden/pages_figures.json)."""
import json
import os

import pytest

from memory_hierarchy_reuse_gb300 import model

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_figures.json")))


def test_square_4096_block_32_traffic():
    g = GOLD["square_4096_block_32"]
    N, T, e = g["N"], g["block"], g["elem_bytes"]
    assert model.flops(N, N, N) / 1e9 == pytest.approx(g["gflop"], rel=5e-3)
    assert 2 * N * N * e / 2 ** 20 == g["inputs_mib"]
    naive = model.naive_loads(N, N, N)
    tiled = model.tiled_loads(N, N, N, T)
    assert naive / 1e8 == pytest.approx(g["naive_elements_1e8"], rel=5e-3)
    assert naive * e / 1e9 == pytest.approx(g["naive_gb"], rel=5e-3)
    assert tiled / 1e8 == pytest.approx(g["tiled_elements_1e8"], rel=5e-3)
    assert tiled * e / 1e9 == pytest.approx(g["tiled_gb"], rel=5e-3)
    assert naive == T * tiled  # the reuse factor is T, not T^2


def test_intensity():
    g = GOLD["intensity"]
    assert model.tiled_intensity(16) == g["block_16"]
    assert model.tiled_intensity(32) == g["block_32"]
    assert model.per_element_flops(32) == g["per_element_flop_block_32"]
    assert model.per_element_flops(32) / 4 == g["per_element_flop_per_byte_block_32"]
    # the whole-kernel intensity equals FLOPs over tiled bytes
    N = 1024
    assert model.flops(N, N, N) / (model.tiled_loads(N, N, N, 32) * 4) == pytest.approx(8.0)


def test_tile_step_counts():
    g = GOLD["tile_step_T4"]
    c = model.tile_step_loads(g["T"])
    assert c["tiled"] == g["tiled"] == g["a_tile"] + g["b_tile"]
    assert c["naive"] == g["naive"]
    assert c["naive"] // c["tiled"] == g["ratio"]


def test_whole_matrix_counts_square():
    # (N/T)^2 tiles x N/T steps x 2T^2 elements = 2N^3/T, for several T | N
    for N, T in [(8, 4), (64, 16), (96, 32), (4096, 128)]:
        assert model.tiled_loads(N, N, N, T) == (N // T) ** 3 * 2 * T * T == 2 * N ** 3 // T


def test_ragged_counts():
    # 3000 x 2050 x 1000 with 128 x 128 tiles: A read ceil(2050/128)=17 times,
    # B read ceil(3000/128)=24 times.
    assert model.tiled_loads(3000, 2050, 1000, 128) == 1000 * (3000 * 17 + 2050 * 24)


def test_index_map():
    g = GOLD["index_map"]
    assert model.tile_coord(g["block_x"], g["block_y"], g["thread_x"], g["thread_y"], g["T"]) == (
        g["row"], g["col"])
    # adjacent threadIdx.x -> adjacent columns (coalesced row access)
    r0, c0 = model.tile_coord(1, 2, 0, 1, 4)
    r1, c1 = model.tile_coord(1, 2, 1, 1, 4)
    assert r0 == r1 and c1 == c0 + 1


def test_phase_count():
    g = GOLD["n8_tile4_phases"]
    assert model.cdiv(g["N"], g["T"]) == g["phases"]


def test_roofline_examples():
    g = GOLD["generic_card"]
    assert model.attainable(g["peak_flops"], g["bandwidth"], g["naive_intensity"]) == pytest.approx(
        g["ceiling_flops"])
    assert g["peak_flops"] / g["naive_intensity"] == pytest.approx(g["needed_bandwidth"])
    h = GOLD["h100_ridge"]
    assert model.ridge(h["peak_flops"], h["bandwidth"]) == pytest.approx(h["ridge"], rel=0.01)
    # compute-bound above the ridge, bandwidth-bound below
    assert model.attainable(1.0, 1.0, 2.0) == 1.0
    assert model.attainable(1.0, 1.0, 0.5) == 0.5


def test_split_bytes():
    # 4096^3: read 2 x 64 MiB, write A_small, Bt_big, Bt_small (3 x 64 MiB),
    # and A_big as well when A cannot serve as it
    assert model.split_bytes(4096, 4096, 4096) == 5 * 4096 * 4096 * 4
    assert model.split_bytes(4096, 4096, 4096, a_big_written=True) == 6 * 4096 * 4096 * 4
    # K padded to a multiple of 4 in the written parts only
    assert model.split_bytes(3, 5, 7) == 4 * (3 * 7 + 7 * 5) + 4 * 8 * (3 + 2 * 5)
