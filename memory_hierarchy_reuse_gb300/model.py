"""Counting model of the method: FLOPs, global loads, arithmetic intensity,
roofline, and the pages' thread/tile index map.

Host-side arithmetic only (no GPU). The bench uses it for the algorithmic
FLOPs and bytes it divides by measured times; the tests pin it to the figures
the pages print.

* naive loads: every output reads a row of A and a column of B, 2K elements,
  so 2MNK in total (2N^3 for squares) -- "CUDA 深入浅出（二）", section
  "naive kernel 怎么读数据"; "矩阵乘法 tiling", section 一.
* tiled loads: a BM x BN output tile walks K in steps, loading a BM x BK strip
  of A and a BK x BN strip of B per step, so A is read ceil(N/BN) times and B
  ceil(M/BM) times: K (M ceil(N/BN) + N ceil(M/BM)) elements, which is 2N^3/T
  for T x T tiles of an N x N product -- "矩阵乘法 tiling", section 三;
  "CUDA 深入浅出（二）", section "推广到整个 N×N 矩阵"; "CUDA 编程系列之三",
  section 6.
* per-tile counts: 2T^3 (naive) versus 2T^2 (tiled) loads for one K step of
  one T x T tile -- "CUDA 深入浅出（二）", section "对一个 C_tile 数数".
* intensity of the tiled square kernel: T/4 FLOP/B in fp32 --
  "矩阵乘法 tiling", section 三.
* roofline: attainable = min(peak FLOP/s, bandwidth x intensity), ridge =
  peak / bandwidth -- "CUDA 编程系列之三", sections 1-3.
* index map: row = blockIdx.y * T + threadIdx.y, col = blockIdx.x * T +
  threadIdx.x (threadIdx.x runs along a row of C, so a warp's loads are
  consecutive) -- the ijyty.com page, step ②; "矩阵乘法 tiling", section 四.
"""
from __future__ import annotations


def cdiv(a: int, b: int) -> int:
    return -(-a // b)


def flops(M: int, N: int, K: int) -> int:
    """Multiply-adds counted as 2 FLOPs: 2MNK."""
    return 2 * M * N * K


def naive_loads(M: int, N: int, K: int) -> int:
    """Global element loads of the one-output-per-thread kernel."""
    return 2 * M * N * K


def tiled_loads(M: int, N: int, K: int, BM: int, BN: int | None = None) -> int:
    """Global element loads of A and B when each BM x BN output tile stages its
    row strip of A and column strip of B on chip once per K step."""
    BN = BM if BN is None else BN
    return K * (M * cdiv(N, BN) + N * cdiv(M, BM))


def tile_step_loads(T: int) -> dict:
    """Loads of one K step of one T x T output tile: naive 2T^3, tiled 2T^2."""
    return {"naive": 2 * T ** 3, "tiled": 2 * T ** 2, "ratio": T}


def tiled_intensity(T: int, elem_bytes: int = 4) -> float:
    """FLOP per byte of the square T x T tiled kernel: 2N^3 / (2N^3/T * bytes)."""
    return T / elem_bytes


def per_element_flops(T: int) -> int:
    """FLOPs one staged element serves: it meets T outputs, one multiply-add each."""
    return 2 * T


def ridge(peak_flops: float, bandwidth: float) -> float:
    return peak_flops / bandwidth


def attainable(peak_flops: float, bandwidth: float, intensity: float) -> float:
    return min(peak_flops, bandwidth * intensity)


def tile_coord(block_x: int, block_y: int, thread_x: int, thread_y: int, T: int) -> tuple[int, int]:
    """(row, col) of C owned by a thread of the T x T tiled kernel."""
    return block_y * T + thread_y, block_x * T + thread_x


def compulsory_bytes(M: int, N: int, K: int, in_bytes: int, out_bytes: int = 4) -> int:
    """Bytes that must cross HBM at least once: read A and B, write C."""
    return in_bytes * (M * K + K * N) + out_bytes * M * N


def split_bytes(M: int, N: int, K: int, a_big_written: bool = False) -> int:
    """HBM bytes of the 3xTF32 split pre-pass: read A and B (fp32) once, write
    A's small part and B's big and small parts (fp32 containers, K padded to
    4); A's big part too when TMA cannot read A itself as that part."""
    Kp = cdiv(K, 4) * 4
    return 4 * (M * K + K * N) + 4 * Kp * ((2 if a_big_written else 1) * M + 2 * N)
