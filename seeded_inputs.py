"""Seeded synthetic matrices shared by the CPU oracle and the CUDA path.

This module holds no matrix-multiply arithmetic: it only draws numbers. Both
sides of every parity check take their inputs from here, so that the oracle and
the kernels see bit-identical operands.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014), used counter-style: draw ``i`` of stream
``seed`` is ``mix(seed + (i + 1) * GOLDEN)`` where ``mix`` is the published
64-bit finaliser. It is written here with numpy uint64 arithmetic (wrapping
modulo 2**64), so the stream is identical on x86_64 and aarch64 and does not
depend on the torch or numpy RNG versions.

Element ``(r, c)`` of a ``rows x cols`` matrix is draw ``r * cols + c`` (two
draws, ``2i`` and ``2i + 1``, for the normal distribution), so a matrix's
values do not depend on the leading dimension it is later stored with.

Distributions (the workloads' three):

* ``uniform``: ``(x >> 40) * 2**-23 - 1``, i.e. uniform on [-1, 1) with step
  2**-23; every value is exact in fp32.
* ``normal``: Box-Muller in float64 from two draws, rounded once to fp32.
* ``int``: ``(x >> 32) mod 5 - 2``, i.e. integers in {-2, ..., 2}.

``bf16_rne`` rounds fp32 samples to bfloat16 (round to nearest, ties to even)
and returns both the 16-bit patterns and their exact fp32 widening.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Draws ``start .. start+count-1`` of stream ``seed`` as uint64."""
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + idx * GOLDEN)


def _fill(out: np.ndarray, seed: int, dist: str, s: int, e: int) -> None:
    """Elements s .. e-1 of the matrix (draws depend only on the index)."""
    if dist == "uniform":
        x = splitmix64(seed, s, e - s)
        out[s:e] = ((x >> np.uint64(40)).astype(np.float64) * 2.0 ** -23 - 1.0)
    elif dist == "int":
        x = splitmix64(seed, s, e - s)
        out[s:e] = ((x >> np.uint64(32)) % np.uint64(5)).astype(np.int64) - 2
    elif dist == "normal":
        x = splitmix64(seed, 2 * s, 2 * (e - s))
        u1 = ((x[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
        u2 = (x[1::2] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
        out[s:e] = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    else:
        raise ValueError(f"unknown distribution {dist!r}")


def _threads() -> int:
    try:
        return max(1, min(16, len(os.sched_getaffinity(0))))
    except (AttributeError, OSError):
        return max(1, min(16, os.cpu_count() or 1))


def matrix(rows: int, cols: int, seed: int, dist: str = "uniform") -> np.ndarray:
    """A C-contiguous float32 ``rows x cols`` matrix drawn from ``dist``.

    Element ``(r, c)`` depends only on its index ``r * cols + c``, so large
    matrices are filled in chunks on several host threads with identical
    results."""
    if dist not in ("uniform", "int", "normal"):
        raise ValueError(f"unknown distribution {dist!r}")
    n = rows * cols
    out = np.empty(n, dtype=np.float32)
    chunks = [(s, min(n, s + _CHUNK)) for s in range(0, n, _CHUNK)]
    if len(chunks) > 1 and _threads() > 1:
        with ThreadPoolExecutor(max_workers=_threads()) as ex:
            list(ex.map(lambda se: _fill(out, seed, dist, *se), chunks))
    else:
        for s, e in chunks:
            _fill(out, seed, dist, s, e)
    return out.reshape(rows, cols)


def bf16_rne(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Round finite fp32 values to bf16, ties to even.

    Returns ``(bits, widened)``: the uint16 bf16 patterns and the same values
    widened back to fp32 (exact).
    """
    src = np.ascontiguousarray(x, dtype=np.float32)
    flat = src.reshape(-1).view(np.uint32)
    bits = np.empty(flat.size, dtype=np.uint16)

    def one(se):
        s, e = se
        u = flat[s:e].astype(np.uint64)
        bias = ((u >> np.uint64(16)) & np.uint64(1)) + np.uint64(0x7FFF)
        bits[s:e] = ((u + bias) >> np.uint64(16)).astype(np.uint16)

    chunks = [(s, min(flat.size, s + _CHUNK)) for s in range(0, flat.size, _CHUNK)]
    if len(chunks) > 1 and _threads() > 1:
        with ThreadPoolExecutor(max_workers=_threads()) as ex:
            list(ex.map(one, chunks))
    else:
        for se in chunks:
            one(se)
    bits = bits.reshape(src.shape)
    widened = (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
    return bits, widened


def padded(x: np.ndarray, ld: int, fill: float = np.nan) -> np.ndarray:
    """Store ``x`` (rows x cols) in a row-major buffer of leading dimension
    ``ld >= cols``; the pad columns hold ``fill`` (NaN by default, so that any
    read of them poisons a result)."""
    rows, cols = x.shape
    if ld < cols:
        raise ValueError("ld < cols")
    buf = np.full((rows, ld), fill, dtype=x.dtype)
    buf[:, :cols] = x
    return buf
