"""Helpers shared by the GPU parity tests: seeded operands, a call through the
C ABI on device buffers with poisoned padding, and the comparison with the CPU
oracle by the normalised error max |C - C_ref| / sum_k |A_ik||B_kj|."""
from __future__ import annotations

import contextlib
import ctypes

import numpy as np

import seeded_inputs as si

# Tolerances on the normalised error (fp32 paths and bf16 against the oracle
# on the bf16-rounded inputs).
TOL = {"f32": 1e-5, "3xtf32": 1e-5, "bf16": 1e-2}
ENTRY = {"f32": "gemm_f32", "3xtf32": "gemm_f32_3xtf32", "bf16": "gemm_bf16_f32acc"}
GUARD = np.float32(-7.25)  # written into C's padding; must survive every call


def operands(M, N, K, seed, dist, path):
    """fp32 A (M x K), B (K x N) as the kernel sees them (bf16-rounded for the
    bf16 path), plus the bf16 bit patterns when path == 'bf16'."""
    A = si.matrix(M, K, seed, dist)
    B = si.matrix(K, N, seed + 1, dist)
    if path == "bf16":
        ab, A = si.bf16_rne(A)
        bb, B = si.bf16_rne(B)
        return A.reshape(M, K), B.reshape(K, N), ab.reshape(M, K), bb.reshape(K, N)
    return A, B, None, None


class DeviceCall:
    """Device copies of the operands (optionally padded with NaN and/or shifted
    off 16-byte alignment) and an output buffer with guard-filled padding."""

    def __init__(self, path, A, B, Ab=None, Bb=None, lda=None, ldb=None, ldc=None, offset=0):
        import torch

        self.torch = torch
        self.path = path
        M, K = A.shape
        N = B.shape[1]
        self.M, self.N, self.K = M, N, K
        self.lda = lda or K
        self.ldb = ldb or N
        self.ldc = ldc or N
        if path == "bf16":
            a_host = si.padded(Ab, self.lda, fill=0) if K else Ab
            b_host = si.padded(Bb, self.ldb, fill=0) if N else Bb
            # bf16 NaN pattern in the pads
            if self.lda > K:
                a_host[:, K:] = 0x7FC1
            if self.ldb > N:
                b_host[:, N:] = 0x7FC1
            a_t = torch.from_numpy(a_host.view(np.int16).copy())
            b_t = torch.from_numpy(b_host.view(np.int16).copy())
        else:
            a_t = torch.from_numpy(si.padded(A, self.lda))
            b_t = torch.from_numpy(si.padded(B, self.ldb))
        self.a_store = self._shifted(a_t, offset)
        self.b_store = self._shifted(b_t, offset)
        c_host = np.full((M, self.ldc), GUARD, np.float32)
        c_host[:, :N] = np.nan  # every entry of C must be written
        self.c_host_init = c_host
        self.c_store = self._shifted(torch.from_numpy(c_host.copy()), offset)

    def _shifted(self, t, offset):
        """Copy t to the device starting `offset` elements into a fresh buffer."""
        torch = self.torch
        flat = t.reshape(-1)
        buf = torch.empty(flat.numel() + offset + 16, dtype=t.dtype, device="cuda")
        view = buf[offset:offset + flat.numel()]
        view.copy_(flat.cuda())
        return view

    def run(self, lib, stream=None, check=True):
        rc = getattr(lib, ENTRY[self.path])(self.a_store.data_ptr(), self.b_store.data_ptr(),
                                            self.c_store.data_ptr(), self.M, self.N, self.K,
                                            self.lda, self.ldb, self.ldc, stream)
        assert rc == lib.MHR_OK, lib.gemm_status_string(rc)
        if check:
            assert lib.gemm_check(stream) == lib.MHR_OK
        return self

    def result(self):
        c = self.c_store.cpu().numpy().reshape(self.M, self.ldc)
        # guard band: nothing outside the logical M x N block was written
        assert np.array_equal(c[:, self.N:], self.c_host_init[:, self.N:])
        return np.ascontiguousarray(c[:, :self.N])


def normalised_error(C, Cref, S):
    """max |C - Cref| / S over entries with S > 0; entries with S == 0 must match exactly."""
    C = C.astype(np.float64)
    Cref = Cref.astype(np.float64)
    assert np.all(np.isfinite(C)), "non-finite output"
    zero = S == 0
    if np.any(zero):
        assert np.array_equal(C[zero], Cref[zero])
    if np.all(zero):
        return 0.0
    return float(np.max(np.abs(C - Cref)[~zero] / S[~zero]))


def sample_indices(M, N, seed, n_random=4096, rows=(), cols=()):
    """Sampled output coordinates: random entries plus whole chosen rows/cols."""
    rng = np.random.default_rng(seed)
    r = [rng.integers(0, M, n_random)]
    c = [rng.integers(0, N, n_random)]
    for row in rows:
        r.append(np.full(N, row))
        c.append(np.arange(N))
    for col in cols:
        r.append(np.arange(M))
        c.append(np.full(M, col))
    return np.concatenate(r).astype(np.int64), np.concatenate(c).astype(np.int64)


@contextlib.contextmanager
def pair_tile_n(mhr, columns):
    """Run the enclosed calls with the 3xTF32 CTA-pair tiles forced to
    `columns` wide (0: the planner's choice)."""
    old = mhr.gemm_testing_set_pair_tile_n(columns)
    try:
        yield
    finally:
        mhr.gemm_testing_set_pair_tile_n(old)
