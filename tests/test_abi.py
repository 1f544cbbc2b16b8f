"""The C-ABI library: it builds, loads, exports every declared symbol, and
rejects bad arguments before touching the GPU (CPU only: no compute calls)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def lib():
    from memory_hierarchy_reuse_gb300 import build as b

    b.build()
    import memory_hierarchy_reuse_gb300 as m

    m.load()
    return m


def declared_functions():
    names = []
    for h in sorted(os.listdir(INCLUDE)):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(INCLUDE, h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b(\w+)\s*\([^;{]*\)\s*;", text, flags=re.M)
    return names


def test_headers_declare_the_abi():
    names = set(declared_functions())
    assert {"gemm_f32", "gemm_f32_3xtf32", "gemm_bf16_f32acc", "gemm_check",
            "gemm_status_string", "gemm_release", "gemm_version"} <= names


def test_every_declared_symbol_is_exported(lib):
    exported = subprocess.run(["nm", "-D", "--defined-only", lib.LIB_PATH], capture_output=True,
                              text=True, check=True).stdout
    syms = {line.split()[-1] for line in exported.splitlines() if " T " in line}
    for name in declared_functions():
        assert name in syms, name
        assert hasattr(ctypes.CDLL(lib.LIB_PATH), name)
    # nothing else leaks out of the library's own code
    assert {s for s in syms if s.startswith("gemm")} == set(declared_functions())
    assert set(lib.EXPORTS) == set(declared_functions())


def test_version_and_strings(lib):
    assert lib.gemm_version() == 10000
    assert lib.gemm_status_string(0) == "MHR_OK"
    for code in range(1, 5):
        assert lib.gemm_status_string(code).startswith("MHR_ERR")
    assert lib.gemm_status_string(99) == "unknown mhr_status"


@pytest.mark.parametrize("entry", ["gemm_f32", "gemm_f32_3xtf32", "gemm_bf16_f32acc",
                                   "gemm_f32_3xtf32_noalloc", "ladder0", "ladder2"])
def test_argument_validation_without_gpu(lib, entry):
    if entry.startswith("ladder"):
        rung = int(entry[-1])
        f = lambda *a: lib.gemm_f32_ladder(rung, *a)  # noqa: E731
    else:
        f = getattr(lib, entry)
    P, Q, R = 0x10000, 0x20000000, 0x40000000  # fake, disjoint, 16-byte aligned addresses
    bad = [
        (P, Q, R, -1, 4, 4, 4, 4, 4),          # negative M
        (P, Q, R, 4, -1, 4, 4, 4, 4),          # negative N
        (P, Q, R, 4, 4, -1, 4, 4, 4),          # negative K
        (None, Q, R, 4, 4, 4, 4, 4, 4),        # null A
        (P, None, R, 4, 4, 4, 4, 4, 4),        # null B
        (P, Q, None, 4, 4, 4, 4, 4, 4),        # null C
        (P, Q, R, 4, 4, 8, 7, 4, 4),           # lda < K
        (P, Q, R, 4, 8, 4, 4, 7, 8),           # ldb < N
        (P, Q, R, 4, 8, 4, 4, 8, 7),           # ldc < N
        (P, Q, P + 8, 4, 4, 4, 4, 4, 4),       # C overlaps A
        (P, Q, Q + 4, 4, 4, 4, 4, 4, 4),       # C overlaps B
        (P, Q, R, 1 << 40, 4, 4, 4, 4, 4),     # M too large
        (P, Q, R, 4, 4, 4, 4, 4, 1 << 62),     # extent overflows
    ]
    for args in bad:
        assert f(*args, None) == lib.MHR_ERR_INVALID_ARG, args
    # empty products are valid no-ops, even with null pointers
    assert f(None, None, None, 0, 5, 5, 5, 5, 5, None) == lib.MHR_OK
    assert f(None, None, None, 5, 0, 5, 5, 5, 5, None) == lib.MHR_OK
    # K == 0 needs C but not A or B; it is checked, then needs the device
    assert f(None, None, None, 2, 2, 0, 0, 0, 2, None) == lib.MHR_ERR_INVALID_ARG


def test_ladder_rejects_unknown_rungs_and_huge_m(lib):
    P, Q, R = 0x10000, 0x20000000, 0x40000000
    for rung in (-1, 3):
        assert lib.gemm_f32_ladder(rung, P, Q, R, 4, 4, 4, 4, 4, 4, None) == lib.MHR_ERR_INVALID_ARG
    assert lib.gemm_f32_ladder(0, P, Q, 1 << 45, 65535 * 16 + 1, 1, 1, 1, 1, 1, None) == \
        lib.MHR_ERR_INVALID_ARG


def test_oracle_and_library_are_independent():
    """Neither side imports or links the other."""
    pkg = os.path.join(ROOT, "memory_hierarchy_reuse_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in re.sub(r"(#|//).*", "", text).lower(), f
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith((".py", ".c", ".h")):
            text = open(os.path.join(ROOT, "oracle", f)).read()
            assert "memory_hierarchy_reuse_gb300" not in text and "mhr_" not in text, f
