"""The C ABI used from a plain C program (tests/c_abi/gemm_from_c.c): the
headers compile as strict C, the program links against libmhr_gemm.so and
the CUDA runtime (CPU), and on a GB300 its three calls reproduce the oracle
bit for bit on integer inputs (GPU)."""
import os
import shutil
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")
SRC = os.path.join(ROOT, "tests", "c_abi", "gemm_from_c.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _gcc():
    cc = shutil.which("gcc") or shutil.which("cc")
    if not cc:
        pytest.skip("no C compiler")
    return cc


@pytest.mark.parametrize("header", ["mhr_gemm.h", "mhr_gemm_testing.h"])
def test_headers_are_strict_c(header):
    r = subprocess.run([_gcc(), "-std=c99", "-pedantic", "-Wall", "-Werror", "-fsyntax-only",
                        "-x", "c", os.path.join(INCLUDE, header)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def build_program(out_dir):
    from memory_hierarchy_reuse_gb300 import build as b

    lib = b.build()
    exe = os.path.join(out_dir, "gemm_from_c")
    libdir = os.path.dirname(lib)
    cmd = [_gcc(), "-std=c99", "-O2", "-Wall", "-Werror", "-I", INCLUDE,
           "-I", os.path.join(CUDA, "include"), SRC, "-o", exe,
           "-L", libdir, "-lmhr_gemm", "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_program_builds_and_links(tmp_path):
    exe = build_program(str(tmp_path))
    assert os.access(exe, os.X_OK)


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [(300, 200, 123), (64, 700, 1000)], ids=lambda s: "x".join(map(str, s)))
def test_program_matches_oracle(tmp_path, shape):
    import oracle
    import seeded_inputs as si

    M, N, K = shape
    exe = build_program(str(tmp_path))
    A = si.matrix(M, K, 7001, "int")
    B = si.matrix(K, N, 7002, "int")
    A.tofile(tmp_path / "A.f32")
    B.tofile(tmp_path / "B.f32")
    r = subprocess.run([exe, str(tmp_path), str(M), str(N), str(K)], capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    ref = oracle.gemm(A, B)
    for name in ("C_f32", "C_3xtf32", "C_bf16"):
        C = np.fromfile(tmp_path / f"{name}.f32", dtype=np.float32).reshape(M, N)
        assert np.array_equal(C, ref), name
