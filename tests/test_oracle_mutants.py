"""The oracle's pins catch planted mistakes (CPU only).

Each case copies the oracle's C source, plants one plausible mistake in the
copy (fp32 accumulation, a dropped or shifted term, a sign error, a stride or
index mistake, a wrong final rounding, a wrong normaliser), builds the copy
with the oracle's own build recipe, and runs every pin of
test_oracle_pins.py against it in a child process, which also contains any
crash. At least one pin must fail for every mistake. The committed oracle is
never modified; the unmodified copy must pass every pin (the control case).
"""
import os
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle_gemm.c")

# (name, text in oracle_gemm.c, replacement)
MUTANTS = [
    ("fp32-accumulation", "double s = 0.0, a = 0.0;", "float s = 0.0f; double a = 0.0;"),
    ("last-term-dropped", "for (int64_t k = 0; k < K; ++k) {",
     "for (int64_t k = 0; k + 1 < K; ++k) {"),
    ("first-term-dropped", "for (int64_t k = 0; k < K; ++k) {", "for (int64_t k = 1; k < K; ++k) {"),
    ("sign-of-first-term", "    s += x * y;", "    s += (k == 0 ? -x : x) * y;"),
    ("row-stride-ignores-lda", "const float* arow = A + i * lda;",
     "const float* arow = A + i * K;"),
    ("b-column-mirrored", "double y = (double)B[k * ldb + j];",
     "double y = (double)B[k * ldb + (ldb - 1 - j)];"),
    ("rounding-toward-zero", "C[i * ldc + j] = (float)s;",
     "C[i * ldc + j] = (s != (double)(float)s && fabs((double)(float)s) > fabs(s)) ? "
     "nextafterf((float)s, 0.0f) : (float)s;"),
    ("abs-sum-signed", "    a += fabs(x) * fabs(y);", "    a += fabs(x) * y;"),
    # row and column swapped in the sampled entries (where both stay in range)
    ("entries-transposed", "double s = dot_entry(A, B, K, lda, ldb, rows[t], cols[t], &a);",
     "const int sw = rows[t] < N && cols[t] < M; "
     "double s = dot_entry(A, B, K, lda, ldb, sw ? cols[t] : rows[t], sw ? rows[t] : cols[t], "
     "&a);"),
]

# Child process: load a copy of the oracle package built from the mutated
# source, then call every pin in test_oracle_pins.py on it; exit code = the
# number of pins that failed.
RUNNER = textwrap.dedent("""
    import importlib.util, inspect, os, sys
    root, src = sys.argv[1], sys.argv[2]
    sys.path.insert(0, root)
    sys.path.insert(0, os.path.join(root, "tests"))
    spec = importlib.util.spec_from_file_location(
        "oracle_copy", os.path.join(root, "oracle", "__init__.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod._SRC = src
    mod._LIB = os.path.join(os.path.dirname(src), "liboracle_gemm.so")
    mod._lib = None
    try:
        mod.build()
    except Exception:
        sys.exit(200)  # the copy did not build: not a caught mistake
    import test_oracle_pins as pins
    failed = 0
    for name, fn in sorted(vars(pins).items()):
        if not name.startswith("test_") or not callable(fn):
            continue
        params = inspect.signature(fn).parameters
        if "oracle_lib" not in params:
            continue
        kwargs = {"oracle_lib": mod}
        if "dist" in params:
            runs = [dict(kwargs, dist=d) for d in ("uniform", "normal")]
        else:
            runs = [kwargs]
        for kw in runs:
            try:
                fn(**kw)
            except Exception:
                failed += 1
    sys.exit(min(failed, 100))
""")


def run_pins(src_path):
    """Exit code of the child: the number of failed pins, 200 if the copy did
    not build, negative if it crashed."""
    r = subprocess.run([sys.executable, "-c", RUNNER, ROOT, src_path], capture_output=True,
                       text=True, timeout=300)
    return r.returncode


def planted(tmp_path, name, old, new):
    text = open(SRC).read()
    assert text.count(old) >= 1, (name, old)
    d = tmp_path / name
    d.mkdir()
    p = d / "oracle_gemm.c"
    p.write_text(text.replace(old, new))
    return str(p)


def test_unmodified_copy_passes_every_pin(tmp_path):
    src = planted(tmp_path, "control", "int oracle_max_threads", "int oracle_max_threads")
    assert run_pins(src) == 0


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(tmp_path, name, old, new):
    rc = run_pins(planted(tmp_path, name, old, new))
    assert rc != 200, f"the copy with {name!r} did not build"
    assert rc != 0, f"no pin caught the planted mistake {name!r}"
