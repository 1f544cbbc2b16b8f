"""The committed measurement evidence is well formed (CPU only)."""
import json
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = os.path.join(ROOT, "profiles")


def test_traffic_entries_point_at_summaries():
    import bench

    d = json.load(open(os.path.join(PROFILES, "ncu_traffic.json")))
    kernels = [k for k in d if not k.startswith("_")]
    assert kernels
    for kernel in kernels:
        assert kernel.split("<")[0] in bench.KERNEL_SOURCES, kernel
        for workload, e in d[kernel].items():
            assert workload in bench.WORKLOADS
            assert e["dram_bytes_per_launch"] > 0
            assert len(e["source_digest"]) == 16
            assert os.path.exists(os.path.join(ROOT, e["capture"])), e["capture"]


def test_summaries_state_their_commands():
    names = [f for f in os.listdir(PROFILES) if f.endswith(".md")]
    assert names
    for f in names:
        text = open(os.path.join(PROFILES, f)).read()
        assert "ncu " in text and "--clock-control none" in text, f
        assert "bench.py" in text, f


def test_profiles_hold_only_text():
    for f in os.listdir(PROFILES):
        assert f.endswith((".md", ".txt", ".json")), f


def test_source_digest_ignores_comments_and_layout():
    """Stored counters stay valid across comment-only edits of a kernel's
    sources, and become stale on any change to its code."""
    import bench

    code = "int f(int x) {\n  return x + 1;  // one more\n}\n/* block\n comment */\n"
    assert bench._code_only(code) == "int f(int x) { return x + 1; }"
    assert bench._code_only(code.replace("// one more", "// two more")) == bench._code_only(code)
    assert bench._code_only(code.replace("x + 1", "x + 2")) != bench._code_only(code)
