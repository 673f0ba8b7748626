"""The source digest that ties a recorded ncu traffic figure to the kernels it was taken
from: it follows the code and ignores comments and blank space, and bench.py reports a
recorded figure only while the digest of its sources still matches."""
import json
import os

from sparse_teacher_kl_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_code_only_ignores_comments_and_blank_space():
    a = b"int f(int x) {\n  return x + 1;  // one more\n}\n"
    b = b"/* header\n   comment */\nint f(int x) {\n\n    return x + 1;\n}\n// trailing\n"
    c = b"int f(int x) {\n  return x + 2;\n}\n"
    assert build._code_only(a) == build._code_only(b)
    assert build._code_only(a) != build._code_only(c)


def test_source_digest_follows_code_not_comments(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    src.write_text("__global__ void k(int* p) { *p = 1; }\n")
    monkeypatch.setattr(build, "CSRC", str(tmp_path))
    d0 = build.source_digest(["k.cu"])
    src.write_text("// a note\n\n    __global__ void k(int* p) { *p = 1; }  /* store */\n")
    assert build.source_digest(["k.cu"]) == d0
    src.write_text("__global__ void k(int* p) { *p = 2; }\n")
    assert build.source_digest(["k.cu"]) != d0


def test_recorded_traffic_entries_are_well_formed():
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
        rec = json.load(f)
    entries = [(w, k, v) for w, ks in rec["kernels"].items() for k, v in ks.items()]
    assert entries
    for w, k, v in entries:
        assert isinstance(v["bytes_per_launch"], int) and v["bytes_per_launch"] > 0, (w, k)
        assert len(v["digest"]) == 16 and all(ch in "0123456789abcdef" for ch in v["digest"]), (w, k)
        for name in v["sources"]:
            assert os.path.exists(os.path.join(build.CSRC, name)), (w, k, name)
