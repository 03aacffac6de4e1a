"""Host logic of bench.py that needs no GPU: which stored ncu traffic figure a
bench line may carry."""
import json
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import bench  # noqa: E402


def test_code_only_drops_comments_and_blank_space():
    a = "int x = 1;  // one\n/* a\n block */ float y;\n"
    b = "int x = 1;\nfloat   y; // another comment\n"
    assert bench._code_only(a) == bench._code_only(b) == "int x = 1; float y;"
    assert bench._code_only("int x = 2;") != bench._code_only("int x = 1;")


def test_traffic_is_reported_only_for_the_captured_code(tmp_path, monkeypatch):
    # a copy of the stage-1 sources: a comment edit keeps the capture, a code edit drops it
    csrc = tmp_path / "mla_decode_attention_split_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in bench.STAGE1_SOURCES:
        src = os.path.join(bench.ROOT, "mla_decode_attention_split_gb300", "csrc", f)
        (csrc / f).write_text(open(src, encoding="utf-8").read(), encoding="utf-8")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = bench._stage1_source_sha()
    (tmp_path / "profiles" / "stage1_dram_traffic.json").write_text(
        json.dumps({"w": {"source_sha": sha, "dram_bytes_per_launch": 123}}))
    assert bench._ncu_traffic("w") == 123.0
    assert bench._ncu_traffic("other") is None
    f = csrc / bench.STAGE1_SOURCES[0]
    f.write_text(f.read_text(encoding="utf-8") + "\n// a note\n", encoding="utf-8")
    assert bench._ncu_traffic("w") == 123.0
    f.write_text(f.read_text(encoding="utf-8") + "\nstatic int extra_symbol;\n", encoding="utf-8")
    assert bench._ncu_traffic("w") is None

