"""Host logic of bench.py's DRAM-traffic lookup, on CPU.

profiles/traffic.txt holds, per workload, DRAM bytes measured with ncu and a
sha256 of that workload's kernel sources.  The figure may only be reported
while the sources still match; a changed source must turn it into null.
The lookup is exercised on a scratch copy of the layout, so these tests do not
depend on whether the committed figures are current.
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _fake_tree(tmp_path, monkeypatch):
    csrc = tmp_path / "nvfp4_expert_ffn_gemv_b300" / "csrc"
    csrc.mkdir(parents=True)
    names = sorted({n for v in bench.TRAFFIC_SOURCES.values() for n in v})
    for n in names:
        (csrc / n).write_text(f"// {n}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    lines = [f"{w} kernels=x sha256={bench._sources_digest(bench.TRAFFIC_SOURCES[w])} traffic_bytes={1000 + i}"
             for i, w in enumerate(("decode_b1", "decode_b64", "prefill"))]
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.txt").write_text("# comment\n" + "\n".join(lines) + "\n")
    return csrc


def test_traffic_reported_while_sources_match(tmp_path, monkeypatch):
    _fake_tree(tmp_path, monkeypatch)
    assert bench._traffic("decode_b1") == 1000
    assert bench._traffic("decode_b64") == 1001
    assert bench._traffic("prefill") == 1002
    assert bench._traffic("stack") is None          # no line for it
    assert bench._traffic("no_such_workload") is None


def test_traffic_null_once_a_listed_source_changes(tmp_path, monkeypatch):
    csrc = _fake_tree(tmp_path, monkeypatch)
    (csrc / "prefill.cu").write_text("// changed\n")
    assert bench._traffic("prefill") is None
    assert bench._traffic("decode_b1") == 1000      # prefill.cu is not one of its sources
    (csrc / "common.cuh").write_text("// changed\n")
    assert bench._traffic("decode_b1") is None      # a shared header is


def test_traffic_sources_exist_in_the_package():
    d = os.path.join(ROOT, "nvfp4_expert_ffn_gemv_b300", "csrc")
    for names in bench.TRAFFIC_SOURCES.values():
        for n in names:
            assert os.path.isfile(os.path.join(d, n)), n
