"""Host logic of bench.py's DRAM-traffic lookup, on CPU.

profiles/traffic.txt holds, per workload, DRAM bytes measured with ncu and a
sha256 of that workload's kernel sources.  The figure may only be reported
while the sources still match; a changed source must turn it into null.
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_traffic_reported_while_sources_match():
    for w in ("decode_b1", "stack", "decode_b64", "prefill"):
        v = bench._traffic(w)
        assert isinstance(v, int) and v > 0, w
    # the stack runs the batch-1 chain once per layer
    assert bench._traffic("stack") == 47 * bench._traffic("decode_b1")


def test_traffic_null_once_a_source_changes(monkeypatch):
    real = bench._sources_digest
    monkeypatch.setattr(bench, "_sources_digest", lambda names: real(names)[::-1])
    for w in ("decode_b1", "stack", "decode_b64", "prefill"):
        assert bench._traffic(w) is None, w


def test_traffic_digest_covers_listed_files_only():
    # every listed source exists, and the digest depends on the file list
    d = os.path.join(ROOT, "nvfp4_expert_ffn_gemv_b300", "csrc")
    for names in bench.TRAFFIC_SOURCES.values():
        for n in names:
            assert os.path.isfile(os.path.join(d, n)), n
    a = bench._sources_digest(("decode_b1.cu",))
    b = bench._sources_digest(("decode_b1.cu", "common.cuh"))
    assert a != b
