"""bench.py's host-side bookkeeping, without a GPU: the stored ncu traffic is reported only for the
kernel sources it was captured from, and the committed traffic table is well formed."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_stored_traffic_follows_the_sources(monkeypatch):
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        entries = json.load(f)
    e = entries[0]
    # the entry's own sources: its bytes
    monkeypatch.setattr(bench, "sources_sha", lambda paths: e["source_sha256"])
    assert bench.stored_traffic(e["kernel"], e["workload"], ["any"]) == e["bytes_per_launch"]
    # changed sources: nothing (the counters no longer describe the kernel)
    monkeypatch.setattr(bench, "sources_sha", lambda paths: "0" * 64)
    assert bench.stored_traffic(e["kernel"], e["workload"], ["any"]) is None
    # another workload or kernel: nothing
    monkeypatch.setattr(bench, "sources_sha", lambda paths: e["source_sha256"])
    assert bench.stored_traffic(e["kernel"], "no_such_workload", ["any"]) is None
    assert bench.stored_traffic("no_such_kernel", e["workload"], ["any"]) is None


def test_traffic_table_is_well_formed():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        entries = json.load(f)
    assert entries
    seen = set()
    for e in entries:
        assert set(e) >= {"kernel", "workload", "bytes_per_launch", "source_sha256", "from"}
        assert e["bytes_per_launch"] > 0 and len(e["source_sha256"]) == 64
        assert os.path.exists(os.path.join(ROOT, e["from"].split(" ")[0].rstrip(",")))
        key = (e["kernel"], e["workload"])
        assert key not in seen  # one capture per kernel and workload
        seen.add(key)


def test_sources_sha_depends_on_content(tmp_path):
    a, b = tmp_path / "a.cu", tmp_path / "b.cu"
    a.write_text("x")
    b.write_text("y")
    assert bench.sources_sha([str(a)]) != bench.sources_sha([str(b)])
    assert bench.sources_sha([str(a)]) == bench.sources_sha([str(a)])
