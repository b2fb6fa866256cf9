"""Host-side pieces of bench.py: the traffic figures and their source hashes."""
import os

import bench


def test_traffic_entries_name_existing_profiles_and_sources():
    for (workload, op), t in bench.TRAFFIC.items():
        assert op in ("encode", "decode")
        assert os.path.isfile(os.path.join(bench.ROOT, t["profile"]))
        assert t["bytes"] > 0 and len(t["sha256"]) == 64
        bench.sources_sha256(t["sources"])  # every source file exists


def test_traffic_reported_only_for_the_captured_sources(monkeypatch):
    key = next(iter(bench.TRAFFIC))
    t = bench.TRAFFIC[key]
    monkeypatch.setattr(bench, "sources_sha256", lambda names: t["sha256"])
    assert bench.measured_traffic(*key) == (t["bytes"], t["profile"])
    monkeypatch.setattr(bench, "sources_sha256", lambda names: "0" * 64)
    assert bench.measured_traffic(*key) == (None, None)
    assert bench.measured_traffic("no_such_workload", "encode") == (None, None)
