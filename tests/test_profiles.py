"""The committed ncu records behind the bench line's roofline.traffic (CPU only).

profiles/traffic.json maps kernel@workload to the DRAM bytes of one captured
launch, the digest of that kernel's sources at capture time and the summary that
holds the capture's command.  bench.py reports the bytes only while the digest
still matches the sources."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _records():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as fh:
        return json.load(fh)


def test_every_record_names_an_existing_capture_with_its_command():
    for key, rec in _records().items():
        kernel, workload = key.split("@")
        assert kernel and workload, key
        for field in ("source_digest", "dram_bytes_per_launch", "dram_bytes_read", "dram_bytes_write", "capture"):
            assert field in rec, (key, field)
        assert abs(rec["dram_bytes_read"] + rec["dram_bytes_write"] - rec["dram_bytes_per_launch"]) < 1.0, key
        path = os.path.join(ROOT, rec["capture"])
        assert os.path.exists(path), (key, rec["capture"])
        text = open(path).read()
        assert "ncu " in text and "--clock-control none" in text and "bench.py" in text, rec["capture"]


def test_traffic_is_reported_only_for_current_sources(monkeypatch):
    recs = _records()
    for key, rec in recs.items():
        kernel, workload = key.split("@")
        got = bench.recorded_traffic(kernel, workload)
        if rec["source_digest"] == bench.source_digest(kernel):
            assert got == rec["dram_bytes_per_launch"], key
        else:
            assert got is None, key
    # a changed source retires the record
    kernel, workload = next(iter(recs)).split("@")
    monkeypatch.setattr(bench, "source_digest", lambda k=None: "0000000000000000")
    assert bench.recorded_traffic(kernel, workload) is None
    assert bench.recorded_traffic("no_such_kernel", workload) is None
