"""CPU tests of bench.py's host-side helpers (no GPU): the committed DRAM-traffic
record is used only while the kernel source it was taken from is unchanged, the
peaks file is read with its fallbacks, and the algorithmic constants follow from
their stated formulas."""
import json
import os

import bench


def test_recorded_traffic_matches_current_source():
    rec = json.load(open(os.path.join(bench.ROOT, "profiles", "roofline_traffic.json")))
    t = bench.recorded_traffic(rec["kernel"])
    assert t == rec["dram_read_bytes"] + rec["dram_write_bytes"]
    assert bench.recorded_traffic("some_other_kernel") is None


def test_recorded_traffic_is_dropped_when_the_source_changes(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    src = tmp_path / "k.cu"
    src.write_text("kernel v1")
    rec = {"kernel": "k", "source": "k.cu", "source_sha256": "0" * 64, "dram_read_bytes": 1, "dram_write_bytes": 2}
    (prof / "roofline_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("k") is None           # hash differs from the file's
    import hashlib
    rec["source_sha256"] = hashlib.sha256(b"kernel v1").hexdigest()
    (prof / "roofline_traffic.json").write_text(json.dumps(rec))
    assert bench.recorded_traffic("k") == 3


def test_algorithmic_constants():
    K = V = 128
    # q, k, v, graw (4 x 256 B) + b (2 B) + out (256 B)
    assert bench.BYTES_PER_TOKEN_HEAD == 4 * 2 * K + 2 + 2 * V
    assert bench.STATE_BYTES_PER_SEQ_HEAD == 2 * K * V * 4
    assert bench.BWD_FLOPS_PER_TOKEN_HEAD == 2 * (2 * 3 + 11) * K * V


def test_whole_job_value_is_units_over_max_time():
    assert bench.whole_job_value(1000, 2.0, 1) == 1000 / 2e-3
    assert bench.whole_job_value(1000, 2.0, 4) == 4 * 1000 / 2e-3
