"""CPU tests of bench.py's host-side helpers (no GPU): the committed DRAM-traffic
record is used only while the kernel source it was taken from is unchanged, the
peaks file is read with its fallbacks, and the algorithmic constants follow from
their stated formulas."""
import json
import os

import bench


def test_recorded_traffic_follows_the_current_source():
    import hashlib
    rec = json.load(open(os.path.join(bench.ROOT, "profiles", "roofline_traffic.json")))
    src = open(os.path.join(bench.ROOT, rec["source"]), "rb").read()
    t = bench.recorded_traffic(rec["kernel"])
    if hashlib.sha256(src).hexdigest() == rec["source_sha256"]:
        assert t == rec["dram_read_bytes"] + rec["dram_write_bytes"]
    else:
        assert t is None     # counters taken on another version of the kernel source
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
    # chunk-form backward in units of one 64 x 64 x 128 product (u) per (chunk, value head):
    # prep 1.25 u (A, P sub-block pairs) + 3 u (W, U, N); chains 4 u + 6 u; value side 14 u;
    # key side 3 u + 2.5 u (pair products) = 33.75 u, 2 flops per multiply-add, 64 tokens
    u = 64 * 64 * 128
    assert bench.BWD_FLOPS_PER_TOKEN_HEAD == 2 * int(33.75 * u) // 64


def test_whole_job_value_is_units_over_max_time():
    assert bench.whole_job_value(1000, 2.0, 1) == 1000 / 2e-3
    assert bench.whole_job_value(1000, 2.0, 4) == 4 * 1000 / 2e-3


def test_per_config_algorithmic_work():
    # the dense workload counts q and k once per q/k head: with H_qk = H_v it is the headline formula
    units, nbytes, flops = bench.fwd_alg(2, 16384, 32, 32, 2)
    assert units == 2 * 16384 * 32
    assert nbytes == units * bench.BYTES_PER_TOKEN_HEAD + 2 * 32 * bench.STATE_BYTES_PER_SEQ_HEAD
    assert flops == units * bench.FLOPS_PER_TOKEN_HEAD
    # grouped value heads: q, k read once per group of four value heads
    _, gb, _ = bench.fwd_alg(1, 32768, 16, 64, 2)
    assert gb == 32768 * (16 * 512 + 64 * (512 + 2 + 256)) + 2 * 64 * bench.STATE_BYTES_PER_SEQ_HEAD


def test_rate_fields_flag_rates_above_the_copy_peak():
    t = {"ms": 1.0, "p10_ms": 0.9, "p90_ms": 1.1, "reps": 3}
    ok = bench.rate_fields(t, 1000, 10 ** 9, 10 ** 12, hbm_peak=2000.0, tc_peak=2000.0)
    assert ok["GB/s"] == 1000.0 and "note" not in ok and ok["hbm_frac"] == 0.5
    hi = bench.rate_fields(t, 1000, 3 * 10 ** 9, 10 ** 12, hbm_peak=2000.0, tc_peak=2000.0)
    assert "note" in hi


def test_both_arms_print_the_same_config():
    assert bench.bench_config(1) == bench.bench_config(1)
    assert bench.bench_config(2)["parallelism"] == "replicas x2"
