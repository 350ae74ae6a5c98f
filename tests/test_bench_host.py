"""bench.py's host-only pieces that need no GPU: the CPU baseline's all-cores leg."""
import bench


def test_oracle_on_every_core_sums_concurrent_single_threaded_rates():
    r = bench.oracle_all_cores("toy_q8_0", gb_per_process=0.5)
    assert r.get("error") is None, r
    assert 1 <= r["cores"] <= 16
    assert r["value"] > 0
    assert r["kind"] == "oracle"


def test_oracle_samples_differ_by_offset_but_time_the_same_work():
    w = bench.si.WORKLOADS["toy_q8_0"]
    a = bench.oracle_sample(w, sample_offset=0)
    b = bench.oracle_sample(w, sample_offset=3)
    assert a["sample"] == b["sample"]
    assert a["value"] > 0 and b["value"] > 0
