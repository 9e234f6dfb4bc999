"""The benchmark's CPU baselines: the oracle timed on one core and on all host
cores (one single-threaded process per core, each on a disjoint share of the
requests, timed together).  Run on the small fp32 config so it takes seconds."""
import bench


def test_one_core_oracle_timing_reports_its_sample():
    o = bench.time_oracle("tiny_decode_f32", min_seconds=0.2)
    assert o["reps"] >= 1 and o["seconds"] > 0 and o["requests"] == 4
    assert o["bytes_per_rep"] > 0


def test_all_cores_oracle_timing_covers_every_request_once():
    a = bench.time_oracle_all_cores("tiny_decode_f32", min_seconds=0.2)
    # the config has 4 requests: at most 4 worker processes, each with its own requests
    assert 1 <= a["cores"] <= 4
    assert a["requests"] == 4
    assert a["gbs"] > 0 and a["seconds"] >= 0.2
