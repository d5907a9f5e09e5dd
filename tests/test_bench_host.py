"""Host-side arithmetic of bench.py, on CPU."""

import bench
from chunked_prefill_causal_gb300 import workloads as W


def test_ex2_bound_counts_one_exponential_per_unmasked_score():
    w = W.WORKLOADS["long128k"]
    chunks = w.chunks()
    # 64 heads; chunk k has 16384 queries over 16384 k prefix keys plus the causal diagonal
    exps = 64 * sum(16384 * 16384 * k + 16384 * 16385 // 2 for k in range(8))
    r = bench.ex2_bound(w, chunks, 100.0, {"sm_mhz": 2000.0}, 152)
    assert r["exps_per_step"] == exps
    ms = exps / (32 * 152 * 2000e6) * 1e3
    assert abs(r["ms"] - round(ms, 3)) < 1e-9
    assert abs(r["frac_of_attention_time"] - round(ms / 100.0, 4)) < 1e-12


def test_ex2_bound_without_a_clock_is_null():
    w = W.WORKLOADS["gqa32k"]
    assert bench.ex2_bound(w, w.chunks(), 10.0, {"sm_mhz": None, "sm_max_mhz": None}, 152) is None
    assert bench.ex2_bound(w, w.chunks(), 10.0, None, 152) is None


def test_recorded_traffic_is_null_once_the_kernel_sources_change(monkeypatch):
    digest = bench.kernel_sources_digest()
    monkeypatch.setattr(bench, "TRAFFIC", {"long128k": {"sources_sha256": digest, "bytes_per_launch": 1.5e9}})
    assert bench.recorded_traffic("long128k") == 1.5e9
    assert bench.recorded_traffic("gqa32k") is None
    monkeypatch.setattr(bench, "TRAFFIC", {"long128k": {"sources_sha256": "0" * 64, "bytes_per_launch": 1.5e9}})
    assert bench.recorded_traffic("long128k") is None
