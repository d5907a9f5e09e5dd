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


def test_mixed_launch_count_and_combined_bound():
    # varlen append + decode kernel + its merge + one chunk-attention launch per 64 segments
    assert bench.mixed_launches(4, 256) == 4
    assert bench.mixed_launches(0, 256) == 3
    assert bench.mixed_launches(4, 0) == 2
    assert bench.mixed_launches(65, 1) == 5
    # the longer of the prefill FLOPs at the tensor peak and the decode bytes at HBM bandwidth
    assert abs(bench.mixed_bound_ms(7.0e12, 18.5e9, 1750.0, 6700.0) - 4.0) < 1e-9
    assert abs(bench.mixed_bound_ms(1.0e12, 67.0e9, 1000.0, 6700.0) - 10.0) < 1e-9


def test_summary_keeps_the_judged_figures_in_a_short_tail():
    line = {"config": {"workload": "long128k"}, "value": 1500.0,
            "roofline": {"frac": 0.86, "frac_of_burst": 0.78},
            "late_chunks_frac_peak": 0.87, "late_chunks_tflops": 1520.0,
            "per_chunk": [{"k": k, "ms": 3.0 + 6 * k, "tflops": 1400.0 + k, "frac_peak": 0.8} for k in range(8)],
            "gqa32k": {"tflops": 1300.0, "frac": 0.75, "rows": [[k, 4096 * k, 4096, 1.0, 1300.0, 0.75, 0.68]
                                                                  for k in range(8)]},
            "mla512k": {"tflops": 1280.0, "frac": 0.74, "rows": [[k, 24576 * k, 24576, 100.0, 1280.0, 0.74, 0.66]
                                                                   for k in (0, 10, 20, 21)]},
            "kv_append": {"frac_hbm": 0.99},
            "mixed": {"decode_frac_hbm": 1.07, "step_ms": 7.4, "bound_ms": 4.03, "frac_of_bound": 0.5446},
            "cpu_baseline": {"value": 4.2e-2, "cores": 16}}
    s = bench.summary(line, 1924.4)
    assert s["late_frac"] == 0.87 and s["late_frac_burst"] == round(1520.0 / 1924.4, 4)
    assert [r[0] for r in s["k_ms_tflops_frac"]] == list(range(8))
    assert [r[0] for r in s["mla512k"]["k_ms_tflops_frac"]] == [0, 10, 20, 21]
    assert s["mixed_frac_of_bound"] == 0.5446 and s["append_frac_hbm"] == 0.99
    import json
    assert len(json.dumps(s)) < 1400


def test_timeline_intervals_pair_each_issuer_block_with_the_previous_tiles_softmax():
    import numpy as np
    # Synthetic stamps with a 3000-cycle period: softmax of tile j at
    # S ready 3000 j, S in registers +70, first part of P +600, second +1000;
    # the issuer's block j (P V of tile j-1, then Q K^T of tile j) sees the
    # first part at 3000 (j-1) + 800, takes the turn at +1000, sees the second
    # part at +1500 and finishes issuing at +2900.
    buf = np.zeros((4, 64, 4), dtype=np.int64)
    for j in range(64):
        for r in (2, 3):
            buf[r, j] = [3000 * j, 3000 * j + 70, 3000 * j + 600, 3000 * j + 1000]
        for r in (0, 1):
            base = 3000 * (j - 1)
            buf[r, j] = [base + 800, base + 1000, base + 2900, base + 1500]
    iv = bench.timeline_intervals(buf)
    for t in "AB":
        assert iv[f"{t}.softmax: S ready -> S in registers"] == 70
        assert iv[f"{t}.softmax: S in registers -> first part of P signalled"] == 530
        assert iv[f"{t}.softmax: first -> second part of P signalled"] == 400
        assert iv[f"{t}.issuer: first part of P signalled -> seen"] == 200
        assert iv[f"{t}.issuer: seen -> turn"] == 200
        assert iv[f"{t}.issuer: turn -> second part of P seen"] == 500
        assert iv[f"{t}.issuer: second part seen -> block issued"] == 1400
        assert iv[f"{t}.issuer: block issued -> S ready"] == 100
        assert iv[f"{t}.period (S ready to S ready)"] == 3000
