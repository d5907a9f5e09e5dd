"""Pins of the two-rank CPP / VPP / pipelined-packing simulator (host code, CPU).

Sources: the VPP technical review, §2.4 (CPP), §4.2 (Eq. (2), (3a), (3b),
Algorithm 1 and its k = 3 walk-through), §4.4 (VPP-Async order) and §4.5/§4.7
(Algorithm 2, Eq. (4a)).  The worked numbers are in
tests/golden/vpp_schedule_arithmetic.txt.
"""

import os

import pytest

from chunked_prefill_causal_gb300.schedule_sim import (cpp, cpp_requests, drain_idle, drain_window,
                                                       drain_window_from_taus, linear_taus, pack_leading_chunks,
                                                       simulate, vpp, vpp_requests)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "vpp_schedule_arithmetic.txt")


def _golden():
    out = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, *kv = line.split()
            out[name] = {k: int(v) for k, v in (x.split("=") for x in kv)}
    return out


def _tasks_inside(res, rank, t0, t1):
    """Tasks of `rank` that overlap (t0, t1), with the overlapped time."""
    out = []
    for s, e, task in res.intervals[rank]:
        ov = min(e, t1) - max(s, t0)
        if ov > 0:
            out.append((task, ov))
    return out


def _middle_window(res, k):
    return res.start((0, k, 1)), res.end[(0, k, 2)]


def test_eq3b_walkthrough_at_k3():
    g = _golden()["eq3b"]
    k = g["k"]
    tau = linear_taus(8)
    assert (tau[k - 1], tau[k], tau[k + 1]) == (g["tau_prev"], g["tau_k"], g["tau_next"])
    res = vpp(tau)
    t0, t1 = _middle_window(res, k)
    assert t1 - t0 == g["pp1_window"]
    inside = _tasks_inside(res, 0, t0, t1)
    # pp0 runs exactly s3 of C_{k-1} and s0 of C_{k+1}, whole, and is never idle there
    assert sorted(t for t, _ in inside) == [(0, k - 1, 3), (0, k + 1, 0)]
    assert sum(ov for _, ov in inside) == g["pp0_work"] == t1 - t0


def test_eq3b_holds_for_every_interior_chunk():
    n = 12
    res = vpp(linear_taus(n, t=0.75))
    for k in range(1, n - 1):
        t0, t1 = _middle_window(res, k)
        inside = _tasks_inside(res, 0, t0, t1)
        assert sorted(t for t, _ in inside) == [(0, k - 1, 3), (0, k + 1, 0)]
        assert sum(ov for _, ov in inside) == pytest.approx(t1 - t0)


def test_boundary_chunk_zero():
    g = _golden()["boundary"]
    res = vpp(linear_taus(8))
    t0, t1 = _middle_window(res, 0)
    assert t1 - t0 == g["pp1_window"]
    inside = _tasks_inside(res, 0, t0, t1)
    assert [t for t, _ in inside] == [(0, 1, 0)]
    assert inside[0][1] == g["pp0_work"]


def test_eq4a_packing_arithmetic():
    g = _golden()["eq4a"]
    n = g["N"]
    assert drain_window(n, 1.0) == g["window"]
    nxt = linear_taus(n)
    packed, left = pack_leading_chunks(g["window"], nxt)
    assert (packed, left) == (g["packed"], g["left"])
    assert sum(nxt[:packed]) == g["used"]
    assert nxt[packed] == g["next_tau"] > left


def test_drain_window_estimate_is_the_simulated_idle_gap():
    """Hand derivation under tau_k = (k+1) t with no transfer cost: pp1 ends
    s2/C_{N-1} at (N+1)^2 t - N t and pp0 ends s3/C_{N-2} at (N+1)^2 t -
    (2N+1) t, so pp0 waits (N+1) t: Algorithm 2's estimate is exact here."""
    for n in (2, 3, 5, 8, 13):
        for t in (1.0, 0.5):
            res = vpp(linear_taus(n, t))
            assert drain_idle(res, 0, n) == pytest.approx(drain_window(n, t))


def test_general_drain_window_matches_the_simulation():
    """2 tau_{N-1} - tau_{N-2} is the simulated gap for any affine law, and
    (N+1) t when the intercept equals the slope (Eq. (2))."""
    for n in (2, 4, 8):
        assert drain_window_from_taus(linear_taus(n, 0.5)) == pytest.approx(drain_window(n, 0.5))
        for a, b in ((0.5, 1.0), (2.0, 0.25), (1.0, 1.0)):
            tau = [a + b * k for k in range(n)]
            res = vpp(tau)
            assert drain_idle(res, 0, n) == pytest.approx(drain_window_from_taus(tau))
            assert drain_window_from_taus(tau) == pytest.approx(a + b * n)


def test_closed_form_makespans():
    """CPP: rank 1 ends chunk k at 2 t (1 + ... + (k+1)) + 2 (k+1) t, so the
    makespan is N (N+3) t.  VPP: pp1 starts at t and is busy 2 t sum (k+1) =
    N (N+1) t without a gap, then pp0 runs s3/C_{N-1} for N t: (N+1)^2 t."""
    for n in range(1, 20):
        assert cpp(linear_taus(n)).makespan == n * (n + 3)
        assert vpp(linear_taus(n)).makespan == (n + 1) ** 2
        assert vpp(linear_taus(n), async_order=True).makespan == (n + 1) ** 2
    # single chunk: the two schedules coincide
    assert cpp([3.0]).makespan == vpp([3.0]).makespan == 12.0


def test_pp1_has_no_steady_state_bubble_under_the_linear_law():
    for n in (4, 9):
        res = vpp(linear_taus(n))
        iv = res.intervals[1]
        gaps = [iv[i + 1][0] - iv[i][1] for i in range(len(iv) - 1)]
        assert max(gaps) == 0
        # pp0 is idle only in the drain gap
        iv0 = res.intervals[0]
        gaps0 = [iv0[i + 1][0] - iv0[i][1] for i in range(len(iv0) - 1)]
        assert sum(gaps0) == drain_window(n, 1.0)


def test_nonlinear_latencies_bring_steady_state_bubbles_back():
    """§4.2's stated boundary: with tau_k not linear in k, Eq. (3b) fails."""
    n = 8
    for tau in ([float((k + 1) ** 2) for k in range(n)],        # super-linear
                [float((k + 1) ** 0.5) for k in range(n)]):     # sub-linear (sparse attention)
        res = vpp(tau)
        iv = [res.intervals[0], res.intervals[1]]
        mid = res.start((0, 1, 1)), res.end[(0, n - 2, 2)]
        idle = sum(max(0.0, min(iv_r[i + 1][0], mid[1]) - max(iv_r[i][1], mid[0]))
                   for iv_r in iv for i in range(len(iv_r) - 1))
        assert idle > 1e-6


def test_vpp_beats_cpp_and_bubbles_halve():
    for n in (4, 8, 16):
        c, v = cpp(linear_taus(n)), vpp(linear_taus(n))
        assert v.makespan < c.makespan
        # CPP bubble 4 N t (2 N on each rank); VPP 2 (N+1) t
        assert c.bubble == 4 * n
        assert v.bubble == 2 * (n + 1)


def test_packing_fills_the_drain_and_shortens_two_requests():
    taus = [linear_taus(8), linear_taus(8)]
    plain, packed = vpp_requests(taus), vpp_requests(taus, pack=True)
    assert plain.makespan == 2 * 81
    assert drain_idle(plain, 0, 8) == 9
    assert drain_idle(packed, 0, 8) == 3                  # Eq. (4a)'s 3 units to spare
    assert packed.finish(0) == plain.finish(0) == 81      # R is not delayed
    assert packed.makespan < plain.makespan
    assert packed.bubble_ratio < plain.bubble_ratio
    # The later request's packed entry stages ran inside R's drain window.
    assert {t for s, e, t in packed.intervals[0] if t[0] == 1 and e <= packed.start((0, 7, 3))} == \
        {(1, 0, 0), (1, 1, 0), (1, 2, 0)}


def test_overfull_window_delays_the_current_request():
    """§4.7: packing past the window reintroduces delay on R's own path."""
    taus = [linear_taus(8), linear_taus(8)]
    over = vpp_requests(taus, pack=True, window=lambda i: 10.0)   # 1+2+3+4 = 10 > 9
    assert over.finish(0) == 81 + 1


def test_cpp_requests_chain_and_vpp_single_request_match():
    taus = [linear_taus(5)]
    assert vpp_requests(taus).makespan == vpp(taus[0]).makespan
    assert cpp_requests(taus).makespan == cpp(taus[0]).makespan


def test_transfer_latency_delays_only_cross_rank_edges():
    # one chunk: CPP has one cross-rank edge, VPP two (s0->s1 and s2->s3)
    assert cpp([1.0], comm=0.25).makespan == 4.25
    assert vpp([1.0], comm=0.25).makespan == 4.5


def test_bad_orders_are_rejected():
    with pytest.raises(RuntimeError):
        # rank 0 lists chunk 1 before chunk 0, whose KV cache chunk 1 needs
        simulate([[(0, 1, 0), (0, 0, 0)], []], [0, 1], lambda r, k, s: 1.0)
    with pytest.raises(ValueError):
        simulate([[(0, 0, 1)], []], [0, 1], lambda r, k, s: 1.0)
