"""Two-rank pipeline schedules of chunked prefill, driven by per-chunk latencies.

"VPP: Virtual Pipeline Parallelism for Efficient Chunked Prefill in
Long-Context LLM Inference" (technical review):

* §2.4 CPP: chunked prefill on a pipeline of two ranks, each rank holding half
  of the layers; chunks flow rank 0 -> rank 1 in order.
* §4.2 VPP: four virtual stages s0..s3; pp0 holds s0 and s3, pp1 holds s1 and
  s2, so a chunk goes pp0 -> pp1 -> pp1 -> pp0.  While pp1 runs the middle
  stages of C_k, pp0 runs s3 of C_{k-1} and s0 of C_{k+1} (Algorithm 1); the
  VPP-Async variant (§4.4) swaps the order of those two on pp0.
* §4.5 and §4.7, pipelined packing: the tail drain window of a request with N
  chunks is estimated as (N+1) t, and the leading chunks of the next request
  are packed into it greedily while they fit (Algorithm 2).

Model.  Latencies are per virtual stage: tau[k] for one virtual stage of chunk
k (Eq. (2) reads tau_k = (k+1) t when attention dominates).  A CPP stage holds
two virtual stages' worth of layers, so it takes 2 tau[k].  A stage of chunk k
of a request needs (i) the previous stage of the same chunk, plus `comm` when
that ran on the other rank, and (ii) the same stage of chunk k-1 of the same
request, whose KV cache its attention reads.  Each rank runs its own list of
stages in a fixed order, a stage starting once its rank is free and its inputs
are ready.  `comm` is a transfer latency only: it delays the receiver and
occupies neither rank (the reading used for sends that overlap compute).

The drain window is measured on pp0: from the end of s3 of C_{N-2} to the start
of s3 of C_{N-1}, the time pp0 has nothing of the request to run.  Packing puts
s0 of the next request's leading chunks there; pp1 then starts that request's
middle stages as soon as it is done with the current one.
"""

from __future__ import annotations

import dataclasses


@dataclasses.dataclass
class ScheduleResult:
    makespan: float
    busy: list             # busy time per rank
    intervals: list        # per rank: list of (start, end, (request, chunk, stage))
    end: dict              # (request, chunk, stage) -> end time

    @property
    def bubble(self) -> float:
        """Idle time of both ranks inside [0, makespan]."""
        return sum(self.makespan - b for b in self.busy)

    @property
    def bubble_ratio(self) -> float:
        return self.bubble / (len(self.busy) * self.makespan)

    def start(self, task):
        for iv in self.intervals:
            for s, e, t in iv:
                if t == task:
                    return s
        raise KeyError(task)

    def finish(self, request: int) -> float:
        """Time the request's last stage ends (its prefill is complete)."""
        return max(e for (r, _, _), e in self.end.items() if r == request)


def simulate(orders, rank_of_stage, dur, comm: float = 0.0) -> ScheduleResult:
    """Runs two ranks' ordered stage lists (tasks (request, chunk, stage)).

    dur(request, chunk, stage) is a task's latency; rank_of_stage[s] is the
    rank that holds stage s.  Raises RuntimeError if the orders deadlock."""
    end = {}
    free = [0.0] * len(orders)
    pos = [0] * len(orders)
    intervals = [[] for _ in orders]
    remaining = sum(len(o) for o in orders)
    while remaining:
        progressed = False
        for rank, order in enumerate(orders):
            while pos[rank] < len(order):
                task = order[pos[rank]]
                r, k, s = task
                if rank_of_stage[s] != rank:
                    raise ValueError(f"stage {s} is not held by rank {rank}")
                ready = free[rank]
                deps = []
                if s > 0:
                    deps.append(((r, k, s - 1), comm if rank_of_stage[s - 1] != rank else 0.0))
                if k > 0:
                    deps.append(((r, k - 1, s), 0.0))
                if any(d not in end for d, _ in deps):
                    break
                for d, extra in deps:
                    ready = max(ready, end[d] + extra)
                end[task] = ready + float(dur(r, k, s))
                intervals[rank].append((ready, end[task], task))
                free[rank] = end[task]
                pos[rank] += 1
                remaining -= 1
                progressed = True
        if not progressed:
            raise RuntimeError("schedule orders deadlock")
    makespan = max(end.values()) if end else 0.0
    busy = [sum(e - s for s, e, _ in iv) for iv in intervals]
    return ScheduleResult(makespan, busy, intervals, end)


# --------------------------------------------------------------------- orders
def _cpp_orders(requests):
    o0 = [(r, k, 0) for r, n in requests for k in range(n)]
    o1 = [(r, k, 1) for r, n in requests for k in range(n)]
    return [o0, o1]


def _vpp_pp0(r, n, async_order, skip_s0=0):
    """pp0's list for one request (Algorithm 1): s0 of C_0, then for every k
    the pair (s3 of C_{k-1}, s0 of C_{k+1}), then s3 of C_{N-1}.  The first
    `skip_s0` entry stages were already run (packed into an earlier drain)."""
    out = [(r, 0, 0)]
    for k in range(n):
        pair = []
        if k >= 1:
            pair.append((r, k - 1, 3))
        if k + 1 < n:
            pair.append((r, k + 1, 0))
        out += pair[::-1] if async_order else pair
    out.append((r, n - 1, 3))
    return [t for t in out if not (t[2] == 0 and t[1] < skip_s0)]


def _vpp_pp1(r, n):
    return [(r, k, s) for k in range(n) for s in (1, 2)]


def cpp(tau, comm: float = 0.0) -> ScheduleResult:
    """CPP (§2.4): rank i runs stage i of every chunk in order."""
    n = len(tau)
    return simulate(_cpp_orders([(0, n)]), [0, 1], lambda r, k, s: 2.0 * tau[k], comm)


def vpp(tau, comm: float = 0.0, async_order: bool = False) -> ScheduleResult:
    """V-shaped VPP (Algorithm 1), or VPP-Async's order with async_order."""
    n = len(tau)
    orders = [_vpp_pp0(0, n, async_order), _vpp_pp1(0, n)]
    return simulate(orders, [0, 1, 1, 0], lambda r, k, s: float(tau[k]), comm)


def linear_taus(n: int, t: float = 1.0):
    """Eq. (2): tau_k = (k+1) t."""
    return [(k + 1) * t for k in range(n)]


def drain_window(n_chunks: int, t: float) -> float:
    """Algorithm 2's estimate of the tail drain window: (N+1) t."""
    return (n_chunks + 1) * t


def drain_window_from_taus(tau) -> float:
    """The drain window from per-chunk latencies: while pp1 runs the two
    middle stages of C_{N-1} (2 tau_{N-1}), pp0 has only s3 of C_{N-2}
    (tau_{N-2}) left, so it waits 2 tau_{N-1} - tau_{N-2}.  This is exact
    when the two start together, as they do in the balanced steady state of
    any affine law a + b k, where it equals a + b N; under Eq. (2) it is
    2 N t - (N-1) t = (N+1) t, Algorithm 2's estimate."""
    if len(tau) < 2:
        raise ValueError("a drain window needs at least two chunks")
    return 2.0 * tau[-1] - tau[-2]


def pack_leading_chunks(window: float, next_taus):
    """Greedy packing of Algorithm 2: takes the next request's chunks from
    j = 0 while each fits the window left.  Returns (count, window left)."""
    left = float(window)
    n = 0
    for tau in next_taus:
        if tau > left:
            break
        left -= tau
        n += 1
    return n, left


def drain_idle(res: ScheduleResult, request: int, n_chunks: int) -> float:
    """pp0's idle time in the request's drain: from the end of s3 of C_{N-2}
    to the start of s3 of C_{N-1}, less whatever else pp0 ran there."""
    if n_chunks < 2:
        raise ValueError("a drain window needs at least two chunks")
    t0 = res.end[(request, n_chunks - 2, 3)]
    t1 = res.start((request, n_chunks - 1, 3))
    busy = sum(max(0.0, min(e, t1) - max(s, t0)) for s, e, _ in res.intervals[0])
    return (t1 - t0) - busy


def vpp_requests(taus, comm: float = 0.0, async_order: bool = False, pack: bool = False,
                 window=None) -> ScheduleResult:
    """Back-to-back requests under VPP, each with its own chunk latencies.

    Without packing a request's stages follow the previous request's on both
    ranks.  With packing (Algorithm 2) pp0 runs s0 of the next request's
    leading chunks in the current request's drain window, between s3 of
    C_{N-2} and s3 of C_{N-1}; as many are packed as fit `window(i)`
    (default: drain_window_from_taus of request i, which is the (N+1) t
    estimate under Eq. (2)), checked against the next request's s0
    latencies."""
    orders = [[], []]
    skip = [0] * len(taus)
    for i, tau in enumerate(taus):
        n = len(tau)
        pp0 = _vpp_pp0(i, n, async_order, skip_s0=skip[i])
        if pack and i + 1 < len(taus) and n >= 2:
            w = drain_window_from_taus(tau) if window is None else window(i)
            p, _ = pack_leading_chunks(w, taus[i + 1])
            skip[i + 1] = p
            # pp0's list for this request ends with s3 of C_{N-1}: packed
            # entry stages go right before it
            pp0 = pp0[:-1] + [(i + 1, j, 0) for j in range(p)] + pp0[-1:]
        orders[0] += pp0
        orders[1] += _vpp_pp1(i, n)
    return simulate(orders, [0, 1, 1, 0], lambda r, k, s: float(taus[r][k]), comm)


def cpp_requests(taus, comm: float = 0.0) -> ScheduleResult:
    """Back-to-back requests under CPP."""
    orders = _cpp_orders([(i, len(t)) for i, t in enumerate(taus)])
    return simulate(orders, [0, 1], lambda r, k, s: 2.0 * taus[r][k], comm)
