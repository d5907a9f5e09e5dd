#!/usr/bin/env python
"""Chunked-prefill causal attention benchmark (one GB300 per rank).

One step = the whole prefill of one sequence of the chosen workload, chunk by
chunk: for every chunk k, append its K/V to the paged cache (block 64) and run
causal chunk attention of its queries over the cached prefix plus itself
(plus the LSE merge when the key range is split).  The metric is chunk
attention TFLOP/s (algorithmic FLOPs 2 (dq + dv) Hq (C P + C (C + 1) / 2) per
chunk, masked pairs not counted), reported for the whole step and per chunk
index, next to prefill tokens/s.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload long128k]
  python bench.py --impl reference      # the fp64 CPU oracle on host cores

With N > 1 (torchrun) every rank runs its own replica (weak scaling, no
collective on the data path); rank 0 prints one JSON line.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from chunked_prefill_causal_gb300 import workloads as W  # noqa: E402

METRIC = "chunk-attn TFLOP/s & % BF16 tensor peak vs chunk index; prefill tokens/s"

# DRAM bytes (read + write) per launch of the chunk-attention kernel, averaged
# over the 8 launches of one long128k step, from one ncu capture of
# dram__bytes_read.sum + dram__bytes_write.sum.  Valid only for the kernel sources whose
# digest is recorded with it; any change to them makes the figure stale (null).
TRAFFIC = {"long128k": {"sources_sha256": "83c21427d4320d7fd32e41bfa222dfc8ce86417cd0bfd8eeadb43e13dee4f593", "bytes_per_launch": 1.1879e9}}
KERNEL_SOURCES = ["chunk_attn_impl.cuh", "chunk_attn.cuh", "ptx.cuh"]


def kernel_sources_digest():
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "chunked_prefill_causal_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def recorded_traffic(workload):
    rec = TRAFFIC.get(workload)
    if rec and rec["sources_sha256"] == kernel_sources_digest():
        return rec["bytes_per_launch"]
    return None
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def chunk_flops(w, P, C):
    return 2.0 * (w.head_dim_qk + w.head_dim_v) * w.heads * (C * P + C * (C + 1) // 2)


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ dist
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = False
        self.backend = None

    def init(self, backend=None):
        """One process group per job: NCCL when the rank has a GPU, gloo otherwise."""
        if self.world > 1 and not self.pg:
            import torch.distributed as dist
            self.backend = backend or ("nccl" if torch.cuda.is_available() else "gloo")
            dist.init_process_group(self.backend)
            self.pg = True

    def barrier(self):
        if self.pg:
            import torch.distributed as dist
            dist.barrier()

    def max(self, x: float) -> float:
        """The maximum of x over all ranks (the job's time is its slowest rank's)."""
        if not self.pg:
            return x
        import torch.distributed as dist
        t = torch.tensor([x], dtype=torch.float64, device="cuda" if self.backend == "nccl" else "cpu")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())


# ------------------------------------------------------------------ CPU oracle sample
def oracle_inputs(w, seed, device_tensors=None):
    """Host copies of what the oracle needs for sampled rows of the
    workload's last full chunk (the one with the longest prefix): that chunk's
    queries and the K/V of the kv heads of 8 seeded query heads."""
    chunks = w.chunks()
    ci = max(range(len(chunks)), key=lambda i: chunks[i][0] * (chunks[i][1] == w.chunk))
    P, C = chunks[ci]
    rng = np.random.default_rng(seed)
    G = w.group
    heads = rng.choice(w.heads, size=min(8, w.heads), replace=False)
    kvh = sorted(set(int(h) // G for h in heads))
    if device_tensors is not None:
        qc, ks, vs = device_tensors
        q_host = qc[ci].to("cpu")
        k_host = torch.cat([k[:, kvh] for k in ks[:ci + 1]]).to("cpu")
        v_host = torch.cat([v[:, kvh] for v in vs[:ci + 1]]).to("cpu")
    else:
        q_host = W.chunk_tensors(w, ci, "cpu")[0]
        kk, vv = W.sequence_kv(w, P + C, "cpu")
        k_host, v_host = kk[:, kvh], vv[:, kvh]
    return {"ci": ci, "P": P, "C": C, "G": G, "heads": heads,
            "remap": {g: i for i, g in enumerate(kvh)}, "q": q_host,
            "k64": k_host.double().numpy(), "v64": v_host.double().numpy()}


def oracle_sample(w, inp, n_rows, seed, budget_s):
    """Times the fp64 oracle on up to n_rows sampled (token, head) rows.

    Returns (flops_done, seconds, rows_done, description).
    """
    import oracle

    rng = np.random.default_rng(seed)
    G, P, C = inp["G"], inp["P"], inp["C"]
    done_flops, done_rows = 0.0, 0
    t0 = time.perf_counter()
    per_batch = max(1, min(64, n_rows))
    while done_rows < n_rows:
        toks = rng.integers(0, C, size=per_batch)
        hs = rng.choice(inp["heads"], size=per_batch)
        local_heads = np.array([inp["remap"][int(h) // G] * G + int(h) % G for h in hs])
        qrows = inp["q"][toks, hs].double().numpy()
        oracle.attention_rows(qrows, local_heads, P + toks, inp["k64"], inp["v64"], G)
        done_flops += float(np.sum(2.0 * (w.head_dim_qk + w.head_dim_v) * (P + toks + 1)))
        done_rows += per_batch
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    desc = (f"{done_rows} sampled (token, head) rows of chunk {inp['ci']} (prefix {P}) of "
            f"{w.name}, fp64 NumPy oracle, {host_cores()} host cores")
    return done_flops, dt, done_rows, desc


# ------------------------------------------------------------------ reference arm
def run_reference(args, dist_):
    if dist_.rank != 0:
        return 0
    w = W.WORKLOADS[args.workload]
    flops = []
    times = []
    desc = ""
    inp = oracle_inputs(w, 7)
    for s in range(args.warmup + args.steps):
        f, dt, rows, desc = oracle_sample(w, inp, args.ref_rows, 1000 + s, budget_s=60.0)
        if s >= args.warmup:
            flops.append(f)
            times.append(dt)
    value = sum(flops) / sum(times) / 1e12
    cores = host_cores()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.mean(times), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": desc + " per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w):
    return {"workload": w.name, "heads": w.heads, "kv_heads": w.kv_heads,
            "head_dim_qk": w.head_dim_qk, "head_dim_v": w.head_dim_v, "seq_len": w.seq_len,
            "chunk": w.chunk, "chunks": len(w.chunks()), "kv_cache": "paged, block 64" if w.paged
            else "contiguous", "l2": "inputs larger than L2 (whole KV cache and each chunk's Q "
            "exceed 129 MB)" if w.seq_len >= 32768 else "small inputs"}


# ------------------------------------------------------------------ extras
def time_events(fn, iters, stream):
    """Median CUDA-event time (ms) of fn() over iters runs after one warm-up."""
    fn()
    torch.cuda.synchronize()
    times = []
    for _ in range(iters):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
    return statistics.median(times)


class MixedSetup:
    """The mixed micro-batch resident in HBM: 4 prefill chunks + decode rows."""

    def __init__(self, dev, decode_rows=None, fp8=False):
        from chunked_prefill_causal_gb300 import vpp
        m = W.MIXED if decode_rows is None else W.MixedWorkload(n_decode=decode_rows)
        self.m = m
        self.cu, self.ctx = m.batch()
        q, ks, vs = W.mixed_tensors(m, dev)
        table_np, pool = W.mixed_block_tables(m)
        self.table = torch.from_numpy(table_np).to(dev)
        self.kc = torch.zeros((pool, 64, m.kv_heads, m.head_dim_qk), dtype=torch.bfloat16, device=dev)
        self.vc = torch.zeros((pool, 64, m.kv_heads, m.head_dim_v), dtype=torch.bfloat16, device=dev)
        B = len(self.ctx)
        for b in range(B):
            P = int(self.ctx[b]) - int(self.cu[b + 1] - self.cu[b])
            if P > 0:
                vpp.vpp_kv_append(ks[b][:P], vs[b][:P], self.kc, self.vc, 0,
                                  block_table=self.table[b].contiguous())
        self.k_new = torch.cat([ks[b][int(self.ctx[b]) - int(self.cu[b + 1] - self.cu[b]):] for b in range(B)])
        self.v_new = torch.cat([vs[b][int(self.ctx[b]) - int(self.cu[b + 1] - self.cu[b]):] for b in range(B)])
        self.fp8 = fp8
        if fp8:
            # E4M3 pool with static per-kv-head scales from the value recipe
            # (8 standard deviations map to 448, so nothing saturates).
            s = torch.full((m.kv_heads,), 8.0 * m.std / 448.0, dtype=torch.float32, device=dev)
            self.ks8, self.vs8 = s, s.clone()
            self.kc8 = torch.zeros((pool, 64, m.kv_heads, m.head_dim_qk), dtype=torch.uint8, device=dev)
            self.vc8 = torch.zeros((pool, 64, m.kv_heads, m.head_dim_v), dtype=torch.uint8, device=dev)
            for b in range(B):
                P = int(self.ctx[b]) - int(self.cu[b + 1] - self.cu[b])
                if P > 0:
                    vpp.vpp_kv_append_fp8(ks[b][:P], vs[b][:P], self.kc8, self.vc8, self.ks8, self.vs8, 0,
                                          block_table=self.table[b].contiguous())
        del ks, vs
        self.q = q
        self.out = torch.empty((int(self.cu[-1]), m.heads, m.head_dim_v), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((m.heads, int(self.cu[-1])), dtype=torch.float32, device=dev)
        need = vpp.mixed_attn_workspace_size(self.cu, self.ctx, m.heads, m.kv_heads, m.head_dim_qk,
                                             m.head_dim_v)
        self.ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
        n_pre = len(m.prefill_prefixes)
        self.prefill_flops = sum(2.0 * (m.head_dim_qk + m.head_dim_v) * m.heads
                                 * (m.prefill_chunk * p + m.prefill_chunk * (m.prefill_chunk + 1) // 2)
                                 for p in m.prefill_prefixes)
        self.decode_flops = sum(2.0 * (m.head_dim_qk + m.head_dim_v) * m.heads * int(c)
                                for c in self.ctx[n_pre:])
        self.decode_bytes = sum(int(c) for c in self.ctx[n_pre:]) * m.kv_heads * (
            m.head_dim_qk + m.head_dim_v) * 2
        # The decode rows alone, as their own batch.
        self.cu_d = np.arange(B - n_pre + 1, dtype=np.int32)
        self.ctx_d = self.ctx[n_pre:].copy()
        self.q_d = q[int(self.cu[n_pre]):].contiguous()
        self.table_d = self.table[n_pre:].contiguous()
        self.out_d = torch.empty((B - n_pre, m.heads, m.head_dim_v), dtype=torch.bfloat16, device=dev)
        need_d = vpp.mixed_attn_workspace_size(self.cu_d, self.ctx_d, m.heads, m.kv_heads, m.head_dim_qk,
                                               m.head_dim_v)
        self.ws_d = torch.empty(max(need_d, 256), dtype=torch.uint8, device=dev)
        if fp8:
            need8 = vpp.mixed_attn_fp8_workspace_size(self.cu, self.ctx, m.heads, m.kv_heads, m.head_dim_qk,
                                                      m.head_dim_v)
            self.ws8 = torch.empty(max(need8, 256), dtype=torch.uint8, device=dev)
            need8w = vpp.mixed_attn_fp8_widen_workspace_size(self.cu, self.ctx, m.heads, m.kv_heads,
                                                             m.head_dim_qk, m.head_dim_v)
            self.ws8w = torch.empty(max(need8w, 256), dtype=torch.uint8, device=dev)

    def step_fp8(self):
        from chunked_prefill_causal_gb300 import vpp
        vpp.vpp_kv_append_varlen_fp8(self.k_new, self.v_new, self.kc8, self.vc8, self.ks8, self.vs8, self.table,
                                     self.cu, self.ctx)
        vpp.vpp_mixed_attn_fp8(self.q, self.kc8, self.vc8, self.ks8, self.vs8, self.table, self.cu, self.ctx,
                               out=self.out, lse=self.lse, workspace=self.ws8)

    def step_fp8_widened(self):
        """As step_fp8, with a workspace that holds the bf16 widening of the
        prefill segments' contexts."""
        from chunked_prefill_causal_gb300 import vpp
        vpp.vpp_kv_append_varlen_fp8(self.k_new, self.v_new, self.kc8, self.vc8, self.ks8, self.vs8, self.table,
                                     self.cu, self.ctx)
        vpp.vpp_mixed_attn_fp8(self.q, self.kc8, self.vc8, self.ks8, self.vs8, self.table, self.cu, self.ctx,
                               out=self.out, lse=self.lse, workspace=self.ws8w)

    def decode_only_fp8(self):
        from chunked_prefill_causal_gb300 import vpp
        vpp.vpp_mixed_attn_fp8(self.q_d, self.kc8, self.vc8, self.ks8, self.vs8, self.table_d, self.cu_d,
                               self.ctx_d, out=self.out_d, workspace=self.ws_d)

    def step(self):
        from chunked_prefill_causal_gb300 import vpp
        vpp.vpp_kv_append_varlen(self.k_new, self.v_new, self.kc, self.vc, self.table, self.cu, self.ctx)
        vpp.vpp_mixed_attn(self.q, self.kc, self.vc, self.table, self.cu, self.ctx, out=self.out,
                           lse=self.lse, workspace=self.ws)

    def decode_only(self):
        from chunked_prefill_causal_gb300 import vpp
        vpp.vpp_mixed_attn(self.q_d, self.kc, self.vc, self.table_d, self.cu_d, self.ctx_d,
                           out=self.out_d, workspace=self.ws_d)


def mixed_launches(n_prefill, n_decode):
    """Kernel launches of one mixed step: the varlen append, the decode kernel
    and its LSE merge when there are decode rows, and one chunk-attention
    launch per 64 prefill segments."""
    return 1 + (2 if n_decode > 0 else 0) + (n_prefill + 63) // 64


def mixed_bound_ms(prefill_flops, decode_bytes, peak_tf, hbm):
    """Combined lower bound of a mixed step: the tensor-bound prefill work at
    the bf16 peak or the HBM-bound decode reads at the copy bandwidth,
    whichever is longer (the two can overlap at best)."""
    return max(prefill_flops / (peak_tf * 1e12), decode_bytes / (hbm * 1e9)) * 1e3


def measure_mixed(dev, stream, hbm, peak_tf, decode_rows=None):
    ms = MixedSetup(dev, decode_rows)
    step_ms = time_events(ms.step, 10, stream)
    dec_ms = time_events(ms.decode_only, 10, stream)
    gbs = ms.decode_bytes / (dec_ms / 1e3) / 1e9
    bound = mixed_bound_ms(ms.prefill_flops, ms.decode_bytes, peak_tf, hbm)
    n_pre = len(ms.m.prefill_prefixes)
    return {"workload": "mixed: 4 prefill chunks of 2048 at prefixes {0,16384,65536,122880} + "
                        f"{len(ms.ctx_d)} decode rows, ctx ~ U[1024,32768]; 32/8 heads, d 128",
            "step_ms": round(step_ms, 3),
            "bound_ms": round(bound, 3),
            "frac_of_bound": round(bound / step_ms, 4),
            "prefill_tflop": round(ms.prefill_flops / 1e12, 3),
            "decode_only_ms": round(dec_ms, 3),
            "decode_bytes": int(ms.decode_bytes),
            "decode_gbs": round(gbs, 1), "decode_frac_hbm": round(gbs / hbm, 4),
            "prefill_plus_decode_tflops": round((ms.prefill_flops + ms.decode_flops) / (step_ms / 1e3) / 1e12, 1),
            "launches_per_step": mixed_launches(n_pre, len(ms.ctx_d))}


def time_flushed(fn, iters, stream, flush):
    """Median CUDA-event time (ms) of fn() over iters runs, each after a write
    of `flush` (a buffer larger than L2) outside the timed region."""
    fn()
    torch.cuda.synchronize()
    times = []
    for _ in range(iters):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
    return statistics.median(times)


def measure_chunks(dev, stream, name, chunk_ids, peak_tf, peak_burst, iters, warm=False):
    """Chunk attention of chosen chunks of a workload, each timed in isolation
    (L2 flushed before every run) with the K/V of all earlier chunks and its
    own already in the paged cache, through the product call with the
    library's own split choice.  Rows: [k, prefix, chunk, ms, TFLOP/s,
    fraction of the sustained peak, fraction of the burst peak], and with
    warm=True an 8th column: the median ms of back-to-back runs without the
    flush (whatever of the chunk's inputs L2 still holds)."""
    from chunked_prefill_causal_gb300 import vpp
    w = W.WORKLOADS[name]
    chunks = w.chunks()
    ids = sorted(set(range(len(chunks)) if chunk_ids is None else chunk_ids))
    last = ids[-1]
    nb = W.blocks_for(chunks[last][0] + chunks[last][1])
    pool = nb + 64
    table = torch.from_numpy(W.block_table(nb, pool, w.seed + 99)).to(dev)
    kc = torch.zeros((pool, 64, w.kv_heads, w.head_dim_qk), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros((pool, 64, w.kv_heads, w.head_dim_v), dtype=torch.bfloat16, device=dev)
    qs = {}
    for ci in range(last + 1):
        q, k, v = W.chunk_tensors(w, ci, dev)
        vpp.vpp_kv_append(k, v, kc, vc, chunks[ci][0], block_table=table)
        if ci in ids:
            qs[ci] = q
        del q, k, v
    ws_need = max(vpp.chunk_attn_workspace_size(vpp.VPP_BF16, chunks[ci][0], chunks[ci][1], w.heads,
                                                w.kv_heads, w.head_dim_qk, w.head_dim_v) for ci in ids)
    ws = torch.empty(max(ws_need, 256), dtype=torch.uint8, device=dev)
    out = torch.empty((max(chunks[ci][1] for ci in ids), w.heads, w.head_dim_v), dtype=torch.bfloat16,
                      device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    rows = []
    for ci in ids:
        P, C = chunks[ci]
        t = time_flushed(lambda: vpp.vpp_chunk_attn_ex(qs[ci], kc, vc, P, block_table=table, out=out[:C],
                                                       workspace=ws), iters, stream, flush)
        tf = chunk_flops(w, P, C) / (t / 1e3) / 1e12
        rows.append([ci, P, C, round(t, 3), round(tf, 1), round(tf / peak_tf, 4), round(tf / peak_burst, 4)])
        if warm:
            rows[-1].append(round(time_events(lambda: vpp.vpp_chunk_attn_ex(
                qs[ci], kc, vc, P, block_table=table, out=out[:C], workspace=ws), iters, stream), 3))
    if vpp.vpp_last_device_status() != 0:
        raise RuntimeError(f"device status word reported an error during the {name} chunks")
    tot_f = sum(chunk_flops(w, r[1], r[2]) for r in rows)
    tot_ms = sum(r[3] for r in rows)
    tf = tot_f / (tot_ms / 1e3) / 1e12
    return {"workload": name, "heads": [w.heads, w.kv_heads], "head_dims": [w.head_dim_qk, w.head_dim_v],
            "l2": "flushed before each run" + ("; ms_warm without the flush" if warm else ""),
            "columns": ["k", "prefix", "chunk", "ms", "tflops", "frac", "frac_burst"] + (["ms_warm"] if warm else []),
            "rows": rows, "tflops": round(tf, 1), "frac": round(tf / peak_tf, 4),
            "frac_burst": round(tf / peak_burst, 4)}


def measure_cpu_full(dev, stream, gqa_rows):
    """Whole-chunk oracle times (fp64 NumPy on this host's cores) beside the
    GPU's, for the chunks small enough to run in full within the bench: every
    tiny chunk (fp32 inputs, contiguous cache) and gqa32k chunks 0 and 1; the
    other configs' CPU times are extrapolated from the sampled rate.  The
    inputs are the GPU run's, copied to the host.  Rows: [k, prefix, chunk,
    GPU ms, oracle s]."""
    import oracle
    from chunked_prefill_causal_gb300 import vpp
    out = {"cores": host_cores(), "columns": ["k", "prefix", "chunk", "gpu_ms", "oracle_s"], "tiny": [],
           "gqa32k": []}
    w = W.WORKLOADS["tiny"]
    kc = torch.zeros((w.seq_len, w.kv_heads, w.head_dim_qk), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros((w.seq_len, w.kv_heads, w.head_dim_v), dtype=torch.bfloat16, device=dev)
    ks, vs = [], []
    for ci, (P, C) in enumerate(w.chunks()):
        q, k, v = W.chunk_tensors(w, ci, dev)
        vpp.vpp_kv_append(k, v, kc, vc, P)
        ks.append(k.cpu())
        vs.append(v.cpu())
        ws = torch.empty(max(256, vpp.chunk_attn_workspace_size(vpp.VPP_FP32, P, C, w.heads, w.kv_heads,
                                                                w.head_dim_qk, w.head_dim_v)),
                         dtype=torch.uint8, device=dev)
        out_t = torch.empty((C, w.heads, w.head_dim_v), dtype=torch.bfloat16, device=dev)
        t_gpu = time_events(lambda: vpp.vpp_chunk_attn_ex(q, kc, vc, P, out=out_t, workspace=ws), 20, stream)
        qh = q.cpu().double().numpy()
        kh, vh = torch.cat(ks).double().numpy(), torch.cat(vs).double().numpy()
        t0 = time.perf_counter()
        oracle.causal_chunk_attention(qh, kh, vh, P)
        out["tiny"].append([ci, P, C, round(t_gpu, 4), round(time.perf_counter() - t0, 4)])
    w = W.WORKLOADS["gqa32k"]
    gpu_ms = {r[0]: r[3] for r in gqa_rows}
    for ci in (0, 1):
        P, C = w.chunks()[ci]
        qh = W.chunk_tensors(w, ci, dev)[0].cpu().double().numpy()
        kk, vv = W.sequence_kv(w, P + C, dev)
        kh, vh = kk.cpu().double().numpy(), vv.cpu().double().numpy()
        del kk, vv
        t0 = time.perf_counter()
        oracle.causal_chunk_attention(qh, kh, vh, P)
        out["gqa32k"].append([ci, P, C, gpu_ms.get(ci), round(time.perf_counter() - t0, 2)])
    return out


def measure_append(dev, stream, hbm):
    """One MLA-chunk-sized append: 24576 tokens x 128 kv heads x (192 + 128) bf16."""
    from chunked_prefill_causal_gb300 import vpp
    C, H, dq, dv = 24576, 128, 192, 128
    g = torch.Generator(device=dev).manual_seed(77)
    k = torch.randn((C, H, dq), generator=g, device=dev).to(torch.bfloat16)
    v = torch.randn((C, H, dv), generator=g, device=dev).to(torch.bfloat16)
    nb = C // 64 + 8
    table = torch.from_numpy(W.block_table(C // 64, nb, 5)).to(dev)
    kc = torch.empty((nb, 64, H, dq), dtype=torch.bfloat16, device=dev)
    vc = torch.empty((nb, 64, H, dv), dtype=torch.bfloat16, device=dev)
    t = time_events(lambda: vpp.vpp_kv_append(k, v, kc, vc, 0, block_table=table), 10, stream)
    byts = 2 * C * H * (dq + dv) * 2
    return {"tokens": C, "kv_heads": H, "head_dims": [dq, dv], "bytes_moved": byts, "ms": round(t, 4),
            "gbs": round(byts / (t / 1e3) / 1e9, 1), "frac_hbm": round(byts / (t / 1e3) / 1e9 / hbm, 4)}


def measure_fp8(dev, stream, hbm, w, chunks):
    """fp8 (E4M3) KV cache: the quantising append at the MLA-chunk size, the
    mixed batch's decode rows and whole step over an fp8 pool, and the last
    chunk of the chunked-prefill workload through the fp8 path (widening to
    bf16 + the attention kernel) against the bf16 path."""
    from chunked_prefill_causal_gb300 import vpp
    out = {}
    C, H, dq, dv = 24576, 128, 192, 128
    g = torch.Generator(device=dev).manual_seed(77)
    k = torch.randn((C, H, dq), generator=g, device=dev).to(torch.bfloat16)
    v = torch.randn((C, H, dv), generator=g, device=dev).to(torch.bfloat16)
    nb = C // 64 + 8
    table = torch.from_numpy(W.block_table(C // 64, nb, 5)).to(dev)
    kc = torch.empty((nb, 64, H, dq), dtype=torch.uint8, device=dev)
    vc = torch.empty((nb, 64, H, dv), dtype=torch.uint8, device=dev)
    s = torch.full((H,), 8.0 / 448.0, dtype=torch.float32, device=dev)
    t = time_events(lambda: vpp.vpp_kv_append_fp8(k, v, kc, vc, s, s, 0, block_table=table), 10, stream)
    byts = C * H * (dq + dv) * 3
    out["append"] = {"tokens": C, "kv_heads": H, "head_dims": [dq, dv], "bytes_moved": byts, "ms": round(t, 4),
                     "gbs": round(byts / (t / 1e3) / 1e9, 1), "frac_hbm": round(byts / (t / 1e3) / 1e9 / hbm, 4)}
    del k, v, kc, vc
    torch.cuda.empty_cache()

    ms = MixedSetup(dev, fp8=True)
    dec = time_events(ms.decode_only, 10, stream)
    dec8 = time_events(ms.decode_only_fp8, 10, stream)
    step = time_events(ms.step, 10, stream)
    step8 = time_events(ms.step_fp8, 10, stream)
    step8w = time_events(ms.step_fp8_widened, 10, stream)
    b8 = ms.decode_bytes // 2
    out["decode"] = {"rows": len(ms.ctx_d), "bytes_fp8": int(b8), "ms_fp8": round(dec8, 3), "ms_bf16": round(dec, 3),
                     "gbs_fp8": round(b8 / (dec8 / 1e3) / 1e9, 1),
                     "frac_hbm_fp8": round(b8 / (dec8 / 1e3) / 1e9 / hbm, 4),
                     "speedup_vs_bf16": round(dec / dec8, 3)}
    out["mixed_step"] = {"ms_fp8": round(step8, 3), "ms_fp8_widened": round(step8w, 3), "ms_bf16": round(step, 3)}
    del ms
    torch.cuda.empty_cache()

    # Last chunk of the chunked-prefill workload: widening + attention.
    P, C = chunks[-1]
    n = P + C
    s = torch.full((w.kv_heads,), 8.0 * w.std / 448.0, dtype=torch.float32, device=dev)
    kc8 = torch.empty((n, w.kv_heads, w.head_dim_qk), dtype=torch.uint8, device=dev)
    vc8 = torch.empty((n, w.kv_heads, w.head_dim_v), dtype=torch.uint8, device=dev)
    kc16 = torch.empty((n, w.kv_heads, w.head_dim_qk), dtype=torch.bfloat16, device=dev)
    vc16 = torch.empty((n, w.kv_heads, w.head_dim_v), dtype=torch.bfloat16, device=dev)
    q = None
    for ci, (p0, c0) in enumerate(chunks):
        qi, ki, vi = W.chunk_tensors(w, ci, dev)
        vpp.vpp_kv_append_fp8(ki, vi, kc8, vc8, s, s, p0)
        vpp.vpp_kv_append(ki, vi, kc16, vc16, p0)
        q = qi
        del ki, vi
    o = torch.empty((C, w.heads, w.head_dim_v), dtype=torch.bfloat16, device=dev)
    ws8 = torch.empty(max(256, vpp.chunk_attn_fp8_workspace_size(P, C, w.heads, w.kv_heads, w.head_dim_qk,
                                                                 w.head_dim_v, 1)), dtype=torch.uint8, device=dev)
    ws8w = torch.empty(vpp.chunk_attn_fp8_widen_workspace_size(P, C, w.heads, w.kv_heads, w.head_dim_qk,
                                                               w.head_dim_v, 1), dtype=torch.uint8, device=dev)
    t16 = time_events(lambda: vpp.vpp_chunk_attn_ex(q, kc16, vc16, P, out=o, num_splits=1), 5, stream)
    t8 = time_events(lambda: vpp.vpp_chunk_attn_fp8(q, kc8, vc8, s, s, P, out=o, num_splits=1, workspace=ws8),
                     5, stream)
    t8w = time_events(lambda: vpp.vpp_chunk_attn_fp8(q, kc8, vc8, s, s, P, out=o, num_splits=1, workspace=ws8w),
                      5, stream)
    # in the kernel (no copy of the cache) / widened once into a bf16 copy / bf16 cache
    out["prefill_last_chunk"] = {"prefix": P, "chunk": C, "ms_fp8": round(t8, 3), "ms_fp8_widened": round(t8w, 3),
                                 "ms_bf16": round(t16, 3), "widened_copy_bytes": int(ws8w.numel()),
                                 "fp8_overhead": round(t8 / t16 - 1.0, 4)}
    return out


class TopkSetup:
    """The dsa128k workload resident in HBM for top-k sparse prefix attention:
    every chunk's q, the whole context's K/V in a bf16 and an E4M3 paged cache,
    and each chunk's index rows (TOPK listed keys per query token)."""

    def __init__(self, dev):
        from chunked_prefill_causal_gb300 import vpp
        w = W.WORKLOADS["dsa128k"]
        self.w = w
        self.chunks = w.chunks()
        nb = W.blocks_for(w.seq_len)
        self.table = torch.from_numpy(W.block_table(nb, nb + 8, w.seed + 99)).to(dev)
        self.kc = torch.zeros((nb + 8, 64, w.kv_heads, w.head_dim_qk), dtype=torch.bfloat16, device=dev)
        self.vc = torch.zeros_like(self.kc)
        self.kc8 = torch.zeros((nb + 8, 64, w.kv_heads, w.head_dim_qk), dtype=torch.uint8, device=dev)
        self.vc8 = torch.zeros_like(self.kc8)
        # |k|, |v| < 0.5 in this recipe: 0.5 maps to 448
        self.s8 = torch.full((w.kv_heads,), 0.5 / 448.0, dtype=torch.float32, device=dev)
        self.qs, self.idx, self.lens = [], [], []
        for ci, (p0, c0) in enumerate(self.chunks):
            qi, ki, vi = W.chunk_tensors(w, ci, dev)
            vpp.vpp_kv_append(ki, vi, self.kc, self.vc, p0, block_table=self.table)
            vpp.vpp_kv_append_fp8(ki, vi, self.kc8, self.vc8, self.s8, self.s8, p0, block_table=self.table)
            self.qs.append(qi)
            del ki, vi
            idx, lens = W.topk_indices(p0, c0, W.TOPK, ci, device=dev)
            self.idx.append(idx)
            self.lens.append(lens)
        self.out = torch.empty((w.chunk, w.heads, w.head_dim_v), dtype=torch.bfloat16, device=dev)
        self.ws = torch.empty(max(vpp.topk_chunk_attn_workspace_size(w.chunk, W.TOPK, w.heads, w.head_dim_qk), 256),
                              dtype=torch.uint8, device=dev)

    def gathered_bytes(self, ci, fp8=False):
        """Algorithmic bytes of chunk ci: every listed key's K and V rows, all
        kv heads, once per query token that lists it."""
        w = self.w
        n_listed = int(self.lens[ci].to(torch.int64).sum())
        return n_listed * w.kv_heads * (w.head_dim_qk + w.head_dim_v) * (1 if fp8 else 2)

    def run(self, ci, fp8=False):
        from chunked_prefill_causal_gb300 import vpp
        P, C = self.chunks[ci]
        if fp8:
            vpp.vpp_topk_chunk_attn_fp8(self.qs[ci], self.kc8, self.vc8, self.s8, self.s8, P, self.idx[ci],
                                        self.lens[ci], block_table=self.table, out=self.out[:C], workspace=self.ws)
        else:
            vpp.vpp_topk_chunk_attn(self.qs[ci], self.kc, self.vc, P, self.idx[ci], self.lens[ci],
                                    block_table=self.table, out=self.out[:C], workspace=self.ws)


def measure_topk(dev, stream, hbm, peak_tf):
    """Top-k sparse prefix attention (DSA-style) on the dsa128k workload
    (32/8 heads, d 128, 8 chunks of 16384, TOPK listed keys per query token)
    against dense chunk attention on the same shapes, and the two-rank
    schedules simulated on each set of per-chunk latencies."""
    from chunked_prefill_causal_gb300 import vpp
    ts_ = TopkSetup(dev)
    w = ts_.w
    rows, sparse_ms, dense_ms = [], [], []
    for ci, (P, C) in enumerate(ts_.chunks):
        ts = time_events(lambda: ts_.run(ci), 5, stream)
        ts8 = time_events(lambda: ts_.run(ci, fp8=True), 5, stream)
        td = time_events(lambda: vpp.vpp_chunk_attn_ex(ts_.qs[ci], ts_.kc, ts_.vc, P, block_table=ts_.table,
                                                       out=ts_.out[:C], num_splits=1), 3, stream)
        n_listed = int(ts_.lens[ci].to(torch.int64).sum())
        byts = ts_.gathered_bytes(ci)
        fl = 2.0 * (w.head_dim_qk + w.head_dim_v) * w.heads * n_listed
        dfl = 2.0 * (w.head_dim_qk + w.head_dim_v) * w.heads * (C * P + C * (C + 1) // 2)
        sparse_ms.append(ts)
        dense_ms.append(td)
        rows.append({"k": ci, "prefix": P, "sparse_ms": round(ts, 3), "dense_ms": round(td, 3),
                     "gathered_gb": round(byts / 1e9, 2), "sparse_gbs": round(byts / (ts / 1e3) / 1e9, 1),
                     "sparse_fp8_ms": round(ts8, 3), "sparse_fp8_gbs": round(byts / 2 / (ts8 / 1e3) / 1e9, 1),
                     "sparse_tflops": round(fl / (ts / 1e3) / 1e12, 1),
                     "dense_tflops": round(dfl / (td / 1e3) / 1e12, 1)})
    if vpp.vpp_last_device_status() != 0:
        raise RuntimeError("device status word reported an error")
    return {"workload": f"dsa128k: 32/8 heads, d 128, 8 chunks of 16384, {W.TOPK} listed keys per query token",
            "gathered": "each listed key's K and V rows once per query token that lists it; tokens share keys, "
                        "so part of it is served from L2 and the rate can exceed the HBM copy peak",
            "per_chunk": rows,
            "schedule_dense": schedule_summary(dense_ms), "schedule_sparse": schedule_summary(sparse_ms)}


def run_topk(args, dist_):
    """Top-k sparse prefix attention of dsa128k as the step: the chunks named
    by --topk-chunks (default all 8), one vpp_topk_chunk_attn[_fp8] launch each
    over the cache of the whole context.  Reports gathered bytes per second."""
    from chunked_prefill_causal_gb300 import vpp

    dist_.init()
    dev = torch.device("cuda", dist_.local)
    torch.cuda.set_device(dev)
    vpp.load()
    stream = torch.cuda.current_stream()
    fp8 = args.kv_dtype == "fp8"
    ts_ = TopkSetup(dev)
    sel = [int(c) for c in args.topk_chunks.split(",")] if args.topk_chunks else list(range(len(ts_.chunks)))
    if any(c < 0 or c >= len(ts_.chunks) for c in sel):
        raise SystemExit(f"--topk-chunks: chunk indices are 0..{len(ts_.chunks) - 1}")

    def step():
        for ci in sel:
            ts_.run(ci, fp8)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    dist_.barrier()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    dist_.barrier()
    if vpp.vpp_last_device_status() != 0:
        raise RuntimeError("device status word reported an error")
    el = dist_.max(e0.elapsed_time(e1) / 1e3)
    byts = sum(ts_.gathered_bytes(ci, fp8) for ci in sel)
    if dist_.rank == 0:
        print(json.dumps({
            "metric": "top-k gathered bytes per second", "value": byts * args.steps * dist_.world / el / 1e9,
            "unit": "GB/s", "n_gpus": dist_.world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * el / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp8" if fp8 else "bf16", "data": "synthetic",
            "config": {"workload": "dsa128k top-k", "chunks": sel, "topk": W.TOPK, "heads": ts_.w.heads,
                       "kv_heads": ts_.w.kv_heads, "head_dim": ts_.w.head_dim_qk,
                       "kv_cache": "E4M3 codes, per-kv-head scales" if fp8 else "bf16"}}), flush=True)
    return 0


def measure_cost_model(dev, stream, n_batches=48, n_train=32, seed=11):
    """Times random mixed micro-batches through vpp_mixed_attn and fits the
    micro-batch latency model (cost_model.py) to them: MAPE on held-out
    batches for the full model and for token counts alone, and the error of
    the online (RLS) predictions."""
    from chunked_prefill_causal_gb300 import vpp
    from chunked_prefill_causal_gb300.cost_model import LatencyModel, MicroBatch, mape
    H, Hkv, d = 32, 8, 128
    rng = np.random.default_rng(seed)
    specs = []
    for _ in range(n_batches):
        pre = [(int(rng.integers(0, 1536)) * 64, int(rng.choice([256, 512, 1024, 2048, 4096])))
               for _ in range(int(rng.integers(0, 4)))]
        dec = [int(x) for x in rng.integers(1024, 32769, size=int(rng.integers(0, 129)))]
        if not pre and not dec:
            dec = [4096]
        specs.append(MicroBatch(tuple(pre), tuple(dec)))
    max_tokens = max(sum(p + c for p, c in b.prefill) + sum(b.decode) for b in specs)
    pool = W.blocks_for(max_tokens) + 512
    kc = torch.zeros((pool, 64, Hkv, d), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    times = []
    for b in specs:
        qlen = [c for _, c in b.prefill] + [1] * len(b.decode)
        ctx = [p + c for p, c in b.prefill] + list(b.decode)
        cu = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
        ctx = np.asarray(ctx, dtype=np.int32)
        need = [W.blocks_for(int(c)) for c in ctx]
        table = np.zeros((len(ctx), max(need)), dtype=np.int32)
        off = 0
        for i, n in enumerate(need):
            table[i, :n] = np.arange(off, off + n)
            off += n
        table_d = torch.from_numpy(table).to(dev)
        q = torch.randn((int(cu[-1]), H, d), device=dev).to(torch.bfloat16)
        out = torch.empty_like(q)
        wsz = vpp.mixed_attn_workspace_size(cu, ctx, H, Hkv, d, d)
        ws = torch.empty(max(wsz, 256), dtype=torch.uint8, device=dev)
        t = time_events(lambda: vpp.vpp_mixed_attn(q, kc, vc, table_d, cu, ctx, out=out, workspace=ws), 5, stream)
        times.append(t)
    tr, te = slice(0, n_train), slice(n_train, n_batches)
    full = LatencyModel()
    full.fit_all(specs[tr], times[tr])
    tok = LatencyModel()
    tok.fit_offline(specs[tr], times[tr])
    online = LatencyModel(forgetting=0.98)
    online.alpha = tok.alpha.copy()
    online_pred = [online.update(b, t) for b, t in zip(specs, times)]
    return {"batches": n_batches, "train": n_train,
            "heldout_mape_full": round(mape([full.predict(b) for b in specs[te]], times[te]), 4),
            "heldout_mape_tokens_only": round(mape([tok.predict(b) for b in specs[te]], times[te]), 4),
            "online_rls_mape_last16": round(mape(online_pred[-16:], times[-16:]), 4),
            "coefficients_ms": {"alpha": [round(float(x), 6) for x in full.alpha],
                                "beta": [round(float(x), 6) for x in full.beta],
                                "units": "alpha: [1, N/2^10]; beta: [sum Lpast*Lpre/2^30, sum Lpre^2/2^30, "
                                         "sum Ldec/2^20]"},
            "latency_ms_range": [round(min(times), 3), round(max(times), 3)]}


def schedule_summary(tau_ms):
    """Two-rank CPP vs V-shaped VPP vs VPP with pipelined packing, simulated
    on the measured per-chunk attention latencies tau_k (one layer, ms): a
    stage's time scales with its layer count, which leaves every ratio as is."""
    from chunked_prefill_causal_gb300 import schedule_sim as S
    n = len(tau_ms)
    c, v = S.cpp(tau_ms), S.vpp(tau_ms)
    two_plain = S.vpp_requests([tau_ms, tau_ms])
    two_packed = S.vpp_requests([tau_ms, tau_ms], pack=True)
    two_cpp = S.cpp_requests([tau_ms, tau_ms])
    packed, _ = S.pack_leading_chunks(S.drain_window_from_taus(tau_ms), tau_ms) if n > 1 else (0, 0.0)
    eq3b = [abs(tau_ms[k - 1] + tau_ms[k + 1] - 2 * tau_ms[k]) / (2 * tau_ms[k]) for k in range(1, n - 1)]
    r = lambda x: round(float(x), 4)
    return {"chunks": n, "tau_ms": [r(t) for t in tau_ms],
            "eq3b_max_rel_residual": r(max(eq3b)) if eq3b else None,
            "boundary_tau1_over_2tau0": r(tau_ms[1] / (2 * tau_ms[0])) if n > 1 else None,
            "cpp_ms": r(c.makespan), "vpp_ms": r(v.makespan), "vpp_speedup": r(c.makespan / v.makespan),
            "cpp_bubble_ratio": r(c.bubble_ratio), "vpp_bubble_ratio": r(v.bubble_ratio),
            "drain_idle_ms": r(S.drain_idle(v, 0, n)) if n > 1 else None,
            "drain_estimate_ms": r(S.drain_window_from_taus(tau_ms)) if n > 1 else None,
            "drain_estimate_eq2_ms": r(S.drain_window(n, tau_ms[0])),
            "two_requests": {"cpp_ms": r(two_cpp.makespan), "vpp_ms": r(two_plain.makespan),
                             "vpp_packed_ms": r(two_packed.makespan), "packed_chunks": packed,
                             "cpp_bubble_ratio": r(two_cpp.bubble_ratio),
                             "vpp_bubble_ratio": r(two_plain.bubble_ratio),
                             "vpp_packed_bubble_ratio": r(two_packed.bubble_ratio)}}


# ------------------------------------------------------------------ our arm
# exp2 throughput of the MUFU unit on GB300, ex2.approx.ftz.f32 with enough
# independent work: 32 per cycle per SM (measured: 31.2 at 128 threads per SM,
# 32.0 at 256 to 1024).
EX2_PER_CLK_PER_SM = 32


def ex2_bound(w, chunks, attn_ms_step, clk, sms):
    """The secondary bound of the softmax: one exp2 per unmasked score per
    head, at the MUFU rate of `sms` SMs at the sampled clock, against the
    step's attention time."""
    exps = sum(w.heads * (C * P + C * (C + 1) // 2) for P, C in chunks)
    mhz = (clk or {}).get("sm_mhz") or (clk or {}).get("sm_max_mhz")
    if not mhz:
        return None
    ms = exps / (EX2_PER_CLK_PER_SM * sms * mhz * 1e6) * 1e3
    return {"exps_per_step": exps, "per_clk_per_sm": EX2_PER_CLK_PER_SM, "sm_mhz": mhz, "ms": round(ms, 3),
            "frac_of_attention_time": round(ms / attn_ms_step, 4)}


def run_ours(args, dist_):
    from chunked_prefill_causal_gb300 import vpp

    dist_.init()
    dev = torch.device("cuda", dist_.local)
    torch.cuda.set_device(dev)
    vpp.load()
    w = W.WORKLOADS[args.workload]
    chunks = w.chunks()
    pk, pk_src = peaks()
    peak_tf = float(pk.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    peak_tf_burst = float(pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm = float(pk.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))

    # Inputs resident in HBM.
    qs, ks, vs = [], [], []
    for ci in range(len(chunks)):
        q, k, v = W.chunk_tensors(w, ci, dev)
        qs.append(q)
        ks.append(k)
        vs.append(v)
    nb_need = W.blocks_for(w.seq_len)
    pool = nb_need + 64
    table = torch.from_numpy(W.block_table(nb_need, pool, w.seed + 99)).to(dev)
    kc = torch.zeros((pool, 64, w.kv_heads, w.head_dim_qk), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros((pool, 64, w.kv_heads, w.head_dim_v), dtype=torch.bfloat16, device=dev)
    Cmax = max(c for _, c in chunks)
    out = torch.empty((Cmax, w.heads, w.head_dim_v), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.heads, Cmax), dtype=torch.float32, device=dev)
    ws_need = max(vpp.chunk_attn_workspace_size(vpp.VPP_BF16, P, C, w.heads, w.kv_heads,
                                                w.head_dim_qk, w.head_dim_v) for P, C in chunks)
    ws = torch.empty(max(ws_need, 256), dtype=torch.uint8, device=dev)
    splits = [vpp.chunk_attn_num_splits(P, C, w.heads, w.kv_heads, w.head_dim_qk, w.head_dim_v)
              for P, C in chunks]
    launches_per_step = sum(2 + (1 if s > 1 else 0) for s in splits)
    stream = torch.cuda.current_stream()
    flops = [chunk_flops(w, P, C) for P, C in chunks]

    def step(events=None):
        for ci, (P, C) in enumerate(chunks):
            vpp.vpp_kv_append(ks[ci], vs[ci], kc, vc, P, block_table=table)
            if events is not None:
                events[ci][0].record(stream)
            vpp.vpp_chunk_attn_ex(qs[ci], kc, vc, P, block_table=table,
                                  out=out[:C], lse=lse[:, :C] if C == Cmax else None,
                                  workspace=ws)
            if events is not None:
                events[ci][1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if vpp.vpp_last_device_status() != 0:
        raise RuntimeError("device status word reported an error during warm-up")

    ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in chunks]
          for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dist_.local)
    dist_.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)  # let the sampler take its first reading
    t_start.record(stream)
    for s in range(args.steps):
        step(ev[s])
    t_end.record(stream)
    torch.cuda.synchronize()
    dist_.barrier()
    clk = clocks.stop()
    status = vpp.vpp_last_device_status()
    if status != 0:
        raise RuntimeError(f"device status word reported {status} in the timed region")
    elapsed = t_start.elapsed_time(t_end) / 1e3
    elapsed = dist_.max(elapsed)
    total_flops = sum(flops) * args.steps * dist_.world
    value = total_flops / elapsed / 1e12

    per_chunk_ms = [statistics.median(ev[s][ci][0].elapsed_time(ev[s][ci][1]) for s in range(args.steps))
                    for ci in range(len(chunks))]
    attn_ms_step = sum(per_chunk_ms)
    per_chunk = []
    for ci, (P, C) in enumerate(chunks):
        tf = flops[ci] / (per_chunk_ms[ci] / 1e3) / 1e12
        per_chunk.append({"k": ci, "prefix": P, "chunk": C, "ms": round(per_chunk_ms[ci], 4),
                          "tflops": round(tf, 1), "frac_peak": round(tf / peak_tf, 4),
                          "splits": splits[ci]})
    # Affine fit of latency vs chunk index (the per-stage law tau_k of the pages
    # is linear in k; attention alone grows like (2k + 1)).
    ks_idx = np.arange(len(chunks))
    full = [i for i, (_, C) in enumerate(chunks) if C == w.chunk]
    fit = None
    if len(full) >= 3:
        a, b = np.polyfit(ks_idx[full], np.array(per_chunk_ms)[full], 1)
        pred = a * ks_idx[full] + b
        y = np.array(per_chunk_ms)[full]
        r2 = 1 - np.sum((y - pred) ** 2) / np.sum((y - y.mean()) ** 2)
        fit = {"ms_per_k": round(float(a), 4), "ms_at_k0": round(float(b), 4), "r2": round(float(r2), 5)}

    achieved = sum(flops) / (attn_ms_step / 1e3) / 1e12
    late = [c for c in per_chunk if c["k"] >= len(chunks) // 2]
    late_tf = sum(flops[c["k"]] for c in late) / (sum(c["ms"] for c in late) / 1e3) / 1e12

    # Algorithmic DRAM bytes of one chunk-attention launch, averaged over the
    # step: Q and out once, lse, and every visible K/V row once.
    alg_bytes = statistics.mean(
        C * w.heads * (w.head_dim_qk + w.head_dim_v) * 2 + C * w.heads * 4
        + (P + C) * w.kv_heads * (w.head_dim_qk + w.head_dim_v) * 2 for P, C in chunks)
    traffic = args.traffic if args.traffic is not None else recorded_traffic(w.name)

    # KV append bandwidth on this workload's chunks (bytes read + written).
    app_bytes = [2 * C * w.kv_heads * (w.head_dim_qk + w.head_dim_v) * 2 for _, C in chunks]

    # End to end through the C ABI with host buffers: every step copies the
    # step's Q/K/V from pinned host memory, runs it and copies out + lse back.
    e2e = None
    if not args.no_e2e:
        hq = [q.to("cpu").pin_memory() for q in qs]
        hk = [k.to("cpu").pin_memory() for k in ks]
        hv = [v.to("cpu").pin_memory() for v in vs]
        ho = torch.empty((len(chunks), Cmax, w.heads, w.head_dim_v), dtype=torch.bfloat16).pin_memory()
        hl = torch.empty((len(chunks), w.heads, Cmax), dtype=torch.float32).pin_memory()
        # Double-buffered pipeline: chunk k+1's inputs are copied in (h2d
        # stream) and chunk k-1's results copied out (d2h stream) while chunk k
        # runs on the compute stream; events order the reuse of each buffer.
        dq2 = [torch.empty_like(qs[0]) for _ in range(2)]
        dk2 = [torch.empty_like(ks[0]) for _ in range(2)]
        dv2 = [torch.empty_like(vs[0]) for _ in range(2)]
        do2 = [torch.empty((Cmax, w.heads, w.head_dim_v), dtype=torch.bfloat16, device=dev) for _ in range(2)]
        dl2 = [torch.empty((w.heads, Cmax), dtype=torch.float32, device=dev) for _ in range(2)]
        h2d_s = torch.cuda.Stream(device=dev)
        d2h_s = torch.cuda.Stream(device=dev)
        h2d = sum(t.numel() * t.element_size() for t in hq + hk + hv)
        d2h = sum(C * w.heads * w.head_dim_v * 2 + w.heads * C * 4 for _, C in chunks)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_comp = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        state = {"first": True}

        def e2e_step():
            for ci, (P, C) in enumerate(chunks):
                b = ci & 1
                with torch.cuda.stream(h2d_s):
                    if not state["first"] or ci >= 2:
                        h2d_s.wait_event(ev_comp[b])     # the compute that read buffer b is done
                    dq2[b][:C].copy_(hq[ci], non_blocking=True)
                    dk2[b][:C].copy_(hk[ci], non_blocking=True)
                    dv2[b][:C].copy_(hv[ci], non_blocking=True)
                    ev_in[b].record(h2d_s)
                stream.wait_event(ev_in[b])
                if not state["first"] or ci >= 2:
                    stream.wait_event(ev_out[b])         # out/lse of buffer b were copied back
                vpp.vpp_kv_append(dk2[b][:C], dv2[b][:C], kc, vc, P, block_table=table)
                vpp.vpp_chunk_attn_ex(dq2[b][:C], kc, vc, P, block_table=table, out=do2[b][:C],
                                      lse=dl2[b] if C == Cmax else None, workspace=ws)
                ev_comp[b].record(stream)
                with torch.cuda.stream(d2h_s):
                    d2h_s.wait_event(ev_comp[b])
                    ho[ci, :C].copy_(do2[b][:C], non_blocking=True)
                    hl[ci].copy_(dl2[b], non_blocking=True)
                    ev_out[b].record(d2h_s)
            state["first"] = False

        e2e_step()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        dist_.barrier()
        torch.cuda.synchronize()
        t_host0 = time.perf_counter()
        e0.record(stream)
        h2d_s.wait_stream(stream)
        d2h_s.wait_stream(stream)
        for _ in range(args.steps):
            e2e_step()
        stream.wait_stream(d2h_s)
        stream.wait_stream(h2d_s)
        e1.record(stream)
        torch.cuda.synchronize()
        et = dist_.max(max(e0.elapsed_time(e1) / 1e3, time.perf_counter() - t_host0))
        e2e = {"value": sum(flops) * args.steps * dist_.world / et / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": 1e3 * et / args.steps}

    cpu = None
    if dist_.rank == 0 and dist_.world == 1 and not args.no_cpu_baseline:
        inp = oracle_inputs(w, 7, device_tensors=(qs, ks, vs))
        f, dt, rows, desc = oracle_sample(w, inp, args.cpu_rows, 7, budget_s=args.cpu_budget)
        rate = f / dt
        cpu = {"value": rate / 1e12, "unit": "TFLOP/s", "cores": host_cores(), "kind": "oracle",
               "sample": desc,
               # A sampled row costs in proportion to the keys it attends, so a
               # whole chunk's oracle time is its FLOPs at the sampled rate.
               "per_chunk_s_extrapolated": [round(fl / rate, 1) for fl in flops]}

    extras = {}
    if not args.no_extras:
        del qs, ks, vs
        torch.cuda.empty_cache()
        extras["gqa32k"] = measure_chunks(dev, stream, "gqa32k", None, peak_tf, peak_tf_burst, 10, warm=True)
        torch.cuda.empty_cache()
        extras["mla512k"] = measure_chunks(dev, stream, "mla512k", [0, 10, 20, 21], peak_tf, peak_tf_burst, 3)
        torch.cuda.empty_cache()
        extras["kv_append"] = measure_append(dev, stream, hbm)
        if not args.no_cpu_baseline:
            extras["cpu_full"] = measure_cpu_full(dev, stream, extras["gqa32k"]["rows"])
        extras["mixed"] = measure_mixed(dev, stream, hbm, peak_tf)
        torch.cuda.empty_cache()
        extras["cost_model"] = measure_cost_model(dev, stream)
        torch.cuda.empty_cache()
        extras["fp8_kv"] = measure_fp8(dev, stream, hbm, w, chunks)
        torch.cuda.empty_cache()
        extras["topk_sparse"] = measure_topk(dev, stream, hbm, peak_tf)

    if dist_.rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": dist_.world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * elapsed / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": workload_config(w),
            "clocks": clk, "e2e": e2e, "gpu_launches": launches_per_step * args.steps,
            "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak_tf,
                         "unit": "TFLOP/s", "frac": round(achieved / peak_tf, 4),
                         "traffic": traffic,
                         "algorithmic_bytes": round(alg_bytes),
                         "traffic_vs_algorithmic": round(traffic / alg_bytes, 3) if traffic else None,
                         "peak_source": f"bf16_tflops_sustained ({pk_src})",
                         "frac_of_burst": round(achieved / peak_tf_burst, 4)},
            "cpu_baseline": cpu,
            "per_chunk": per_chunk,
            "late_chunks_tflops": round(late_tf, 1),
            "late_chunks_frac_peak": round(late_tf / peak_tf, 4),
            "ex2_bound": ex2_bound(w, chunks, attn_ms_step, clk,
                                   torch.cuda.get_device_properties(dev).multi_processor_count),
            "latency_fit_vs_k": fit,
            "schedule": schedule_summary(per_chunk_ms) if len(per_chunk_ms) > 1 else None,
            "prefill_tokens_per_s": round(w.seq_len / (attn_ms_step / 1e3), 1),
            "kv_append_bytes_per_step": int(sum(app_bytes)),
            "hbm_peak_gbs": hbm,
        }
        line.update(extras)
        line["summary"] = summary(line, peak_tf_burst)
        print(json.dumps(line), flush=True)
    return 0


def summary(line, peak_burst):
    """The figures the targets are judged on, compact, as the last key of the
    line: per-chunk TFLOP/s and fractions of the sustained peak, the late
    chunks of the bench workload, the other configs' chunks, append and
    decode against HBM, the mixed step against its combined bound."""
    r4 = lambda x: None if x is None else round(float(x), 4)
    out = {"workload": line["config"]["workload"], "tflops": round(line["value"], 1),
           "frac": line["roofline"]["frac"], "frac_burst": line["roofline"]["frac_of_burst"],
           "late_frac": line.get("late_chunks_frac_peak"),
           "late_frac_burst": r4(line.get("late_chunks_tflops", 0) / peak_burst),
           "k_ms_tflops_frac": [[c["k"], c["ms"], c["tflops"], c["frac_peak"]] for c in line.get("per_chunk", [])]}
    for name in ("gqa32k", "mla512k"):
        if name in line:
            m = line[name]
            out[name] = {"tflops": m["tflops"], "frac": m["frac"],
                         "k_ms_tflops_frac": [[r[0], r[3], r[4], r[5]] for r in m["rows"]]}
    if "kv_append" in line:
        out["append_frac_hbm"] = line["kv_append"]["frac_hbm"]
    if "mixed" in line:
        mx = line["mixed"]
        out["decode_frac_hbm"] = mx["decode_frac_hbm"]
        out["mixed_ms"] = mx["step_ms"]
        out["mixed_bound_ms"] = mx["bound_ms"]
        out["mixed_frac_of_bound"] = mx["frac_of_bound"]
    if "fp8_kv" in line:
        f8 = line["fp8_kv"]
        out["fp8_decode_frac_hbm"] = f8["decode"]["frac_hbm_fp8"]
        pl = f8["prefill_last_chunk"]
        out["fp8_last_chunk_ms"] = [pl["ms_fp8"], pl.get("ms_fp8_widened"), pl["ms_bf16"]]
    if line.get("cpu_baseline"):
        out["cpu_tflops"] = r4(line["cpu_baseline"]["value"])
        out["cpu_cores"] = line["cpu_baseline"]["cores"]
    cf = line.get("cpu_full")
    if cf:
        # whole-chunk oracle seconds: tiny chunks 0..3, gqa32k chunks 0 and 1
        out["cpu_full_s"] = {"tiny": [r[4] for r in cf["tiny"]], "gqa32k": [r[4] for r in cf["gqa32k"]]}
    return out


def run_mixed(args, dist_):
    """The mixed micro-batch as the step: varlen append of the batch's new
    tokens, then vpp_mixed_attn (prefill chunks + split-KV decode rows)."""
    from chunked_prefill_causal_gb300 import vpp

    dist_.init()
    dev = torch.device("cuda", dist_.local)
    torch.cuda.set_device(dev)
    vpp.load()
    pk, pk_src = peaks()
    hbm = float(pk.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    stream = torch.cuda.current_stream()
    fp8 = args.kv_dtype == "fp8"
    ms = MixedSetup(dev, args.decode_rows, fp8=fp8)
    step = ms.step_fp8 if fp8 else ms.step
    decode_only = ms.decode_only_fp8 if fp8 else ms.decode_only
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    dist_.barrier()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    dist_.barrier()
    if vpp.vpp_last_device_status() != 0:
        raise RuntimeError("device status word reported an error")
    el = dist_.max(e0.elapsed_time(e1) / 1e3)
    dec_ms = time_events(decode_only, 5, stream)
    dec_bytes = ms.decode_bytes // 2 if fp8 else ms.decode_bytes  # one byte per cached element
    gbs = dec_bytes / (dec_ms / 1e3) / 1e9
    peak_tf = float(pk.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    bound = mixed_bound_ms(ms.prefill_flops, dec_bytes, peak_tf, hbm)
    step_ms = 1e3 * el / args.steps
    n_pre = len(ms.m.prefill_prefixes)
    if dist_.rank == 0:
        print(json.dumps({
            "metric": METRIC, "value": (ms.prefill_flops + ms.decode_flops) * args.steps * dist_.world / el / 1e12,
            "unit": "TFLOP/s", "n_gpus": dist_.world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * el / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "mixed", "decode_rows": len(ms.ctx_d), "heads": 32, "kv_heads": 8,
                       "head_dim": 128, "kv_cache": "E4M3 codes, per-kv-head scales" if fp8 else "bf16"},
            "gpu_launches": mixed_launches(n_pre, len(ms.ctx_d)) * args.steps,
            "bound_ms": round(bound, 3), "frac_of_bound": round(bound / step_ms, 4),
            "decode_only_ms": round(dec_ms, 3), "decode_gbs": round(gbs, 1),
            "decode_frac_hbm": round(gbs / hbm, 4), "hbm_peak_source": pk_src}), flush=True)
    return 0


def timeline_intervals(buf, tiles=range(8, 60)):
    """Median per-tile intervals (SM cycles) from one CTA's tracing-build
    stamps [role][tile][event].  Roles 0/1 are the issuers of query tiles A/B;
    their block j issues P V of tile j-1, then Q K^T of tile j (events: first
    part of P(j-1) seen, turn taken, block issued, second part of P(j-1)
    seen).  Roles 2/3 are the first softmax threads of A/B (events: S(j)
    ready, S in registers, first part of P stored and signalled, second
    part stored and signalled)."""
    med = lambda xs: int(np.median(list(xs)))
    out = {}
    for x in range(2):
        sm, iss = buf[2 + x], buf[x]
        t = "AB"[x]
        out[f"{t}.softmax: S ready -> S in registers"] = med(sm[j, 1] - sm[j, 0] for j in tiles)
        out[f"{t}.softmax: S in registers -> first part of P signalled"] = med(sm[j, 2] - sm[j, 1] for j in tiles)
        out[f"{t}.softmax: first -> second part of P signalled"] = med(sm[j, 3] - sm[j, 2] for j in tiles)
        out[f"{t}.issuer: first part of P signalled -> seen"] = med(iss[j + 1, 0] - sm[j, 2] for j in tiles)
        out[f"{t}.issuer: seen -> turn"] = med(iss[j + 1, 1] - iss[j + 1, 0] for j in tiles)
        out[f"{t}.issuer: turn -> second part of P seen"] = med(iss[j + 1, 3] - iss[j + 1, 1] for j in tiles)
        out[f"{t}.issuer: second part seen -> block issued"] = med(iss[j + 1, 2] - iss[j + 1, 3] for j in tiles)
        out[f"{t}.issuer: block issued -> S ready"] = med(sm[j + 1, 0] - iss[j + 1, 2] for j in tiles)
        out[f"{t}.period (S ready to S ready)"] = med(sm[j + 1, 0] - sm[j, 0] for j in tiles)
    return out


def run_timeline(args):
    """Builds a copy of the library with -DVPP_TIMELINE=<cta> beside the
    product one (the d 128 kernel then records clock64 stamps for CTA 0 and
    CTA <cta>), runs one chunk of a workload unsplit, and prints the kernel
    time and the median per-tile intervals as one JSON object."""
    import ctypes
    from chunked_prefill_causal_gb300 import build as B, vpp
    out_dir = os.path.join(ROOT, "chunked_prefill_causal_gb300", "_build_timeline")
    lib = vpp.load(B.build(extra_flags=(f"-DVPP_TIMELINE={args.timeline_cta}",), out_dir=out_dir,
                           lib_name="libvpp_timeline.so"))
    lib.vpp_timeline_read.argtypes = [ctypes.c_void_p]
    lib.vpp_timeline_clear.argtypes = []
    w = W.WORKLOADS[args.workload]
    if (w.head_dim_qk, w.head_dim_v) != (128, 128):
        raise SystemExit("--timeline: the stamps are compiled into the d 128 kernel only")
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    P, C = w.chunks()[args.timeline]
    nb = W.blocks_for(P + C)
    table = torch.from_numpy(W.block_table(nb, nb + 8, w.seed + 99)).to(dev)
    kc = torch.zeros((nb + 8, 64, w.kv_heads, w.head_dim_qk), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros((nb + 8, 64, w.kv_heads, w.head_dim_v), dtype=torch.bfloat16, device=dev)
    q = None
    for ci, (p0, _c0) in enumerate(w.chunks()[: args.timeline + 1]):
        qi, ki, vi = W.chunk_tensors(w, ci, dev)
        vpp.vpp_kv_append(ki, vi, kc, vc, p0, block_table=table)
        q = qi
        del ki, vi
    out = torch.empty((C, w.heads, w.head_dim_v), dtype=torch.bfloat16, device=dev)
    run = lambda: vpp.vpp_chunk_attn_ex(q, kc, vc, P, block_table=table, out=out, num_splits=1)
    for _ in range(args.warmup):
        run()
    torch.cuda.synchronize()
    if lib.vpp_timeline_clear() != 0:
        raise RuntimeError("timeline clear failed")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    run()
    e1.record()
    torch.cuda.synchronize()
    buf = np.zeros((2, 4, 64, 4), dtype=np.int64)
    if lib.vpp_timeline_read(buf.ctypes.data_as(ctypes.c_void_p)) != 0:
        raise RuntimeError("timeline read failed")
    res = {"workload": w.name, "chunk": args.timeline, "prefix": P, "chunk_len": C,
           "kernel_ms": round(e0.elapsed_time(e1), 3), "cta0": timeline_intervals(buf[0]),
           f"cta{args.timeline_cta}": timeline_intervals(buf[1])}
    print(json.dumps(res, indent=1))
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(W.WORKLOADS) + ["mixed", "topk"], default="long128k")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the KV-append and mixed-batch measurements")
    ap.add_argument("--decode-rows", type=int, default=None,
                    help="with --workload mixed: decode rows of the micro-batch (default 256)")
    ap.add_argument("--kv-dtype", choices=["bf16", "fp8"], default="bf16",
                    help="with --workload mixed or topk: the KV cache's element type")
    ap.add_argument("--topk-chunks", default=None,
                    help="with --workload topk: comma-separated dsa128k chunk indices (default all)")
    ap.add_argument("--cpu-rows", type=int, default=4096)
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--ref-rows", type=int, default=256)
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch of the chunk kernel from an ncu capture")
    ap.add_argument("--timeline", type=int, default=None, metavar="CHUNK",
                    help="trace one chunk of the workload with the clock64-stamp build of the d 128 kernel")
    ap.add_argument("--timeline-cta", type=int, default=500)
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)  # at least three untimed warm-up steps
    if args.timeline is not None:
        return run_timeline(args)
    dist_ = Dist()
    if args.impl == "reference":
        if args.workload in ("mixed", "topk"):
            args.workload = "long128k"
        return run_reference(args, dist_)
    if args.workload == "mixed":
        return run_mixed(args, dist_)
    if args.workload == "topk":
        return run_topk(args, dist_)
    return run_ours(args, dist_)


if __name__ == "__main__":
    sys.exit(main())
