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
# over the 8 launches of one long128k step, from one ncu capture
# (profiles/chunk_attn_long128k.md).  Valid only for the kernel sources whose
# digest is recorded with it; any change to them makes the figure stale (null).
TRAFFIC = {"long128k": {"sources_sha256": "7c36a21a363d67e387c1560676e33157d7e5f4a5895506d79c3fd4fb61441c62", "bytes_per_launch": 1.2117e9}}
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

    def init(self, backend="nccl"):
        if self.world > 1 and not self.pg:
            import torch.distributed as dist
            dist.init_process_group(backend)
            self.pg = True

    def barrier(self):
        if self.pg:
            import torch.distributed as dist
            dist.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch.distributed as dist
        t = torch.tensor([x], dtype=torch.float64, device="cuda")
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


# ------------------------------------------------------------------ our arm
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
        dq_ = torch.empty_like(qs[0])
        dk_ = torch.empty_like(ks[0])
        dv_ = torch.empty_like(vs[0])
        lse_e = torch.empty((w.heads, Cmax), dtype=torch.float32, device=dev)
        h2d = sum(t.numel() * t.element_size() for t in hq + hk + hv)
        d2h = sum(C * w.heads * w.head_dim_v * 2 + w.heads * C * 4 for _, C in chunks)

        def e2e_step():
            for ci, (P, C) in enumerate(chunks):
                dq_[:C].copy_(hq[ci], non_blocking=True)
                dk_[:C].copy_(hk[ci], non_blocking=True)
                dv_[:C].copy_(hv[ci], non_blocking=True)
                vpp.vpp_kv_append(dk_[:C], dv_[:C], kc, vc, P, block_table=table)
                o = vpp.vpp_chunk_attn_ex(dq_[:C], kc, vc, P, block_table=table, out=out[:C],
                                          lse=lse_e[:, :C] if C == Cmax else None, workspace=ws)
                ho[ci, :C].copy_(o, non_blocking=True)
                hl[ci].copy_(lse_e, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        dist_.barrier()
        e0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        et = dist_.max(e0.elapsed_time(e1) / 1e3)
        e2e = {"value": sum(flops) * args.steps * dist_.world / et / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": 1e3 * et / args.steps}

    cpu = None
    if dist_.rank == 0 and dist_.world == 1 and not args.no_cpu_baseline:
        inp = oracle_inputs(w, 7, device_tensors=(qs, ks, vs))
        f, dt, rows, desc = oracle_sample(w, inp, args.cpu_rows, 7, budget_s=args.cpu_budget)
        cpu = {"value": f / dt / 1e12, "unit": "TFLOP/s", "cores": host_cores(), "kind": "oracle",
               "sample": desc}

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
            "latency_fit_vs_k": fit,
            "prefill_tokens_per_s": round(w.seq_len / (attn_ms_step / 1e3), 1),
            "kv_append_bytes_per_step": int(sum(app_bytes)),
            "hbm_peak_gbs": hbm,
        }
        print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(W.WORKLOADS), default="long128k")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-rows", type=int, default=4096)
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--ref-rows", type=int, default=256)
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch of the chunk kernel from an ncu capture")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)  # at least three untimed warm-up steps
    dist_ = Dist()
    if args.impl == "reference":
        return run_reference(args, dist_)
    return run_ours(args, dist_)


if __name__ == "__main__":
    sys.exit(main())
