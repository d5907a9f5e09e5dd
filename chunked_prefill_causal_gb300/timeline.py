"""Device-side timeline of the chunk-attention kernel (tracing build).

Builds a separate copy of the library with -DVPP_TIMELINE=<cta>, which makes
the d 128 kernel record clock64 stamps for CTA 0 and CTA <cta>.  The stamps
come from the two MMA issuers (P of the previous tile seen, turn taken, P V
issued, block issued) and from the first softmax thread of each query tile (S
ready, S in registers, exponentials done, P signalled).  It runs one chunk of
a workload and prints median per-tile intervals in SM cycles over tiles 8..59.
The product library is not touched.

    python -m chunked_prefill_causal_gb300.timeline --workload long128k --chunk 7
"""

from __future__ import annotations

import argparse
import ctypes
import json
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
OUT_DIR = os.path.join(HERE, "_build_timeline")


def build(cta: int = 500) -> str:
    from chunked_prefill_causal_gb300 import build as b
    return b.build(extra_flags=(f"-DVPP_TIMELINE={cta}",), out_dir=OUT_DIR, lib_name="libvpp_timeline.so")


def intervals(buf: np.ndarray, tiles=range(8, 60)) -> dict:
    """Median intervals (cycles) from one CTA's stamps [role][tile][event]."""
    out = {}
    med = lambda xs: int(np.median(list(xs)))
    for x in range(2):
        sm, iss = buf[2 + x], buf[x]
        t = "AB"[x]
        out[f"{t}.softmax: S ready -> S in registers"] = med(sm[j, 1] - sm[j, 0] for j in tiles)
        out[f"{t}.softmax: exponentials"] = med(sm[j, 2] - sm[j, 1] for j in tiles)
        out[f"{t}.softmax: store P + signal"] = med(sm[j, 3] - sm[j, 2] for j in tiles)
        out[f"{t}.issuer: P signalled -> seen"] = med(iss[j + 1, 0] - sm[j, 3] for j in tiles)
        out[f"{t}.issuer: seen -> turn"] = med(iss[j + 1, 1] - iss[j + 1, 0] for j in tiles)
        out[f"{t}.issuer: turn -> P V issued (8 TS MMAs)"] = med(iss[j + 1, 3] - iss[j + 1, 1] for j in tiles)
        out[f"{t}.issuer: P V issued -> Q K^T issued (8 SS MMAs)"] = med(iss[j + 1, 2] - iss[j + 1, 3] for j in tiles)
        out[f"{t}.issuer: block issued -> S ready"] = med(sm[j + 1, 0] - iss[j + 1, 2] for j in tiles)
        out[f"{t}.period (S ready to S ready)"] = med(sm[j + 1, 0] - sm[j, 0] for j in tiles)
    return out


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="long128k")
    ap.add_argument("--chunk", type=int, default=7)
    ap.add_argument("--cta", type=int, default=500)
    args = ap.parse_args(argv)
    import torch
    from chunked_prefill_causal_gb300 import vpp, workloads as W
    lib = vpp.load(build(args.cta))
    lib.vpp_timeline_read.argtypes = [ctypes.c_void_p]
    lib.vpp_timeline_clear.argtypes = []
    w = W.WORKLOADS[args.workload]
    if (w.head_dim_qk, w.head_dim_v) != (128, 128):
        raise SystemExit("the timeline stamps are compiled into the d 128 kernel only")
    dev = torch.device("cuda")
    P, C = w.chunks()[args.chunk]
    nb = W.blocks_for(P + C)
    table = torch.from_numpy(W.block_table(nb, nb + 8, w.seed + 99)).to(dev)
    kc = torch.zeros((nb + 8, 64, w.kv_heads, w.head_dim_qk), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros((nb + 8, 64, w.kv_heads, w.head_dim_v), dtype=torch.bfloat16, device=dev)
    q = None
    for ci, (p0, c0) in enumerate(w.chunks()[: args.chunk + 1]):
        qi, ki, vi = W.chunk_tensors(w, ci, dev)
        vpp.vpp_kv_append(ki, vi, kc, vc, p0, block_table=table)
        q = qi
    out = torch.empty((C, w.heads, w.head_dim_v), dtype=torch.bfloat16, device=dev)
    run = lambda: vpp.vpp_chunk_attn_ex(q, kc, vc, P, block_table=table, out=out, num_splits=1)
    for _ in range(3):
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
    res = {"workload": w.name, "chunk": args.chunk, "prefix": P, "chunk_len": C,
           "kernel_ms": round(e0.elapsed_time(e1), 3), "cta0": intervals(buf[0]), f"cta{args.cta}": intervals(buf[1])}
    print(json.dumps(res, indent=1))


if __name__ == "__main__":
    main()
