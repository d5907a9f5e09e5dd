"""Top-k sparse prefix attention (DSA-style): fp64 CPU oracle.

TEST INFRASTRUCTURE ONLY.  Nothing in the product package imports, calls or
links this module; only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code, table or helper with the CUDA path.

Sources:

* [VPP review] "VPP: Virtual Pipeline Parallelism for Efficient Chunked
  Prefill in Long-Context LLM Inference", §7 (GLM's DSA sparse attention):
  sparse attention slows the growth of a chunk's attention cost with its
  prefix, so the linear per-chunk latency law of Eq. (2) stops holding.
* [GLM PP note] "02 · 并行策略与 PP 切分", §5.1: DSA selects a top-k set of
  earlier tokens for every query token (an indexer computes the indices,
  some layers reuse another layer's indices), and the main attention reads
  only those tokens.

Readings: query token i of a chunk, at absolute
position P + i, attends exactly the key positions listed in its index row,
idx[i, :len[i]], each in 0 .. P + i; the same row serves every head (one
index set per token, as with a single latent KV head); within the row the
keys enter Eq. (1) of the VPP review (§2.2) as in dense attention,
softmax(q k^T * scale) v over the listed keys.  A position listed twice
counts twice.  The indexer itself is not modelled: indices are inputs.

Everything is computed in float64 on the input values taken as exact.
"""

from __future__ import annotations

import numpy as np


def _scale(head_dim_qk: int, scale):
    return 1.0 / np.sqrt(float(head_dim_qk)) if scale is None else float(scale)


def topk_rows(q_rows, idx_rows, lens, k, v, kv_group: int, scale=None, positions=None):
    """Attention of single query tokens over their listed keys.

    q_rows: [R, Hq, dq]; idx_rows: [R, kmax] key positions; lens: [R] number
    of listed keys per row (1 .. kmax); k: [T, Hkv, dq], v: [T, Hkv, dv] in
    token order.  positions (optional, [R]): each row's absolute position,
    checked against the causal rule (every listed key <= position).
    Returns out [R, Hq, dv] and lse [Hq, R] (natural log of the softmax
    denominator).
    """
    q_rows = np.asarray(q_rows, dtype=np.float64)
    idx_rows = np.asarray(idx_rows, dtype=np.int64)
    lens = np.asarray(lens, dtype=np.int64)
    R, Hq, dq = q_rows.shape
    dv = v.shape[2]
    s = _scale(dq, scale)
    out = np.zeros((R, Hq, dv))
    lse = np.zeros((Hq, R))
    for r in range(R):
        n = int(lens[r])
        if not 1 <= n <= idx_rows.shape[1]:
            raise ValueError("every row lists 1 .. kmax keys")
        keys = idx_rows[r, :n]
        if keys.min() < 0 or (positions is not None and keys.max() > int(positions[r])):
            raise ValueError("listed keys must lie in 0 .. position")
        kk = np.asarray(k[keys], dtype=np.float64)      # [n, Hkv, dq]
        vv = np.asarray(v[keys], dtype=np.float64)
        for h in range(Hq):
            g = h // kv_group
            scores = s * (kk[:, g, :] @ q_rows[r, h])
            m = scores.max()
            e = np.exp(scores - m)
            den = e.sum()
            out[r, h] = (e @ vv[:, g, :]) / den
            lse[h, r] = m + np.log(den)
    return out, lse


def topk_chunk_attention(q, k, v, prefix_len: int, idx, lens, scale=None):
    """Every query token of a chunk (prefix P) over its listed keys.

    q: [C, Hq, dq]; idx: [C, kmax]; lens: [C]; k, v: the sequence's cache in
    token order (at least P + C tokens).  Returns out [C, Hq, dv], lse [Hq, C].
    """
    C, Hq, _ = q.shape
    Hkv = k.shape[1]
    pos = int(prefix_len) + np.arange(C)
    return topk_rows(q, idx, lens, k, v, Hq // Hkv, scale, positions=pos)


def topk_flops(lens, heads: int, head_dim_qk: int, head_dim_v: int) -> float:
    """2 (dq + dv) Hq sum_i len_i: one multiply-add per (query head, listed key, dim)."""
    return 2.0 * (head_dim_qk + head_dim_v) * heads * float(np.sum(np.asarray(lens, dtype=np.int64)))
