"""fp64 CPU oracle for one chunked-prefill causal-attention step.

TEST INFRASTRUCTURE ONLY.  Nothing in the product package imports, calls or
links this module; only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code, table or helper with the CUDA path.

Sources (cited by page title, section and equation):

* [VPP review] "VPP: Virtual Pipeline Parallelism for Efficient Chunked Prefill
  in Long-Context LLM Inference" (English technical review).
  - §2.2, Eq. (1): Attn(Q, K, V) = softmax(Q K^T / sqrt(d)) V, and the causal
    rule that token i attends only to tokens <= i.
  - §2.3: chunked prefill -- fixed-size chunks processed in order; a later
    chunk attends to the whole cached prefix (all earlier chunks' K/V) plus
    itself.
  - §2.1: prefill fills the KV cache, decode reads it, one token per step.
* [GLM PP note] "02 · 并行策略与 PP 切分" (deployment note).
  - §1: paged KV pool with block_size = 64 tokens per block.
  - §7: context-parallel decode needs the attention backend to return the
    log-sum-exp (LSE) so that partial results over disjoint key ranges can be
    merged.
* [FastPP summary] "Revisiting Pipeline Parallelism for LLM Serving".
  - section "预备知识：分块与三种气泡": a mixed micro-batch holds prefill
    chunks (many tokens per request) and decode requests (one token each).

Readings where the pages are silent:

* d in Eq. (1) is the per-head query/key dimension: scale = 1/sqrt(head_dim_qk).
* Query i of a chunk with prefix P sits at absolute position P + i and attends
  keys 0 .. P + i inclusive; the chunk's own K/V are in the cache first.
* GQA: query head h reads kv head h // (heads // kv_heads).
* LSE is the natural log of the softmax denominator, ln sum_j exp(s_j).

Everything is computed in float64 on the input values taken as exact.
Parity unpinned: none -- every function here is pinned by tests under
``tests/`` (brute force, a library routine, closed forms, invariants).
"""

from __future__ import annotations

import numpy as np

BLOCK_SIZE = 64  # [GLM PP note] §1: tokens per KV block


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def default_scale(head_dim_qk: int) -> float:
    """[VPP review] §2.2 Eq. (1): scores are divided by sqrt(d)."""
    return 1.0 / np.sqrt(float(head_dim_qk))


def causal_chunk_attention(q, k, v, prefix_len: int, scale: float | None = None,
                           row_block: int = 1024):
    """Attention of one prefill chunk over its cached prefix plus itself.

    q: [C, Hq, dq]; k: [P + C, Hkv, dq]; v: [P + C, Hkv, dv], key positions
    0 .. P + C - 1 (prefix first, then the chunk's own tokens).
    Returns out [C, Hq, dv] and lse [Hq, C], both float64.

    Eq. (1) of [VPP review] §2.2 with the causal rule "token i attends to
    tokens <= i", applied to query i of the chunk at absolute position
    prefix_len + i (§2.3).  Rows are processed in groups of ``row_block`` only
    to bound memory; every row is computed independently from the definition.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    C, Hq, dq = q.shape
    T, Hkv, dk = k.shape
    dv = v.shape[2]
    P = int(prefix_len)
    assert dk == dq and v.shape[:2] == (T, Hkv)
    assert T == P + C, "k/v must hold exactly the prefix plus the chunk"
    assert Hq % Hkv == 0
    G = Hq // Hkv
    s = default_scale(dq) if scale is None else float(scale)
    out = np.zeros((C, Hq, dv))
    lse = np.zeros((Hq, C))
    keys = np.arange(T)
    for r0 in range(0, C, row_block):
        r1 = min(C, r0 + row_block)
        pos = P + np.arange(r0, r1)                     # absolute query positions
        allowed = keys[None, :] <= pos[:, None]         # causal rule: j <= i
        n_keys = int(pos[-1]) + 1
        for h in range(Hq):
            g = h // G                                  # GQA: contiguous groups
            scores = s * (q[r0:r1, h, :] @ k[:n_keys, g, :].T)
            scores = np.where(allowed[:, :n_keys], scores, -np.inf)
            m = scores.max(axis=1, keepdims=True)       # finite: key 0 is always allowed
            e = np.exp(scores - m)
            den = e.sum(axis=1)
            out[r0:r1, h, :] = (e @ v[:n_keys, g, :]) / den[:, None]
            lse[h, r0:r1] = m[:, 0] + np.log(den)
    return out, lse


def causal_attention_probs(q, k, prefix_len: int, scale: float | None = None):
    """The softmax weights of Eq. (1) for every (query, head) row.

    Returns probs [C, Hq, P + C] (masked entries exactly 0) and the scores'
    natural-log normaliser lse [Hq, C].  Used to pin the softmax itself.
    """
    q, k = _f64(q), _f64(k)
    C, Hq, dq = q.shape
    T, Hkv, _ = k.shape
    P = int(prefix_len)
    G = Hq // Hkv
    s = default_scale(dq) if scale is None else float(scale)
    allowed = np.arange(T)[None, :] <= (P + np.arange(C))[:, None]
    probs = np.zeros((C, Hq, T))
    lse = np.zeros((Hq, C))
    for h in range(Hq):
        scores = np.where(allowed, s * (q[:, h, :] @ k[:, h // G, :].T), -np.inf)
        m = scores.max(axis=1, keepdims=True)
        e = np.exp(scores - m)
        den = e.sum(axis=1, keepdims=True)
        probs[:, h, :] = e / den
        lse[h] = m[:, 0] + np.log(den[:, 0])
    return probs, lse


def attention_rows(q_rows, heads_of_rows, positions, k, v, kv_group: int,
                   scale: float | None = None):
    """Single output rows of Eq. (1), for sampled checks at full size.

    q_rows: [R, dq] query vectors; heads_of_rows: [R] query-head index;
    positions: [R] absolute positions p (row attends keys 0..p);
    k: [T, Hkv, dq], v: [T, Hkv, dv] with T > max(p).
    Returns out [R, dv], lse [R].  Rows sharing a head are evaluated together
    (one matrix product per head), each against its own key range.
    """
    q_rows = _f64(q_rows)
    heads_of_rows = np.asarray(heads_of_rows)
    positions = np.asarray(positions, dtype=np.int64)
    R, dq = q_rows.shape
    dv = v.shape[2]
    s = default_scale(dq) if scale is None else float(scale)
    out = np.zeros((R, dv))
    lse = np.zeros(R)
    for h in np.unique(heads_of_rows):
        idx = np.nonzero(heads_of_rows == h)[0]
        g = int(h) // kv_group
        n_keys = int(positions[idx].max()) + 1
        kg = _f64(k[:n_keys, g, :])
        vg = _f64(v[:n_keys, g, :])
        scores = s * (q_rows[idx] @ kg.T)
        allowed = np.arange(n_keys)[None, :] <= positions[idx][:, None]
        scores = np.where(allowed, scores, -np.inf)
        m = scores.max(axis=1, keepdims=True)
        e = np.exp(scores - m)
        den = e.sum(axis=1)
        out[idx] = (e @ vg) / den[:, None]
        lse[idx] = m[:, 0] + np.log(den)
    return out, lse


def split_key_range_attention(q, k, v, prefix_len: int, bounds, scale=None):
    """Eq. (1) restricted to disjoint key ranges, one partial result each.

    bounds: increasing key boundaries b_0 = 0 < b_1 < ... < b_S = P + C.
    Range s covers keys [b_s, b_{s+1}) intersected with the causal window.
    Returns a list of (out_s [C,Hq,dv], lse_s [Hq,C]); a row with no visible
    key in a range gets out 0 and lse -inf.  This is the partial-result form
    that [GLM PP note] §7 says context-parallel attention must return.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    C, Hq, dq = q.shape
    T, Hkv, _ = k.shape
    dv = v.shape[2]
    P = int(prefix_len)
    G = Hq // Hkv
    s = default_scale(dq) if scale is None else float(scale)
    pos = P + np.arange(C)
    parts = []
    for b0, b1 in zip(bounds[:-1], bounds[1:]):
        keys = np.arange(b0, b1)
        allowed = keys[None, :] <= pos[:, None]
        out = np.zeros((C, Hq, dv))
        lse = np.full((Hq, C), -np.inf)
        for h in range(Hq):
            g = h // G
            scores = np.where(allowed, s * (q[:, h, :] @ k[b0:b1, g, :].T), -np.inf)
            vis = allowed.any(axis=1)
            m = np.where(vis, scores.max(axis=1), 0.0)
            e = np.exp(scores - m[:, None])
            den = e.sum(axis=1)
            o = np.zeros((C, dv))
            o[vis] = (e[vis] @ v[b0:b1, g, :]) / den[vis, None]
            out[:, h, :] = o
            lse[h, vis] = m[vis] + np.log(den[vis])
        parts.append((out, lse))
    return parts


def merge_partials(parts):
    """Combine partial results over disjoint key ranges into the full result.

    With L = ln sum_s exp(lse_s), out = sum_s exp(lse_s - L) * out_s.  This
    follows from Eq. (1): each partial is a softmax over its own keys, and the
    weight of range s in the full softmax is exp(lse_s) / exp(L).
    """
    lses = np.stack([p[1] for p in parts])          # [S, Hq, C]
    outs = np.stack([p[0] for p in parts])          # [S, C, Hq, dv]
    m = lses.max(axis=0)
    w = np.exp(lses - m[None])                      # exp(-inf) = 0 for empty ranges
    tot = w.sum(axis=0)
    lse = m + np.log(tot)
    wn = w / tot[None]                              # [S, Hq, C]
    out = np.einsum("shc,schd->chd", wn, outs)
    return out, lse


# ---------------------------------------------------------------- paged cache

def gather_paged(cache, block_table, n_tokens: int):
    """Token-ordered view of a paged cache.

    cache: [num_blocks, 64, Hkv, d]; token j of the sequence lives in block
    block_table[j // 64], row j % 64 ([GLM PP note] §1, block_size 64).
    Returns [n_tokens, Hkv, d] (same dtype as cache).
    """
    cache = np.asarray(cache)
    bt = np.asarray(block_table, dtype=np.int64)
    j = np.arange(int(n_tokens))
    return cache[bt[j // BLOCK_SIZE], j % BLOCK_SIZE]


def kv_append(cache, block_table, new, prefix_len: int):
    """Copy a chunk's new K (or V) rows into their cache slots (in place).

    new: [C, Hkv, d]; token i goes to position prefix_len + i of the sequence,
    i.e. block block_table[(P+i)//64], row (P+i)%64.  A bit copy: prefill
    fills the cache that later chunks and decode read ([VPP review] §2.1).
    """
    bt = np.asarray(block_table, dtype=np.int64)
    pos = int(prefix_len) + np.arange(new.shape[0])
    cache[bt[pos // BLOCK_SIZE], pos % BLOCK_SIZE] = new
    return cache


def mixed_batch_attention(q, k_seqs, v_seqs, cu_seqlens_q, ctx_lens, scale=None):
    """A mixed micro-batch: prefill chunks and single-token decode rows.

    q: [total_q, Hq, dq] with sequence b owning rows cu[b]:cu[b+1];
    k_seqs[b], v_seqs[b]: that sequence's cached keys/values in token order,
    at least ctx_lens[b] tokens.  Sequence b's queries are its last
    q_len_b = cu[b+1]-cu[b] positions, so its prefix is ctx_b - q_len_b
    ([FastPP summary] "预备知识"; a decode row is the q_len = 1 case).
    Returns out [total_q, Hq, dv], lse [Hq, total_q].
    """
    cu = np.asarray(cu_seqlens_q, dtype=np.int64)
    B = len(cu) - 1
    Hq = q.shape[1]
    dv = v_seqs[0].shape[2]
    out = np.zeros((q.shape[0], Hq, dv))
    lse = np.zeros((Hq, q.shape[0]))
    for b in range(B):
        a, e = int(cu[b]), int(cu[b + 1])
        if e == a:
            continue
        ctx = int(ctx_lens[b])
        P = ctx - (e - a)
        assert P >= 0
        o, l = causal_chunk_attention(q[a:e], k_seqs[b][:ctx], v_seqs[b][:ctx], P, scale)
        out[a:e] = o
        lse[:, a:e] = l
    return out, lse


def chunk_flops(prefix_len: int, chunk_len: int, heads: int, head_dim_qk: int,
                head_dim_v: int) -> float:
    """Algorithmic FLOPs of one chunk: 2 (dq + dv) Hq (C P + C (C + 1) / 2).

    One multiply-add per (query, visible key, dim) for Q K^T and for P V;
    masked pairs are not counted.
    """
    C, P = int(chunk_len), int(prefix_len)
    pairs = C * P + C * (C + 1) // 2
    return 2.0 * (head_dim_qk + head_dim_v) * heads * pairs
