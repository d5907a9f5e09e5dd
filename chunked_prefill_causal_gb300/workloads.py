"""Seeded synthetic workloads: shapes, value distributions and paged layouts.

This module holds no attention arithmetic.  It only draws inputs and lays out
block tables, and both the CUDA path (tests, bench) and the CPU oracle read the
same stored values from it.

The workloads mirror the pages' setups (cited by page title):

* ``tiny``     -- 2 q heads / 1 kv head, head_dim 64, 512 tokens in 4 chunks
  of 128, float32 N(0,1), contiguous cache.
* ``gqa32k``   -- GQA 32 q / 8 kv heads (the GQA model of the VPP technical
  review, §6 "Experimental Setup"), head_dim 128, 32768 tokens in 8 chunks of
  4096, N(0,1)/sqrt(128) rounded to bf16, paged cache (64-token blocks, the
  block size of the "02 · 并行策略与 PP 切分" note, §1).
* ``long128k`` -- GQA 64 / 8 heads, head_dim 128, 131072 tokens in 8 chunks of
  16384 (a 128K prompt in 8 fixed chunks, VPP review §3, Figure 1b).
* ``mla512k``  -- 128 heads, qk dim 192 (128 + 64 rope), v dim 128, 524288
  tokens in 24576-token chunks with a partial last chunk of 8192 (the
  DeepSeek-V3.1 512K runs with a 24K chunk budget, VPP review §3 and §4.6).
* ``mla24k``   -- the mla512k head shapes on a 24576-token sequence in three
  chunks of 8192: a case of a few GB that a profiler can capture whole.
* ``dsa128k``  -- GQA 32 / 8, head_dim 128, 131072 tokens in 8 chunks of
  16384, for top-k sparse prefix attention: every query token lists up to
  ``TOPK`` earlier keys (DSA-style, VPP technical review §7).
* ``mixed``    -- GQA 32 / 8, head_dim 128: four prefill chunks of 2048 tokens
  at prefixes {0, 16384, 65536, 122880} plus 256 decode rows whose context is
  uniform on [1024, 32768] ("Revisiting Pipeline Parallelism for LLM Serving",
  section "预备知识": mixed prefill + decode micro-batches).

Random values come from torch generators seeded per (workload, tensor, piece)
so that any chunk or sequence can be regenerated on its own, on CPU or GPU.
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

BLOCK = 64


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    heads: int
    kv_heads: int
    head_dim_qk: int
    head_dim_v: int
    seq_len: int
    chunk: int
    dtype: str            # "bf16" or "fp32" (the input tensors' type)
    paged: bool
    seed: int
    std: float            # value std before rounding

    @property
    def group(self) -> int:
        return self.heads // self.kv_heads

    def chunks(self):
        """(prefix_len, chunk_len) of each chunk in order; last may be partial."""
        out = []
        P = 0
        while P < self.seq_len:
            C = min(self.chunk, self.seq_len - P)
            out.append((P, C))
            P += C
        return out


WORKLOADS = {
    "tiny": Workload("tiny", 2, 1, 64, 64, 512, 128, "fp32", False, 1, 1.0),
    "gqa32k": Workload("gqa32k", 32, 8, 128, 128, 32768, 4096, "bf16", True, 2, 1 / math.sqrt(128)),
    "long128k": Workload("long128k", 64, 8, 128, 128, 131072, 16384, "bf16", True, 3, 1 / math.sqrt(128)),
    "mla512k": Workload("mla512k", 128, 128, 192, 128, 524288, 24576, "bf16", True, 4, 1 / math.sqrt(192)),
    "mla24k": Workload("mla24k", 128, 128, 192, 128, 24576, 8192, "bf16", True, 7, 1 / math.sqrt(192)),
    "dsa128k": Workload("dsa128k", 32, 8, 128, 128, 131072, 16384, "bf16", True, 8, 1 / math.sqrt(128)),
}

# Listed keys per query token of the top-k (DSA-style) workloads; the pages
# give no value, 2048 is the reading.
TOPK = 2048


def topk_indices(prefix_len: int, chunk_len: int, topk: int = TOPK, seed: int = 0, device="cpu"):
    """Synthetic top-k key lists of a chunk's query tokens (seeded).

    Token i sits at p = prefix_len + i.  If p + 1 <= topk it lists every key
    0 .. p; otherwise it lists one key drawn uniformly from each of topk - 1
    equal strata of 0 .. p - 1, then p itself (so the entries are distinct
    and spread over the whole prefix).  Returns int32 torch tensors on
    ``device``: idx [C, topk] with the valid entries first and -1 padding,
    and lens [C].  The draws come from a torch generator on ``device``, so a
    seed gives one list on CPU and another on a GPU.
    """
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1_000_003 + 17)
    C = int(chunk_len)
    pos = int(prefix_len) + torch.arange(C, dtype=torch.int64, device=device)
    lens = torch.clamp(pos + 1, max=topk)
    ar = torch.arange(topk, dtype=torch.int64, device=device)
    idx = torch.where(ar[None, :] <= pos[:, None], ar[None, :].expand(C, topk), torch.full_like(ar[None, :], -1))
    sparse = pos + 1 > topk
    if bool(sparse.any()):
        rows = torch.nonzero(sparse).squeeze(1)
        ps = pos[rows][:, None]
        m = topk - 1
        j = torch.arange(m, dtype=torch.int64, device=device)[None, :]
        lo = (j * ps) // m
        hi = ((j + 1) * ps) // m
        u = torch.rand((rows.numel(), m), generator=g, device=device, dtype=torch.float64)
        picks = lo + torch.floor(u * (hi - lo).to(torch.float64)).to(torch.int64)
        idx[rows] = torch.cat([picks, ps], dim=1)
    return idx.to(torch.int32), lens.to(torch.int32)


@dataclasses.dataclass(frozen=True)
class MixedWorkload:
    name: str = "mixed"
    heads: int = 32
    kv_heads: int = 8
    head_dim_qk: int = 128
    head_dim_v: int = 128
    prefill_chunk: int = 2048
    prefill_prefixes: tuple = (0, 16384, 65536, 122880)
    n_decode: int = 256
    decode_ctx_lo: int = 1024
    decode_ctx_hi: int = 32768
    seed: int = 5
    ctx_seed: int = 6
    std: float = 1 / math.sqrt(128)

    def batch(self):
        """Host arrays (cu_seqlens_q, ctx_lens) of the micro-batch."""
        rng = np.random.default_rng(self.ctx_seed)
        dec_ctx = rng.integers(self.decode_ctx_lo, self.decode_ctx_hi + 1, size=self.n_decode)
        qlen = [self.prefill_chunk] * len(self.prefill_prefixes) + [1] * self.n_decode
        ctx = [p + self.prefill_chunk for p in self.prefill_prefixes] + [int(c) for c in dec_ctx]
        cu = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
        return cu, np.asarray(ctx, dtype=np.int32)


MIXED = MixedWorkload()


def _torch_dtype(name):
    return torch.bfloat16 if name == "bf16" else torch.float32


def _gen(shape, seed, std, dtype, device, piece_rows=1 << 15):
    """N(0, std^2) values cast to ``dtype`` (bf16 rounding is RNE), drawn in
    row pieces from generators seeded (seed, piece) to bound temporaries."""
    out = torch.empty(shape, dtype=dtype, device=device)
    n = shape[0]
    for i, r0 in enumerate(range(0, n, piece_rows)):
        r1 = min(n, r0 + piece_rows)
        g = torch.Generator(device=device)
        g.manual_seed(seed * 1_000_003 + i)
        x = torch.randn((r1 - r0,) + tuple(shape[1:]), generator=g, device=device, dtype=torch.float32)
        out[r0:r1] = (x * std).to(dtype)
    return out


def chunk_tensors(w: Workload, chunk_index: int, device="cpu"):
    """Q [C, Hq, dq], K [C, Hkv, dq], V [C, Hkv, dv] of one chunk."""
    P, C = w.chunks()[chunk_index]
    dt = _torch_dtype(w.dtype)
    base = w.seed * 100_000 + chunk_index * 10
    q = _gen((C, w.heads, w.head_dim_qk), base + 0, w.std, dt, device)
    k = _gen((C, w.kv_heads, w.head_dim_qk), base + 1, w.std, dt, device)
    v = _gen((C, w.kv_heads, w.head_dim_v), base + 2, w.std, dt, device)
    return q, k, v


def sequence_kv(w: Workload, upto: int, device="cpu"):
    """K, V of token positions 0 .. upto-1 (concatenated chunk draws)."""
    ks, vs = [], []
    for ci, (P, C) in enumerate(w.chunks()):
        if P >= upto:
            break
        _, k, v = chunk_tensors(w, ci, device)
        n = min(C, upto - P)
        ks.append(k[:n])
        vs.append(v[:n])
    return torch.cat(ks), torch.cat(vs)


def block_table(n_blocks_needed: int, pool_blocks: int, seed: int):
    """A seeded random choice of distinct pool blocks, in random order."""
    rng = np.random.default_rng(seed)
    return rng.permutation(pool_blocks)[:n_blocks_needed].astype(np.int32)


def blocks_for(tokens: int) -> int:
    return (tokens + BLOCK - 1) // BLOCK


def mixed_tensors(m: MixedWorkload, device="cpu"):
    """Per-sequence K/V (token order, full context) and the packed new Q.

    Returns (q [total_q, Hq, dq] bf16, ks, vs) where ks[b], vs[b] hold the
    ctx_lens[b] tokens of sequence b, the last q_len_b of which are new.
    """
    cu, ctx = m.batch()
    ks, vs, qs = [], [], []
    for b in range(len(ctx)):
        base = m.seed * 1_000_000 + b * 10
        ks.append(_gen((int(ctx[b]), m.kv_heads, m.head_dim_qk), base + 1, m.std, torch.bfloat16, device))
        vs.append(_gen((int(ctx[b]), m.kv_heads, m.head_dim_v), base + 2, m.std, torch.bfloat16, device))
        qs.append(_gen((int(cu[b + 1] - cu[b]), m.heads, m.head_dim_qk), base + 0, m.std,
                       torch.bfloat16, device))
    return torch.cat(qs), ks, vs


def mixed_block_tables(m: MixedWorkload, slack_blocks: int = 7):
    """Disjoint random blocks of one pool for every sequence of the batch.

    Returns (table [B, max_blocks] int32 padded with -1, pool_blocks).
    """
    _, ctx = m.batch()
    need = [blocks_for(int(c)) for c in ctx]
    pool = sum(need) + slack_blocks
    perm = np.random.default_rng(m.seed + 77).permutation(pool).astype(np.int32)
    maxb = max(need)
    table = np.full((len(ctx), maxb), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[off:off + n]
        off += n
    return table, pool


def sample_rows(n_tokens_per_chunk, heads, n_rows: int, seed: int, tile_tokens: int = 16):
    """Seeded, stratified sample of (chunk, token, head) rows.

    ``heads`` is a head count or an explicit list of heads to draw from.
    Equal rows per chunk; each chunk always includes its first and last
    token and tokens on both sides of tile boundaries (multiples of
    ``tile_tokens``) so that diagonal-tile edges are exercised.
    """
    rng = np.random.default_rng(seed)
    head_pool = np.arange(heads) if np.isscalar(heads) else np.asarray(heads)
    n_chunks = len(n_tokens_per_chunk)
    per = max(1, n_rows // n_chunks)
    rows = []
    for ci, C in enumerate(n_tokens_per_chunk):
        fixed = {0, C - 1}
        n_b = max(1, C // tile_tokens)
        for b in rng.choice(n_b, size=min(8, n_b), replace=False):
            t = int(b) * tile_tokens
            fixed.update({max(0, t - 1), min(C - 1, t)})
        toks = sorted(fixed)
        toks += list(rng.integers(0, C, size=max(0, per - len(toks))))
        toks = np.array(toks[:per])
        hs = rng.choice(head_pool, size=len(toks))
        rows += [(ci, int(t), int(h)) for t, h in zip(toks, hs)]
    return rows


def head_subset(heads: int, n: int, seed: int):
    """A seeded subset of n query heads (sorted)."""
    rng = np.random.default_rng(seed)
    return np.sort(rng.choice(heads, size=min(n, heads), replace=False))
