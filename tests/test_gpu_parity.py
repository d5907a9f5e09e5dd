"""GPU parity: the sm_103a kernels (through the C ABI) against the fp64 oracle.

Small cases span several 128-key tiles and ragged query/key tails; the
oracle computes every output row.  Tolerances: max-abs 2e-2 and relative L2
5e-3 on the bf16 output (bf16 inputs, fp32 accumulation), 1e-2 on the LSE.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from chunked_prefill_causal_gb300 import vpp
from tests.helpers import LSE_ABS, assert_close, errors, random_table, to_np64

pytestmark = pytest.mark.gpu

DEV = "cuda"


def gen(shape, seed, std, dtype=torch.bfloat16):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to(dtype)


def make_seq(L, Hq, Hkv, dq, dv, seed, std=None):
    std = std if std is not None else 1 / math.sqrt(dq)
    q = gen((L, Hq, dq), seed, std)
    k = gen((L, Hkv, dq), seed + 1, std)
    v = gen((L, Hkv, dv), seed + 2, std)
    return q, k, v


class Cache:
    """A paged (NaN-filled pool, random block order) or contiguous cache
    holding a sequence's K/V, written through vpp_kv_append."""

    def __init__(self, k, v, paged, seed=0, append_chunk=None, cap_extra=0):
        L, Hkv, dq = k.shape
        dv = v.shape[2]
        nan = float("nan")
        if paged:
            need = (L + 63) // 64
            pool = need + 5
            self.table = torch.from_numpy(random_table(need, pool, seed)).to(DEV)
            self.k = torch.full((pool, 64, Hkv, dq), nan, dtype=torch.bfloat16, device=DEV)
            self.v = torch.full((pool, 64, Hkv, dv), nan, dtype=torch.bfloat16, device=DEV)
        else:
            self.table = None
            self.k = torch.full((L + cap_extra, Hkv, dq), nan, dtype=torch.bfloat16, device=DEV)
            self.v = torch.full((L + cap_extra, Hkv, dv), nan, dtype=torch.bfloat16, device=DEV)
        step = append_chunk or L
        for P in range(0, L, step):
            C = min(step, L - P)
            vpp.vpp_kv_append(k[P:P + C].to(DEV), v[P:P + C].to(DEV), self.k, self.v, P,
                              block_table=self.table)


def run_and_check(q, k, v, P, C, paged, num_splits=0, seed=0, scale=0.0):
    cache = Cache(k[:P + C], v[:P + C], paged, seed)
    Hq = q.shape[1]
    lse = torch.empty((Hq, C), dtype=torch.float32, device=DEV)
    out = vpp.vpp_chunk_attn_ex(q[P:P + C].to(DEV), cache.k, cache.v, P, block_table=cache.table,
                                lse=lse, num_splits=num_splits, softmax_scale=scale)
    torch.cuda.synchronize()
    assert vpp.vpp_last_device_status() == 0
    ref, ref_lse = oracle.causal_chunk_attention(to_np64(q[P:P + C]), to_np64(k[:P + C]),
                                                 to_np64(v[:P + C]), P,
                                                 scale=(scale if scale > 0 else None))
    assert_close(to_np64(out), ref)
    assert np.abs(to_np64(lse) - ref_lse).max() <= LSE_ABS
    return out, lse


SMALL = [  # Hq, Hkv, dq, dv, P, C, paged
    (2, 1, 64, 64, 0, 128, False),
    (2, 1, 64, 64, 384, 128, False),
    (8, 2, 128, 128, 0, 1, True),
    (8, 2, 128, 128, 0, 333, True),
    (8, 2, 128, 128, 77, 200, True),
    (8, 2, 128, 128, 640, 37, True),
    (8, 2, 128, 128, 1000, 129, False),
    (32, 8, 128, 128, 500, 100, True),
    (16, 2, 128, 128, 130, 70, True),     # G = 8
    (32, 2, 128, 128, 63, 17, True),      # G = 16
    (4, 4, 192, 128, 0, 300, True),       # MLA-shaped, G = 1
    (4, 4, 192, 128, 700, 129, True),
    (4, 2, 64, 128, 250, 90, True),
    (4, 2, 128, 64, 250, 90, True),
    (4, 2, 192, 64, 250, 90, False),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "H%d-%d_d%d-%d_P%d_C%d_%s" % (
    c[0], c[1], c[2], c[3], c[4], c[5], "paged" if c[6] else "contig"))
def test_chunk_attention_small(case):
    Hq, Hkv, dq, dv, P, C, paged = case
    q, k, v = make_seq(P + C, Hq, Hkv, dq, dv, seed=hash(case) % 10000)
    run_and_check(q, k, v, P, C, paged, seed=P + C)


def test_plain_entry_point_contiguous_cache():
    """vpp_chunk_attn: contiguous cache, d_qk = d_v, bf16, default scale."""
    Hq, Hkv, d, P, C = 8, 2, 128, 300, 260
    q, k, v = make_seq(P + C, Hq, Hkv, d, d, seed=41)
    kc = k.to(DEV).contiguous()
    vc = v.to(DEV).contiguous()
    lse = torch.empty((Hq, C), dtype=torch.float32, device=DEV)
    out = vpp.vpp_chunk_attn(q[P:].to(DEV), kc, vc, P, lse=lse)
    torch.cuda.synchronize()
    ref, ref_lse = oracle.causal_chunk_attention(to_np64(q[P:]), to_np64(k), to_np64(v), P)
    assert_close(to_np64(out), ref)
    assert np.abs(to_np64(lse) - ref_lse).max() <= LSE_ABS


def test_tiny_workload_fp32_all_chunks():
    """tiny: 2/1 heads, d 64, 512 tokens in 4 chunks of 128, float32 inputs
    (rounded to bf16 at the boundary), contiguous cache."""
    from chunked_prefill_causal_gb300 import workloads as W
    w = W.WORKLOADS["tiny"]
    L = w.seq_len
    kc = torch.full((L, 1, 64), float("nan"), dtype=torch.bfloat16, device=DEV)
    vc = torch.full_like(kc, float("nan"))
    ks, vs = [], []
    for ci, (P, C) in enumerate(w.chunks()):
        q, k, v = W.chunk_tensors(w, ci, DEV)
        assert q.dtype == torch.float32
        vpp.vpp_kv_append(k, v, kc, vc, P)
        ks.append(k)
        vs.append(v)
        lse = torch.empty((2, C), dtype=torch.float32, device=DEV)
        out = vpp.vpp_chunk_attn_ex(q, kc, vc, P, lse=lse)
        torch.cuda.synchronize()
        ref, ref_lse = oracle.causal_chunk_attention(to_np64(q), to_np64(torch.cat(ks)),
                                                     to_np64(torch.cat(vs)), P)
        assert_close(to_np64(out), ref, what=f"tiny chunk {ci}")
        assert np.abs(to_np64(lse) - ref_lse).max() <= LSE_ABS
    assert vpp.vpp_last_device_status() == 0


@pytest.mark.parametrize("splits", [2, 3, 5])
def test_split_prefix_matches_and_is_deterministic(splits):
    Hq, Hkv, d, P, C = 16, 4, 128, 3000, 100
    q, k, v = make_seq(P + C, Hq, Hkv, d, d, seed=51)
    assert vpp.chunk_attn_num_splits(P, C, Hq, Hkv, d, d, splits) == splits
    out, lse = run_and_check(q, k, v, P, C, True, num_splits=splits, seed=3)
    out2, lse2 = run_and_check(q, k, v, P, C, True, num_splits=splits, seed=3)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    base, _ = run_and_check(q, k, v, P, C, True, num_splits=1, seed=3)
    ma, rl = errors(to_np64(out), to_np64(base))
    assert ma <= 2e-2 and rl <= 5e-3


# Shapes where the library's own plan splits the keys of its heaviest query
# tiles only: tokens from the split token on take S ranges, earlier tokens
# none.  Hq, Hkv, d, P, C, expected (S, split token) on a 152-SM GB300.
HEAVY_SPLIT = [
    (32, 8, 128, 4096, 1536, (3, 1152)),
    (16, 16, 64, 6000, 3072, (3, 2304)),   # G = 1
]


@pytest.mark.parametrize("case", HEAVY_SPLIT, ids=lambda c: "H%d-%d_d%d_P%d_C%d" % c[:5])
def test_auto_plan_splitting_heavy_query_tiles(case):
    """The heavy query tiles' key ranges are merged by the merge kernel; the
    light tiles are written directly by the attention kernel.  Both match the
    oracle row by row, repeat bit for bit, and the light rows equal the
    unsplit kernel's bit for bit."""
    Hq, Hkv, d, P, C, expect = case
    assert vpp.chunk_attn_plan(P, C, Hq, Hkv, d, d) == expect
    S, t0 = expect
    assert t0 % (2 * 128 // (Hq // Hkv)) == 0
    rows = S * (C - t0)
    assert vpp.chunk_attn_workspace_size(vpp.VPP_BF16, P, C, Hq, Hkv, d, d) >= rows * Hq * (d + 1) * 4
    q, k, v = make_seq(P + C, Hq, Hkv, d, d, seed=P + C + Hkv)
    cache = Cache(k, v, True, seed=5)
    qd = q[P:].to(DEV)

    def run(num_splits):
        lse = torch.empty((Hq, C), dtype=torch.float32, device=DEV)
        out = vpp.vpp_chunk_attn_ex(qd, cache.k, cache.v, P, block_table=cache.table, lse=lse,
                                    num_splits=num_splits)
        torch.cuda.synchronize()
        assert vpp.vpp_last_device_status() == 0
        return out, lse

    out, lse = run(0)
    out2, lse2 = run(0)
    base, base_lse = run(1)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    # the light tokens run the unsplit kernel's arithmetic
    assert torch.equal(out[:t0], base[:t0]) and torch.equal(lse[:, :t0], base_lse[:, :t0])
    ref, ref_lse = oracle.causal_chunk_attention(to_np64(q[P:]), to_np64(k), to_np64(v), P)
    assert_close(to_np64(out), ref)
    assert np.abs(to_np64(lse) - ref_lse).max() <= LSE_ABS


def test_zero_query_gives_running_mean_mask_probe():
    """Q = 0 and V[j, c] = bit c of j: the exact output is the running mean,
    so an off-by-one causal mask shows at O(1/p) at every tile boundary."""
    Hq, Hkv, dq, dv, P, C = 8, 2, 128, 64, 250, 300
    L = P + C
    q = torch.zeros((L, Hq, dq), dtype=torch.bfloat16)
    k = gen((L, Hkv, dq), 61, 1.0)
    j = torch.arange(L)
    bits = ((j[:, None] >> torch.arange(dv)[None, :] % 10) & 1).to(torch.bfloat16)
    v = bits[:, None, :].expand(L, Hkv, dv).contiguous()
    out, lse = run_and_check(q, k, v, P, C, True, seed=7)
    pos = P + np.arange(C)
    np.testing.assert_allclose(to_np64(lse)[0], np.log(pos + 1), atol=1e-4)


@pytest.mark.parametrize("offset", [0, 1])
def test_needle_respects_causality(offset):
    Hq, Hkv, d, P, C = 4, 1, 128, 190, 140
    L = P + C
    q, k, v = make_seq(L, Hq, Hkv, d, d, seed=71)
    k = torch.zeros_like(k)
    i_star = 66                     # second 64-token group: a diagonal tile
    j_star = P + i_star + offset
    qv = q[P + i_star, 0].float()
    k[j_star, 0] = (12.0 * math.sqrt(d) * qv / qv.norm() ** 2).to(torch.bfloat16)
    out, _ = run_and_check(q, k, v, P, C, True, seed=9)
    got = to_np64(out)[i_star, 0]
    if offset == 0:
        assert np.abs(got - to_np64(v)[j_star, 0]).max() < 2e-2
    else:
        assert np.abs(got - to_np64(v)[:P + i_star + 1, 0].mean(axis=0)).max() < 2e-2


def test_chunks_in_order_equal_one_full_call():
    Hq, Hkv, d, L, step = 8, 2, 128, 1000, 256
    q, k, v = make_seq(L, Hq, Hkv, d, d, seed=81)
    cache = Cache(k, v, True, seed=11, append_chunk=step)
    full = vpp.vpp_chunk_attn_ex(q.to(DEV), cache.k, cache.v, 0, block_table=cache.table)
    parts = []
    for P in range(0, L, step):
        C = min(step, L - P)
        parts.append(vpp.vpp_chunk_attn_ex(q[P:P + C].to(DEV), cache.k, cache.v, P,
                                           block_table=cache.table))
    torch.cuda.synchronize()
    chunked = torch.cat(parts)
    ma, rl = errors(to_np64(chunked), to_np64(full))
    assert ma <= 2e-2 and rl <= 5e-3
    ref, _ = oracle.causal_chunk_attention(to_np64(q), to_np64(k), to_np64(v), 0)
    assert_close(to_np64(chunked), ref)


def test_paged_equals_contiguous():
    Hq, Hkv, d, P, C = 8, 2, 128, 450, 180
    q, k, v = make_seq(P + C, Hq, Hkv, d, d, seed=91)
    a, la = run_and_check(q, k, v, P, C, True, num_splits=1, seed=1)
    b, lb = run_and_check(q, k, v, P, C, False, num_splits=1)
    assert torch.equal(a, b) and torch.equal(la, lb)


def test_softmax_scale_override():
    Hq, Hkv, d, P, C = 4, 2, 128, 100, 50
    q, k, v = make_seq(P + C, Hq, Hkv, d, d, seed=93)
    run_and_check(q, k, v, P, C, True, scale=0.3)


def test_kv_append_is_a_bit_copy():
    Hkv, dq, dv, nb = 4, 192, 128, 40
    L = 1000
    k = gen((L, Hkv, dq), 5, 1.0)
    v = gen((L, Hkv, dv), 6, 1.0)
    table = random_table((L + 63) // 64, nb, 2)
    kc = torch.zeros((nb, 64, Hkv, dq), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros((nb, 64, Hkv, dv), dtype=torch.bfloat16, device=DEV)
    t = torch.from_numpy(table).to(DEV)
    for P, C in ((0, 300), (300, 1), (301, 699)):
        vpp.vpp_kv_append(k[P:P + C].to(DEV), v[P:P + C].to(DEV), kc, vc, P, block_table=t)
    torch.cuda.synchronize()
    ref_k = np.zeros((nb, 64, Hkv, dq), dtype=np.uint16)
    ref_v = np.zeros((nb, 64, Hkv, dv), dtype=np.uint16)
    oracle.kv_append(ref_k, table, k.view(torch.int16).numpy().view(np.uint16), 0)
    oracle.kv_append(ref_v, table, v.view(torch.int16).numpy().view(np.uint16), 0)
    assert np.array_equal(kc.cpu().view(torch.int16).numpy().view(np.uint16), ref_k)
    assert np.array_equal(vc.cpu().view(torch.int16).numpy().view(np.uint16), ref_v)


def test_kv_append_fp32_rounds_to_nearest_even():
    Hkv, d, L = 1, 64, 256
    g = torch.Generator().manual_seed(3)
    k = torch.randn((L, Hkv, d), generator=g)
    v = torch.randn((L, Hkv, d), generator=g)
    kc = torch.zeros((L, Hkv, d), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    vpp.vpp_kv_append(k.to(DEV), v.to(DEV), kc, vc, 0)
    torch.cuda.synchronize()
    assert torch.equal(kc.cpu(), k.to(torch.bfloat16)) and torch.equal(vc.cpu(), v.to(torch.bfloat16))


def test_kv_append_varlen_places_rows():
    Hkv, d, nb = 2, 128, 64
    ctx = np.array([70, 5, 130, 1], dtype=np.int32)
    qlen = np.array([3, 1, 66, 1], dtype=np.int32)
    cu = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
    maxb = 3
    perm = np.random.default_rng(4).permutation(nb).astype(np.int32)
    table = np.full((4, maxb), -1, dtype=np.int32)
    off = 0
    for b in range(4):
        n = (ctx[b] + 63) // 64
        table[b, :n] = perm[off:off + n]
        off += n
    kn = gen((cu[-1], Hkv, d), 8, 1.0)
    vn = gen((cu[-1], Hkv, d), 9, 1.0)
    kc = torch.zeros((nb, 64, Hkv, d), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    vpp.vpp_kv_append_varlen(kn.to(DEV), vn.to(DEV), kc, vc, torch.from_numpy(table).to(DEV), cu, ctx)
    torch.cuda.synchronize()
    ref = np.zeros((nb, 64, Hkv, d), dtype=np.uint16)
    raw = kn.view(torch.int16).numpy().view(np.uint16)
    for b in range(4):
        oracle.kv_append(ref, table[b], raw[cu[b]:cu[b + 1]], ctx[b] - qlen[b])
    assert np.array_equal(kc.cpu().view(torch.int16).numpy().view(np.uint16), ref)


def test_mixed_batch_small():
    Hq, Hkv, d, nb = 8, 2, 128, 200
    ctx = np.array([300, 700, 64, 129, 1, 2000, 513], dtype=np.int32)
    qlen = np.array([300, 128, 1, 1, 1, 1, 77], dtype=np.int32)
    B = len(ctx)
    cu = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
    maxb = int(max((c + 63) // 64 for c in ctx))
    perm = np.random.default_rng(12).permutation(nb).astype(np.int32)
    table = np.full((B, maxb), -1, dtype=np.int32)
    ks, vs = [], []
    kc = torch.full((nb, 64, Hkv, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    vc = torch.full_like(kc, float("nan"))
    off = 0
    for b in range(B):
        n = (ctx[b] + 63) // 64
        table[b, :n] = perm[off:off + n]
        off += n
        k = gen((int(ctx[b]), Hkv, d), 100 + b, 1 / math.sqrt(d))
        v = gen((int(ctx[b]), Hkv, d), 200 + b, 1 / math.sqrt(d))
        ks.append(k)
        vs.append(v)
        vpp.vpp_kv_append(k.to(DEV), v.to(DEV), kc, vc, 0, block_table=torch.from_numpy(table[b].copy()).to(DEV))
    q = gen((int(cu[-1]), Hq, d), 300, 1 / math.sqrt(d))
    lse = torch.empty((Hq, int(cu[-1])), dtype=torch.float32, device=DEV)
    out = vpp.vpp_mixed_attn(q.to(DEV), kc, vc, torch.from_numpy(table).to(DEV), cu, ctx, lse=lse)
    torch.cuda.synchronize()
    assert vpp.vpp_last_device_status() == 0
    ref, ref_lse = oracle.mixed_batch_attention(to_np64(q), [to_np64(x) for x in ks],
                                                [to_np64(x) for x in vs], cu, ctx)
    assert_close(to_np64(out), ref)
    assert np.abs(to_np64(lse) - ref_lse).max() <= LSE_ABS


def test_mixed_batch_at_the_sequence_limit():
    # 1024 sequences (the plan's limit): 80 prefill segments, more than one
    # chunk-kernel launch holds (64), and 944 decode rows of the split-KV kernel.
    Hq, Hkv, d = 8, 2, 64
    rng = np.random.default_rng(31)
    B, n_pre = 1024, 80
    qlen = np.ones(B, dtype=np.int32)
    qlen[:n_pre] = rng.integers(2, 41, n_pre)
    ctx = (qlen + rng.integers(0, 160, B)).astype(np.int32)
    order = rng.permutation(B)  # prefill segments and decode rows interleaved
    qlen, ctx = qlen[order], ctx[order]
    cu = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
    need = [(int(c) + 63) // 64 for c in ctx]
    maxb, nb = max(need), sum(need) + 4
    perm = rng.permutation(nb).astype(np.int32)
    table = np.full((B, maxb), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        table[b, :need[b]] = perm[off:off + need[b]]
        off += need[b]
    std = 1 / math.sqrt(d)
    k_all = gen((int(ctx.sum()), Hkv, d), 700, std)
    v_all = gen((int(ctx.sum()), Hkv, d), 701, std)
    starts = np.concatenate([[0], np.cumsum(ctx)])
    # the whole cache through one varlen append (every token of every sequence is new)
    kc = torch.full((nb, 64, Hkv, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    vc = torch.full_like(kc, float("nan"))
    tab = torch.from_numpy(table).to(DEV)
    cu_all = starts.astype(np.int32)
    vpp.vpp_kv_append_varlen(k_all.to(DEV), v_all.to(DEV), kc, vc, tab, cu_all, ctx)
    q = gen((int(cu[-1]), Hq, d), 702, std)
    lse = torch.empty((Hq, int(cu[-1])), dtype=torch.float32, device=DEV)
    out = vpp.vpp_mixed_attn(q.to(DEV), kc, vc, tab, cu, ctx, lse=lse)
    torch.cuda.synchronize()
    assert vpp.vpp_last_device_status() == 0
    ks = [to_np64(k_all[starts[b]:starts[b + 1]]) for b in range(B)]
    vs = [to_np64(v_all[starts[b]:starts[b + 1]]) for b in range(B)]
    ref, ref_lse = oracle.mixed_batch_attention(to_np64(q), ks, vs, cu, ctx)
    assert_close(to_np64(out), ref)
    assert np.abs(to_np64(lse) - ref_lse).max() <= LSE_ABS


def test_mixed_batch_replays_in_a_cuda_graph():
    # The decode rows run on a side stream forked from the caller's stream by
    # events; a graph captured from the caller's stream must hold both branches
    # and replay to the eager result bit for bit.
    Hq, Hkv, d, nb = 8, 2, 128, 120
    ctx = np.array([500, 1, 1700, 300, 64], dtype=np.int32)
    qlen = np.array([200, 1, 1, 100, 1], dtype=np.int32)
    B = len(ctx)
    cu = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
    maxb = int(max((c + 63) // 64 for c in ctx))
    perm = np.random.default_rng(21).permutation(nb).astype(np.int32)
    table = np.full((B, maxb), -1, dtype=np.int32)
    kc = torch.zeros((nb, 64, Hkv, d), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    off = 0
    for b in range(B):
        n = (ctx[b] + 63) // 64
        table[b, :n] = perm[off:off + n]
        off += n
        k = gen((int(ctx[b]), Hkv, d), 400 + b, 1 / math.sqrt(d))
        v = gen((int(ctx[b]), Hkv, d), 500 + b, 1 / math.sqrt(d))
        vpp.vpp_kv_append(k.to(DEV), v.to(DEV), kc, vc, 0, block_table=torch.from_numpy(table[b].copy()).to(DEV))
    q = gen((int(cu[-1]), Hq, d), 600, 1 / math.sqrt(d)).to(DEV)
    tab = torch.from_numpy(table).to(DEV)
    need = vpp.mixed_attn_workspace_size(cu, ctx, Hq, Hkv, d, d)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=DEV)
    out_e = torch.empty((int(cu[-1]), Hq, d), dtype=torch.bfloat16, device=DEV)
    lse_e = torch.empty((Hq, int(cu[-1])), dtype=torch.float32, device=DEV)
    vpp.vpp_mixed_attn(q, kc, vc, tab, cu, ctx, out=out_e, lse=lse_e, workspace=ws)
    torch.cuda.synchronize()
    assert vpp.vpp_last_device_status() == 0
    out_g = torch.full_like(out_e, float("nan"))
    lse_g = torch.full_like(lse_e, float("nan"))
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(device=DEV)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph):
            vpp.vpp_mixed_attn(q, kc, vc, tab, cu, ctx, out=out_g, lse=lse_g, workspace=ws)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert vpp.vpp_last_device_status() == 0
    assert torch.equal(out_g.view(torch.int16), out_e.view(torch.int16))
    assert torch.equal(lse_g, lse_e)


def test_empty_chunk_is_a_noop():
    q = torch.empty((0, 8, 128), dtype=torch.bfloat16, device=DEV)
    kc = torch.zeros((64, 2, 128), dtype=torch.bfloat16, device=DEV)
    out = vpp.vpp_chunk_attn(q, kc, kc, 10)
    assert out.shape == (0, 8, 128)


def test_bounded_wait_times_out_and_context_survives():
    assert vpp.vpp_last_device_status() == 0
    vpp.vpp_selftest_wait_timeout(2000)
    assert vpp.vpp_last_device_status() == vpp.VPP_ERR_TIMEOUT
    assert vpp.vpp_last_device_status() == 0   # the read resets the word
    x = torch.ones(4, device=DEV)
    assert float((x * 2).sum()) == 8.0         # the context is still usable


def test_bad_block_table_entry_is_reported_not_faulted():
    Hq, Hkv, d, P, C = 4, 1, 128, 100, 28
    q, k, v = make_seq(P + C, Hq, Hkv, d, d, seed=95)
    cache = Cache(k, v, True, seed=5)
    bad = cache.table.clone()
    bad[1] = 10_000                                  # outside the pool
    vpp.vpp_chunk_attn_ex(q[P:].to(DEV), cache.k, cache.v, P, block_table=bad)
    torch.cuda.synchronize()
    assert vpp.vpp_last_device_status() == vpp.VPP_ERR_INVALID
