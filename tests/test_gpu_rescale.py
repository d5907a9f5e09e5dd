"""GPU parity where the running softmax maximum keeps growing.

Eq. (1) of "VPP: Virtual Pipeline Parallelism for Efficient Chunked Prefill
in Long-Context LLM Inference" (technical review, §2.2) is evaluated online
over key tiles: each row keeps a reference and a denominator and moves both
(together with its output accumulator) when a later tile holds much larger
scores.  Random N(0,1)/sqrt(d) inputs almost never do that, so these cases
are built to do it on many tiles:

* unscaled N(0,1) queries, and keys scaled up with their position
  (K[j] *= 1 + j/256), so later keys score higher;
* one "needle" key per 128-key tile along a direction every query shares,
  whose score grows by about 20 log2 units per tile, placed in the first or
  the second 64-key half of its tile.

Every case is checked against the fp64 oracle at the usual tolerances
(max-abs 2e-2, relative L2 5e-3, LSE 1e-2): chunk attention unsplit and
split, head dims 128 and 192, one and eight query heads per kv head, decode
rows of a mixed batch, and top-k lists that cover every earlier key.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import sparse as osp
from chunked_prefill_causal_gb300 import vpp
from tests.helpers import LSE_ABS, assert_close, random_table, to_np64

pytestmark = pytest.mark.gpu

DEV = "cuda"
LOG2E = 1.4426950408889634


def growing_scores(L, Hq, Hkv, dq, dv, seed, step_log2=20.0):
    """bf16 q [L, Hq, dq], k [L, Hkv, dq], v [L, Hkv, dv] whose scores grow
    along the sequence (see the module docstring)."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    u = torch.randn(dq, generator=g)
    u = u / u.norm()
    q = torch.randn((L, Hq, dq), generator=g) + 2.0 * u
    k = torch.randn((L, Hkv, dq), generator=g) * (1.0 + torch.arange(L, dtype=torch.float32) / 256.0)[:, None, None]
    v = torch.randn((L, Hkv, dv), generator=g) / math.sqrt(dv)
    for t in range((L + 127) // 128):
        j = 128 * t + ((37 * t + 5) % 128)  # alternates between the two 64-key halves
        if j >= L:
            break
        # score ~ q.u * a / sqrt(dq) ~ 2 a / sqrt(dq): step_log2 more per tile
        a = step_log2 * (t + 1) * math.sqrt(dq) / (2.0 * LOG2E)
        k[j] = a * u
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)


def paged_cache(k, v, seed):
    L, Hkv, dq = k.shape
    dv = v.shape[2]
    need = (L + 63) // 64
    pool = need + 4
    table = torch.from_numpy(random_table(need, pool, seed)).to(DEV)
    kc = torch.full((pool, 64, Hkv, dq), float("nan"), dtype=torch.bfloat16, device=DEV)
    vc = torch.full((pool, 64, Hkv, dv), float("nan"), dtype=torch.bfloat16, device=DEV)
    vpp.vpp_kv_append(k.to(DEV), v.to(DEV), kc, vc, 0, block_table=table)
    return kc, vc, table


CHUNK_CASES = [  # Hq, Hkv, dq, dv, P, C
    (8, 8, 128, 128, 1500, 300),    # G = 1
    (16, 2, 128, 128, 1500, 300),   # G = 8
    (4, 4, 192, 128, 1300, 260),    # MLA head dims, G = 1
    (16, 2, 192, 128, 1300, 260),   # MLA head dims, G = 8
]


@pytest.mark.parametrize("splits", [1, 3])
@pytest.mark.parametrize("case", CHUNK_CASES, ids=lambda c: "H%d-%d_d%d-%d_P%d_C%d" % c)
def test_chunk_attention_with_growing_scores(case, splits):
    Hq, Hkv, dq, dv, P, C = case
    q, k, v = growing_scores(P + C, Hq, Hkv, dq, dv, seed=Hq * 7 + dq)
    kc, vc, table = paged_cache(k, v, seed=3)
    lse = torch.empty((Hq, C), dtype=torch.float32, device=DEV)
    out = vpp.vpp_chunk_attn_ex(q[P:].to(DEV), kc, vc, P, block_table=table, lse=lse, num_splits=splits)
    torch.cuda.synchronize()
    assert vpp.vpp_last_device_status() == 0
    ref, ref_lse = oracle.causal_chunk_attention(to_np64(q[P:]), to_np64(k), to_np64(v), P)
    # the case does what it is for: the last rows' scores span well over 2^100
    assert ref_lse[:, -1].max() / math.log(2) > 100
    assert_close(to_np64(out), ref)
    assert np.abs(to_np64(lse) - ref_lse).max() <= LSE_ABS


def test_whole_sequence_in_one_chunk_with_growing_scores():
    # P = 0: every query tile starts from its own first key tile
    Hq, Hkv, d, L = 8, 2, 128, 1200
    q, k, v = growing_scores(L, Hq, Hkv, d, d, seed=91)
    kc, vc, table = paged_cache(k, v, seed=4)
    lse = torch.empty((Hq, L), dtype=torch.float32, device=DEV)
    out = vpp.vpp_chunk_attn_ex(q.to(DEV), kc, vc, 0, block_table=table, lse=lse)
    torch.cuda.synchronize()
    assert vpp.vpp_last_device_status() == 0
    ref, ref_lse = oracle.causal_chunk_attention(to_np64(q), to_np64(k), to_np64(v), 0)
    assert_close(to_np64(out), ref)
    assert np.abs(to_np64(lse) - ref_lse).max() <= LSE_ABS


@pytest.mark.parametrize("Hq,Hkv,d", [(32, 8, 128), (8, 8, 128), (16, 2, 64)])
def test_decode_rows_with_growing_scores(Hq, Hkv, d):
    ctxs = [3000, 2100, 1025, 700, 129]
    B = len(ctxs)
    ks, vs, qs = [], [], []
    for b, c in enumerate(ctxs):
        q, k, v = growing_scores(c, Hq, Hkv, d, d, seed=200 + b)
        ks.append(k)
        vs.append(v)
        qs.append(q[c - 1:c])
    need = [(c + 63) // 64 for c in ctxs]
    pool = sum(need) + 3
    perm = np.random.default_rng(Hq + d).permutation(pool).astype(np.int32)
    table = np.full((B, max(need)), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[off:off + n]
        off += n
    kc = torch.full((pool, 64, Hkv, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    vc = torch.full_like(kc, float("nan"))
    for b in range(B):
        vpp.vpp_kv_append(ks[b].to(DEV), vs[b].to(DEV), kc, vc, 0,
                          block_table=torch.from_numpy(table[b].copy()).to(DEV))
    q = torch.cat(qs)
    cu = np.arange(B + 1, dtype=np.int32)
    ctx = np.array(ctxs, dtype=np.int32)
    lse = torch.empty((Hq, B), dtype=torch.float32, device=DEV)
    out = vpp.vpp_mixed_attn(q.to(DEV), kc, vc, torch.from_numpy(table).to(DEV), cu, ctx, lse=lse)
    torch.cuda.synchronize()
    assert vpp.vpp_last_device_status() == 0
    ref, ref_lse = oracle.mixed_batch_attention(to_np64(q), [to_np64(x) for x in ks], [to_np64(x) for x in vs],
                                                cu, ctx)
    assert_close(to_np64(out), ref)
    assert np.abs(to_np64(lse) - ref_lse).max() <= LSE_ABS


@pytest.mark.parametrize("Hq,Hkv,d", [(8, 2, 128), (16, 8, 64)])
def test_topk_gather_with_growing_scores(Hq, Hkv, d):
    # lists long enough to hold every earlier key: the gather path's online
    # softmax sees the same growing scores as dense attention
    P, C, topk = 1500, 200, 2048
    q, k, v = growing_scores(P + C, Hq, Hkv, d, d, seed=300 + Hq)
    idx = np.zeros((C, topk), dtype=np.int32)
    lens = np.zeros(C, dtype=np.int32)
    for i in range(C):
        n = P + i + 1
        idx[i, :n] = np.arange(n, dtype=np.int32)
        lens[i] = n
    kc, vc, table = paged_cache(k, v, seed=5)
    lse = torch.empty((Hq, C), dtype=torch.float32, device=DEV)
    out = vpp.vpp_topk_chunk_attn(q[P:].to(DEV), kc, vc, P, torch.from_numpy(idx).to(DEV),
                                  torch.from_numpy(lens).to(DEV), block_table=table, lse=lse)
    torch.cuda.synchronize()
    assert vpp.vpp_last_device_status() == 0
    ref, ref_lse = osp.topk_chunk_attention(to_np64(q[P:]), to_np64(k), to_np64(v), P, idx, lens)
    assert_close(to_np64(out), ref)
    assert np.abs(to_np64(lse) - ref_lse).max() <= LSE_ABS
