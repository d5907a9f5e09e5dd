"""GPU parity of top-k sparse prefix attention (DSA-style) against the oracle.

Each query token attends only its listed keys (oracle/sparse.py).  Lists are
drawn by workloads.topk_indices; the pool is NaN-filled so that a read of an
unlisted or unwritten row would show.  Tolerances are those of the bf16 path.
"""

import math

import numpy as np
import pytest
import torch

import oracle.fp8 as ofp8
import oracle.sparse as osp
from chunked_prefill_causal_gb300 import vpp
from chunked_prefill_causal_gb300 import workloads as W
from tests.helpers import LSE_ABS, assert_close, random_table, to_np64

pytestmark = pytest.mark.gpu

DEV = "cuda"


def gen(shape, seed, std):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to(torch.bfloat16)


def paged(k, v, seed):
    L, Hkv, d = k.shape
    need = (L + 63) // 64
    pool = need + 5
    table = torch.from_numpy(random_table(need, pool, seed)).to(DEV)
    kc = torch.full((pool, 64, Hkv, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    vc = torch.full_like(kc, float("nan"))
    for P in range(0, L, 1000):
        C = min(1000, L - P)
        vpp.vpp_kv_append(k[P:P + C].to(DEV), v[P:P + C].to(DEV), kc, vc, P, block_table=table)
    return kc, vc, table


def run_case(Hq, Hkv, d, P, C, topk, seed, paged_cache=True):
    std = 1 / math.sqrt(d)
    q = gen((C, Hq, d), seed, std)
    k = gen((P + C, Hkv, d), seed + 1, std)
    v = gen((P + C, Hkv, d), seed + 2, std)
    idx, lens = W.topk_indices(P, C, topk, seed)
    if paged_cache:
        kc, vc, table = paged(k, v, seed)
    else:
        kc, vc, table = k.to(DEV), v.to(DEV), None
    lse = torch.empty((Hq, C), dtype=torch.float32, device=DEV)
    out = vpp.vpp_topk_chunk_attn(q.to(DEV), kc, vc, P, idx.to(DEV), lens.to(DEV), block_table=table, lse=lse)
    torch.cuda.synchronize()
    assert vpp.vpp_last_device_status() == 0
    ref, ref_lse = osp.topk_chunk_attention(to_np64(q), to_np64(k), to_np64(v), P, idx.numpy(), lens.numpy())
    assert_close(to_np64(out), ref)
    assert np.abs(to_np64(lse) - ref_lse).max() <= LSE_ABS


CASES = [  # Hq, Hkv, d, P, C, topk, paged
    (8, 2, 128, 0, 300, 64, True),        # first 64 tokens list every earlier key, then sparse
    (8, 2, 128, 1000, 129, 256, True),
    (8, 2, 128, 3000, 77, 2048, True),    # two 1024-entry ranges per token, merged
    (8, 2, 128, 500, 60, 1500, False),    # one or two ranges depending on the position
    (4, 4, 64, 700, 50, 300, True),       # G = 1
    (8, 1, 64, 2000, 40, 1100, True),     # G = 8, d 64
    (4, 2, 128, 100, 33, 7, True),        # G = 2, lists shorter than one 16-key step
    # more kv heads per token row (one warp each, 4 gather warps for bf16)
    (16, 8, 128, 1500, 70, 2048, True),
    (12, 6, 64, 900, 45, 1200, False),    # contiguous cache
    (10, 5, 128, 600, 40, 500, True),
    (56, 7, 64, 400, 30, 300, True),      # G = 8
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "H%d-%d_d%d_P%d_C%d_k%d_%s" % (
    c[0], c[1], c[2], c[3], c[4], c[5], "paged" if c[6] else "contig"))
def test_topk_attention_matches_oracle(case):
    Hq, Hkv, d, P, C, topk, pg = case
    run_case(Hq, Hkv, d, P, C, topk, seed=sum(case[:6]) % 991, paged_cache=pg)


@pytest.mark.parametrize("Hq,Hkv,d,topk", [(8, 2, 128, 96), (16, 8, 64, 300)])
def test_invalid_entries_are_masked_and_reported(Hq, Hkv, d, topk):
    P, C = 400, 20
    std = 1 / math.sqrt(d)
    q = gen((C, Hq, d), 61, std)
    k = gen((P + C, Hkv, d), 62, std)
    v = gen((P + C, Hkv, d), 63, std)
    idx, lens = W.topk_indices(P, C, topk, 5)
    idx, lens = idx.numpy().copy(), lens.numpy().copy()
    bad = idx.copy()
    bad[0, 3] = -5                       # negative
    bad[1, 10] = P + 1 + 50              # after the query's own position
    bad[2, :lens[2]] = P + C + 10        # every entry beyond the cache: the row is empty
    if topk > 256:                       # entries in later groups of 128 (resolved ahead of the copies)
        bad[0, 200] = -1
        bad[1, 140] = P + 1 + 7
        bad[1, 299] = P + 1 + 9
    kc, vc, table = paged(k, v, 8)
    lse = torch.empty((Hq, C), dtype=torch.float32, device=DEV)
    out = vpp.vpp_topk_chunk_attn(q.to(DEV), kc, vc, P, torch.from_numpy(bad).to(DEV),
                                  torch.from_numpy(lens).to(DEV), block_table=table, lse=lse)
    torch.cuda.synchronize()
    assert vpp.vpp_last_device_status() == vpp.VPP_ERR_INVALID
    got = to_np64(out)
    got_lse = to_np64(lse)
    # rows 0 and 1: the oracle over the remaining valid entries
    for r in (0, 1):
        keep = [j for j in bad[r, :lens[r]] if 0 <= j <= P + r]
        ref, ref_lse = osp.topk_rows(to_np64(q[r:r + 1]), np.array([keep]), [len(keep)], to_np64(k), to_np64(v),
                                     Hq // Hkv)
        assert_close(got[r:r + 1], ref)
        assert np.abs(got_lse[:, r] - ref_lse[:, 0]).max() <= LSE_ABS
    assert np.all(got[2] == 0) and np.all(np.isneginf(got_lse[:, 2]))
    # untouched rows are unaffected
    ref, ref_lse = osp.topk_chunk_attention(to_np64(q[3:]), to_np64(k[:P + C]), to_np64(v[:P + C]), P + 3,
                                            idx[3:], lens[3:])
    assert_close(got[3:], ref)


def test_bad_list_length_gives_an_empty_row():
    Hq, Hkv, d, P, C, topk = 4, 2, 64, 100, 4, 32
    std = 1 / math.sqrt(d)
    q = gen((C, Hq, d), 71, std)
    k = gen((P + C, Hkv, d), 72, std)
    v = gen((P + C, Hkv, d), 73, std)
    idx, lens = W.topk_indices(P, C, topk, 9)
    lens = lens.clone()
    lens[1] = 0
    lens[2] = topk + 1
    kc, vc, table = paged(k, v, 4)
    lse = torch.empty((Hq, C), dtype=torch.float32, device=DEV)
    out = vpp.vpp_topk_chunk_attn(q.to(DEV), kc, vc, P, idx.to(DEV), lens.to(DEV), block_table=table, lse=lse)
    torch.cuda.synchronize()
    assert vpp.vpp_last_device_status() == vpp.VPP_ERR_INVALID
    got, got_lse = to_np64(out), to_np64(lse)
    for r in (1, 2):
        assert np.all(got[r] == 0) and np.all(np.isneginf(got_lse[:, r]))
    for r in (0, 3):
        ref, ref_lse = osp.topk_rows(to_np64(q[r:r + 1]), idx.numpy()[r:r + 1], lens.numpy()[r:r + 1], to_np64(k),
                                     to_np64(v), Hq // Hkv)
        assert_close(got[r:r + 1], ref)


@pytest.mark.parametrize("Hq,Hkv,d", [(8, 2, 128), (16, 8, 128), (48, 6, 64)])
def test_topk_over_fp8_cache(Hq, Hkv, d):
    P, C, topk = 2500, 50, 2048
    std = 1 / math.sqrt(d)
    q = gen((C, Hq, d), 81, std)
    k = gen((P + C, Hkv, d), 82, std)
    v = gen((P + C, Hkv, d), 83, std)
    ks = (k.float().abs().amax(dim=(0, 2)).numpy() / 448).astype(np.float32)
    vs = (v.float().abs().amax(dim=(0, 2)).numpy() / 448).astype(np.float32)
    need = (P + C + 63) // 64
    table = torch.from_numpy(random_table(need, need + 3, 12)).to(DEV)
    kc = torch.full((need + 3, 64, Hkv, d), 0x7F, dtype=torch.uint8, device=DEV)
    vc = torch.full_like(kc, 0x7F)
    ksd, vsd = torch.from_numpy(ks).to(DEV), torch.from_numpy(vs).to(DEV)
    vpp.vpp_kv_append_fp8(k.to(DEV), v.to(DEV), kc, vc, ksd, vsd, 0, block_table=table)
    idx, lens = W.topk_indices(P, C, topk, 13)
    lse = torch.empty((Hq, C), dtype=torch.float32, device=DEV)
    out = vpp.vpp_topk_chunk_attn_fp8(q.to(DEV), kc, vc, ksd, vsd, P, idx.to(DEV), lens.to(DEV), block_table=table,
                                      lse=lse)
    torch.cuda.synchronize()
    assert vpp.vpp_last_device_status() == 0
    kq = ofp8.dequantize_kv(ofp8.quantize_kv(k.float().numpy(), ks), ks)
    vq = ofp8.dequantize_kv(ofp8.quantize_kv(v.float().numpy(), vs), vs)
    ref, ref_lse = osp.topk_chunk_attention(to_np64(q), kq, vq, P, idx.numpy(), lens.numpy())
    assert_close(to_np64(out), ref)
    assert np.abs(to_np64(lse) - ref_lse).max() <= LSE_ABS


def test_full_size_dsa128k_last_chunk_sampled_rows():
    w = W.WORKLOADS["dsa128k"]
    chunks = w.chunks()
    P, C = chunks[-1]
    dev = torch.device(DEV)
    nb = W.blocks_for(P + C)
    table = torch.from_numpy(W.block_table(nb, nb + 8, w.seed + 99)).to(dev)
    kc = torch.zeros((nb + 8, 64, w.kv_heads, w.head_dim_qk), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    kparts, vparts = [], []
    for ci, (p0, c0) in enumerate(chunks):
        qi, ki, vi = W.chunk_tensors(w, ci, dev)
        vpp.vpp_kv_append(ki, vi, kc, vc, p0, block_table=table)
        kparts.append(ki.cpu())   # the oracle reads the very values the kernel reads
        vparts.append(vi.cpu())
    idx, lens = W.topk_indices(P, C, W.TOPK, 3, device=dev)
    out = vpp.vpp_topk_chunk_attn(qi, kc, vc, P, idx, lens, block_table=table)
    torch.cuda.synchronize()
    assert vpp.vpp_last_device_status() == 0
    rows = np.random.default_rng(4).choice(C, 48, replace=False)
    rows = np.concatenate([[0, C - 1], rows])
    kseq = torch.cat(kparts).float().numpy()
    vseq = torch.cat(vparts).float().numpy()
    ref, _ = osp.topk_rows(to_np64(qi[rows]), idx[rows].cpu().numpy(), lens[rows].cpu().numpy(), kseq, vseq,
                           w.heads // w.kv_heads, positions=P + rows)
    assert_close(to_np64(out[rows]), ref)
