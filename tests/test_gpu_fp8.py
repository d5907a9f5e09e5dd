"""GPU parity of the fp8 (E4M3) KV-cache paths against the oracle.

Codes written by the quantising append are compared bit for bit with the
oracle's quantiser (oracle/fp8.py: the float32 quotient x / scale rounded to
E4M3, ties to even, saturating at 448), including exact ties, quotients that
tie only after float32 rounding, subnormal codes and saturation.  Attention
over the fp8 cache is compared with the fp64 oracle run on the dequantised
cache (code value x scale), to the bf16 path's tolerances: the kernels widen
the codes exactly to f16 operands (every E4M3 value is an f16 value) and
fold the scales in float32.
"""

import math

import numpy as np
import pytest
import torch

import oracle
import oracle.fp8 as ofp8
from chunked_prefill_causal_gb300 import vpp
from tests.helpers import LSE_ABS, assert_close, random_table, to_np64

pytestmark = pytest.mark.gpu

DEV = "cuda"
NAN_CODE = 0x7F


def gen(shape, seed, std):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to(torch.bfloat16)


def amax_scales(x, margin=1.0):
    """One float32 scale per kv head: the head's max |x| maps to 448 / margin."""
    a = x.float().abs().amax(dim=(0, 2)).numpy().astype(np.float64)
    return (np.maximum(a, 1e-30) * margin / 448.0).astype(np.float32)


def codes_of(cache, table, n_tokens):
    """Rows 0 .. n_tokens-1 of a paged uint8 cache, in token order."""
    c = cache.cpu().numpy()
    t = table.cpu().numpy()
    rows = [c[t[j // 64], j % 64] for j in range(n_tokens)]
    return np.stack(rows)


class Fp8Cache:
    """A paged E4M3 cache (pool pre-filled with the NaN code, random block
    order) holding a sequence's K/V, written through vpp_kv_append_fp8."""

    def __init__(self, k, v, ks, vs, seed=0, append_chunk=None, paged=True):
        L, Hkv, dq = k.shape
        dv = v.shape[2]
        self.ks = torch.from_numpy(ks).to(DEV)
        self.vs = torch.from_numpy(vs).to(DEV)
        if paged:
            need = (L + 63) // 64
            pool = need + 5
            self.table = torch.from_numpy(random_table(need, pool, seed)).to(DEV)
            self.k = torch.full((pool, 64, Hkv, dq), NAN_CODE, dtype=torch.uint8, device=DEV)
            self.v = torch.full((pool, 64, Hkv, dv), NAN_CODE, dtype=torch.uint8, device=DEV)
        else:
            self.table = None
            self.k = torch.full((L, Hkv, dq), NAN_CODE, dtype=torch.uint8, device=DEV)
            self.v = torch.full((L, Hkv, dv), NAN_CODE, dtype=torch.uint8, device=DEV)
        step = append_chunk or L
        for P in range(0, L, step):
            C = min(step, L - P)
            vpp.vpp_kv_append_fp8(k[P:P + C].to(DEV), v[P:P + C].to(DEV), self.k, self.v, self.ks, self.vs, P,
                                  block_table=self.table)


# ----------------------------------------------------------------- append
def _special_values():
    """Every E4M3 midpoint (ties), its neighbours one bf16 step away, values
    past 448, subnormal-range values and both zeros, for a head with scale 1."""
    v = ofp8.e4m3_decode(np.arange(0x7F))
    mids = (v[1:] + v[:-1]) / 2
    bf = lambda a: torch.tensor(a, dtype=torch.float64).to(torch.bfloat16)
    up = torch.nextafter(bf(mids).float(), torch.tensor(1e9)).to(torch.bfloat16)  # may round back: harmless
    vals = torch.cat([bf(mids), -bf(mids), up, bf([449.0, 464.0, 1000.0, -3e4, 2.0 ** -10, 3 * 2.0 ** -11,
                                                   -(2.0 ** -12), 0.0, -0.0, 448.0, -448.0])])
    return vals


def test_append_codes_are_bit_exact():
    Hkv, d, L = 6, 64, 700
    k = gen((L, Hkv, d), 1, 0.05)
    v = gen((L, Hkv, d), 2, 0.05)
    # head 0: scale 1 and the special values; heads 1-4: the float32 quotient
    # ties (x, s); head 5: a plain amax scale
    ks = amax_scales(k)
    vs = amax_scales(v, margin=0.7)      # 30% of V's range saturates
    sv = _special_values()
    n = min(sv.numel(), L * d)
    flat = k[:, 0, :].reshape(-1).clone()
    flat[:n] = sv[:n]
    k[:, 0, :] = flat.reshape(L, d)
    ks[0] = 1.0
    from tests.test_oracle_fp8 import QUOTIENT_TIES
    for h, (x, s, _) in enumerate(QUOTIENT_TIES, start=1):
        ks[h] = np.float32(s)
        k[: L // 2, h, : d // 2] = x
    cache = Fp8Cache(k, v, ks, vs, seed=3, append_chunk=250)
    torch.cuda.synchronize()
    assert vpp.vpp_last_device_status() == 0
    got_k = codes_of(cache.k, cache.table, L)
    got_v = codes_of(cache.v, cache.table, L)
    ref_k = ofp8.quantize_kv(k.float().numpy(), ks)
    ref_v = ofp8.quantize_kv(v.float().numpy(), vs)
    assert np.array_equal(got_k, ref_k), np.argwhere(got_k != ref_k)[:5]
    assert np.array_equal(got_v, ref_v), np.argwhere(got_v != ref_v)[:5]
    assert (ref_v & 0x7F == 0x7E).any()                  # saturation happened
    # blocks no token maps to still hold the fill code
    used = set(cache.table.cpu().numpy().tolist())
    spare = [b for b in range(cache.k.shape[0]) if b not in used]
    assert (cache.k[spare].cpu().numpy() == NAN_CODE).all()


def test_append_codes_bit_exact_over_many_scales():
    """8M elements per tensor, 64 kv heads with scales spread over eight decades (the
    quotient x / scale must be the correctly rounded float32 one for every
    code to agree)."""
    Hkv, d, L = 64, 64, 2048
    rng = np.random.default_rng(17)
    k = gen((L, Hkv, d), 21, 1.0)
    v = gen((L, Hkv, d), 22, 0.01)
    ks = (10.0 ** rng.uniform(-5, 3, Hkv)).astype(np.float32)
    vs = (10.0 ** rng.uniform(-7, 1, Hkv)).astype(np.float32)
    kc = torch.full((L, Hkv, d), NAN_CODE, dtype=torch.uint8, device=DEV)
    vc = torch.full((L, Hkv, d), NAN_CODE, dtype=torch.uint8, device=DEV)
    vpp.vpp_kv_append_fp8(k.to(DEV), v.to(DEV), kc, vc, torch.from_numpy(ks).to(DEV),
                          torch.from_numpy(vs).to(DEV), 0)
    torch.cuda.synchronize()
    assert vpp.vpp_last_device_status() == 0
    for got, x, s in ((kc, k, ks), (vc, v, vs)):
        ref = ofp8.quantize_kv(x.float().numpy(), s)
        g = got.cpu().numpy()
        assert np.array_equal(g, ref), (np.count_nonzero(g != ref), np.argwhere(g != ref)[:3])


def test_append_contiguous_and_varlen_place_the_same_codes():
    Hkv, d = 2, 128
    ctx = np.array([100, 64, 1, 300], dtype=np.int32)
    qlen = np.array([40, 64, 1, 129], dtype=np.int32)
    cu = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
    T = int(cu[-1])
    kn = gen((T, Hkv, d), 5, 0.1)
    vn = gen((T, Hkv, d), 6, 0.1)
    ks = amax_scales(kn)
    vs = amax_scales(vn)
    maxb = int(max((c + 63) // 64 for c in ctx))
    nb = 4 * maxb + 3
    perm = np.random.default_rng(9).permutation(nb).astype(np.int32)
    table = np.full((4, maxb), -1, dtype=np.int32)
    off = 0
    for b in range(4):
        n = (int(ctx[b]) + 63) // 64
        table[b, :n] = perm[off:off + n]
        off += n
    kc = torch.full((nb, 64, Hkv, d), NAN_CODE, dtype=torch.uint8, device=DEV)
    vc = torch.full_like(kc, NAN_CODE)
    vpp.vpp_kv_append_varlen_fp8(kn.to(DEV), vn.to(DEV), kc, vc, torch.from_numpy(ks).to(DEV),
                                 torch.from_numpy(vs).to(DEV), torch.from_numpy(table).to(DEV), cu, ctx)
    torch.cuda.synchronize()
    assert vpp.vpp_last_device_status() == 0
    ref = np.full((nb, 64, Hkv, d), NAN_CODE, dtype=np.uint8)
    codes = ofp8.quantize_kv(kn.float().numpy(), ks)
    for b in range(4):
        oracle.kv_append(ref, table[b], codes[cu[b]:cu[b + 1]], int(ctx[b] - qlen[b]))
    assert np.array_equal(kc.cpu().numpy(), ref)
    # contiguous cache: row j holds token j
    cc = torch.full((T + 10, Hkv, d), NAN_CODE, dtype=torch.uint8, device=DEV)
    cv = torch.full((T + 10, Hkv, d), NAN_CODE, dtype=torch.uint8, device=DEV)
    vpp.vpp_kv_append_fp8(kn.to(DEV), vn.to(DEV), cc, cv, torch.from_numpy(ks).to(DEV),
                          torch.from_numpy(vs).to(DEV), 10)
    torch.cuda.synchronize()
    got = cc.cpu().numpy()
    assert np.array_equal(got[10:], codes) and (got[:10] == NAN_CODE).all()


# ----------------------------------------------------------------- attention
def run_fp8(P, C, Hq, Hkv, dq, dv, seed, num_splits=0, paged=True, append_chunk=None, widen=False):
    std = 1 / math.sqrt(dq)
    q = gen((C, Hq, dq), seed, std)
    k = gen((P + C, Hkv, dq), seed + 1, std)
    v = gen((P + C, Hkv, dv), seed + 2, std)
    ks = amax_scales(k) * np.float32(1.0 + 0.01 * seed % 3)
    vs = amax_scales(v)
    cache = Fp8Cache(k, v, ks, vs, seed=seed, append_chunk=append_chunk, paged=paged)
    lse = torch.empty((Hq, C), dtype=torch.float32, device=DEV)
    out = vpp.vpp_chunk_attn_fp8(q.to(DEV), cache.k, cache.v, cache.ks, cache.vs, P, block_table=cache.table,
                                 lse=lse, num_splits=num_splits, widen=widen)
    torch.cuda.synchronize()
    assert vpp.vpp_last_device_status() == 0
    kq = ofp8.dequantize_kv(ofp8.quantize_kv(k.float().numpy(), ks), ks)
    vq = ofp8.dequantize_kv(ofp8.quantize_kv(v.float().numpy(), vs), vs)
    ref, ref_lse = oracle.causal_chunk_attention(to_np64(q), kq, vq, P)
    assert_close(to_np64(out), ref)
    assert np.abs(to_np64(lse) - ref_lse).max() <= LSE_ABS
    return out


FP8_CASES = [  # P, C, Hq, Hkv, dq, dv, paged
    (0, 1, 8, 2, 128, 128, True),
    (0, 300, 8, 2, 128, 128, True),
    (640, 37, 8, 2, 128, 128, True),
    (1000, 129, 32, 8, 128, 128, False),
    (130, 70, 16, 2, 128, 128, True),    # G = 8
    (700, 129, 4, 4, 192, 128, True),    # MLA-shaped
    (250, 90, 4, 2, 64, 64, True),
    (250, 90, 4, 2, 192, 64, False),
    (333, 64, 8, 4, 64, 128, True),
    (200, 200, 2, 1, 128, 64, False),
    (1500, 260, 16, 2, 192, 128, True),  # MLA head dims, G = 8, many tiles
]


@pytest.mark.parametrize("case", FP8_CASES, ids=lambda c: "P%d_C%d_H%d-%d_d%d-%d_%s" % (
    c[0], c[1], c[2], c[3], c[4], c[5], "paged" if c[6] else "contig"))
def test_chunk_attention_over_fp8_cache(case):
    P, C, Hq, Hkv, dq, dv, paged = case
    run_fp8(P, C, Hq, Hkv, dq, dv, seed=sum(case[:6]) % 997, paged=paged, append_chunk=200)


@pytest.mark.parametrize("splits", [1, 3, 0])
def test_fp8_split_prefix_matches(splits):
    run_fp8(2000, 100, 8, 2, 128, 128, seed=41, num_splits=splits)


def test_fp8_heavy_query_tiles_split_by_the_library():
    # The library's own plan for this shape splits only the keys of the tokens
    # from 1152 on (3 ranges); over an E4M3 cache the codes are widened inside
    # the kernel for both segments, and the merge covers the split tokens.
    P, C, Hq, Hkv, d = 4096, 1536, 32, 8, 128
    assert vpp.chunk_attn_plan(P, C, Hq, Hkv, d, d) == (3, 1152)
    run_fp8(P, C, Hq, Hkv, d, d, seed=61)


@pytest.mark.parametrize("case", [(640, 37, 8, 2, 128, 128, True, 0), (700, 129, 4, 4, 192, 128, True, 3),
                                  (250, 90, 4, 2, 192, 64, False, 0)],
                         ids=["d128_paged", "d192_paged_split3", "d192-64_contig"])
def test_fp8_widened_copy_path(case):
    # with room for a bf16 copy of the visible keys the codes are widened once
    # in HBM and the bf16 kernel reads the copy
    P, C, Hq, Hkv, dq, dv, paged, splits = case
    assert vpp.chunk_attn_fp8_widen_workspace_size(P, C, Hq, Hkv, dq, dv, splits) >= \
        2 * (P + C) * Hkv * min(dq, dv) * 2
    run_fp8(P, C, Hq, Hkv, dq, dv, seed=P + dq, paged=paged, num_splits=splits, widen=True)


def test_fp8_workspace_holds_split_partials_only():
    # The codes are widened inside the kernel: without a key split no
    # workspace is needed, and a split needs its float32 partials (which do
    # not depend on the prefix length), refused when the buffer is short.
    P, C, Hq, Hkv, d = 3000, 28, 4, 1, 128
    assert vpp.chunk_attn_fp8_workspace_size(P, C, Hq, Hkv, d, d, 1) == 0
    need = vpp.chunk_attn_fp8_workspace_size(P, C, Hq, Hkv, d, d, 3)
    assert need >= 3 * C * Hq * (d + 1) * 4
    assert vpp.chunk_attn_fp8_workspace_size(30 * P, C, Hq, Hkv, d, d, 3) == need
    k = gen((P + C, Hkv, d), 7, 0.1)
    cache = Fp8Cache(k, k, amax_scales(k), amax_scales(k), seed=1)
    q = gen((C, Hq, d), 8, 0.1).to(DEV)
    small = torch.empty(need - 256, dtype=torch.uint8, device=DEV)
    with pytest.raises(vpp.VppError) as e:
        vpp.vpp_chunk_attn_fp8(q, cache.k, cache.v, cache.ks, cache.vs, P, block_table=cache.table,
                               num_splits=3, workspace=small)
    assert e.value.code == vpp.VPP_ERR_WORKSPACE
    out = vpp.vpp_chunk_attn_fp8(q, cache.k, cache.v, cache.ks, cache.vs, P, block_table=cache.table,
                                 num_splits=1)
    torch.cuda.synchronize()
    assert vpp.vpp_last_device_status() == 0
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("qmul", [1e-5, 3000.0])
def test_fp8_chunk_attention_with_extreme_query_scales(qmul):
    # q is turned into f16 operands in the kernel: very small and very large
    # (but f16-representable) queries must give the oracle's result.
    P, C, Hq, Hkv, d = 700, 150, 8, 2, 128
    q = (gen((C, Hq, d), 61, 1 / math.sqrt(d)).float() * qmul).to(torch.bfloat16)
    k = gen((P + C, Hkv, d), 62, 1 / math.sqrt(d))
    v = gen((P + C, Hkv, d), 63, 1 / math.sqrt(d))
    ks, vs = amax_scales(k), amax_scales(v)
    cache = Fp8Cache(k, v, ks, vs, seed=4)
    lse = torch.empty((Hq, C), dtype=torch.float32, device=DEV)
    out = vpp.vpp_chunk_attn_fp8(q.to(DEV), cache.k, cache.v, cache.ks, cache.vs, P, block_table=cache.table,
                                 lse=lse)
    torch.cuda.synchronize()
    assert vpp.vpp_last_device_status() == 0
    kq = ofp8.dequantize_kv(ofp8.quantize_kv(k.float().numpy(), ks), ks)
    vq = ofp8.dequantize_kv(ofp8.quantize_kv(v.float().numpy(), vs), vs)
    ref, ref_lse = oracle.causal_chunk_attention(to_np64(q), kq, vq, P)
    assert_close(to_np64(out), ref)
    assert np.abs(to_np64(lse) - ref_lse).max() <= LSE_ABS


def test_fp8_query_outside_f16_range_is_reported():
    P, C, Hq, Hkv, d = 200, 40, 4, 1, 64
    q = gen((C, Hq, d), 71, 0.1)
    q[5, 2, 7] = 1.0e5  # beyond f16's largest finite value
    k = gen((P + C, Hkv, d), 72, 0.1)
    cache = Fp8Cache(k, k, amax_scales(k), amax_scales(k), seed=5)
    vpp.vpp_chunk_attn_fp8(q.to(DEV), cache.k, cache.v, cache.ks, cache.vs, P, block_table=cache.table)
    torch.cuda.synchronize()
    assert vpp.vpp_last_device_status() == vpp.VPP_ERR_INVALID
    assert vpp.vpp_last_device_status() == 0  # the report is read once


# ----------------------------------------------------------------- mixed batch
CTX = [1, 2, 15, 16, 17, 63, 64, 65, 1000, 1023, 1024, 1025, 2048, 3001]


def _mixed(ctx, qlen, Hq, Hkv, d, seed, qmul=1.0, widen=False):
    B = len(ctx)
    cu = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
    need = [(int(c) + 63) // 64 for c in ctx]
    maxb = max(need)
    pool = sum(need) + 3
    perm = np.random.default_rng(seed).permutation(pool).astype(np.int32)
    table = np.full((B, maxb), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[off:off + n]
        off += n
    std = 1 / math.sqrt(d)
    ks_ = [gen((int(ctx[b]), Hkv, d), seed + 10 + b, std) for b in range(B)]
    vs_ = [gen((int(ctx[b]), Hkv, d), seed + 500 + b, std) for b in range(B)]
    kscale = amax_scales(torch.cat(ks_))
    vscale = amax_scales(torch.cat(vs_))
    kc = torch.full((pool, 64, Hkv, d), NAN_CODE, dtype=torch.uint8, device=DEV)
    vc = torch.full_like(kc, NAN_CODE)
    ksd, vsd = torch.from_numpy(kscale).to(DEV), torch.from_numpy(vscale).to(DEV)
    for b in range(B):
        vpp.vpp_kv_append_fp8(ks_[b].to(DEV), vs_[b].to(DEV), kc, vc, ksd, vsd, 0,
                              block_table=torch.from_numpy(table[b].copy()).to(DEV))
    q = gen((int(cu[-1]), Hq, d), seed + 999, std)
    if qmul != 1.0:
        q = (q.float() * qmul).to(torch.bfloat16)
    lse = torch.empty((Hq, int(cu[-1])), dtype=torch.float32, device=DEV)
    out = vpp.vpp_mixed_attn_fp8(q.to(DEV), kc, vc, ksd, vsd, torch.from_numpy(table).to(DEV), cu,
                                 np.asarray(ctx, dtype=np.int32), lse=lse, widen=widen)
    torch.cuda.synchronize()
    assert vpp.vpp_last_device_status() == 0
    kq = [ofp8.dequantize_kv(ofp8.quantize_kv(x.float().numpy(), kscale), kscale) for x in ks_]
    vq = [ofp8.dequantize_kv(ofp8.quantize_kv(x.float().numpy(), vscale), vscale) for x in vs_]
    ref, ref_lse = oracle.mixed_batch_attention(to_np64(q), kq, vq, cu, np.asarray(ctx))
    assert_close(to_np64(out), ref)
    assert np.abs(to_np64(lse) - ref_lse).max() <= LSE_ABS


@pytest.mark.parametrize("Hq,Hkv,d", [(32, 8, 128), (8, 8, 128), (64, 8, 64), (64, 8, 128), (4, 1, 64), (128, 8, 128)])
def test_fp8_decode_rows_match_oracle(Hq, Hkv, d):
    _mixed(CTX, [1] * len(CTX), Hq, Hkv, d, seed=Hq + d)


@pytest.mark.parametrize("qmul", [1e-6, 40.0])
def test_fp8_decode_rows_with_extreme_query_scales(qmul):
    # The tensor-core decode scales q by a power of two per head into f16's
    # range: tiny and large queries must give the oracle's result.
    _mixed([1, 17, 1000, 2048, 3001], [1] * 5, 32, 8, 128, seed=5, qmul=qmul)


@pytest.mark.parametrize("widen", [False, True])
def test_fp8_mixed_prefill_and_decode(widen):
    ctx = [300, 700, 64, 129, 1, 2000, 513, 4100]
    qlen = [300, 128, 1, 1, 1, 1, 77, 1]
    _mixed(ctx, qlen, 8, 2, 128, seed=77, widen=widen)


@pytest.mark.parametrize("splits", [1, 3])
@pytest.mark.parametrize("case", [(8, 8, 128, 128, 1500, 300), (16, 2, 128, 128, 1500, 300),
                                  (4, 4, 192, 128, 1300, 260)], ids=lambda c: "H%d-%d_d%d-%d_P%d_C%d" % c)
def test_fp8_chunk_attention_with_growing_scores(case, splits):
    # The running maximum moves on many tiles (keys grow with their position
    # and each 128-key tile holds a needle ~20 log2 units above the last), with
    # the codes widened inside the kernel: the reference, the denominator and
    # the output accumulator must move together over the widened operands.
    from tests.test_gpu_rescale import growing_scores
    Hq, Hkv, dq, dv, P, C = case
    q, k, v = growing_scores(P + C, Hq, Hkv, dq, dv, seed=Hq * 5 + dq)
    ks, vs = amax_scales(k), amax_scales(v)
    cache = Fp8Cache(k, v, ks, vs, seed=splits, append_chunk=400)
    lse = torch.empty((Hq, C), dtype=torch.float32, device=DEV)
    out = vpp.vpp_chunk_attn_fp8(q[P:].to(DEV), cache.k, cache.v, cache.ks, cache.vs, P, block_table=cache.table,
                                 lse=lse, num_splits=splits)
    torch.cuda.synchronize()
    assert vpp.vpp_last_device_status() == 0
    kq = ofp8.dequantize_kv(ofp8.quantize_kv(k.float().numpy(), ks), ks)
    vq = ofp8.dequantize_kv(ofp8.quantize_kv(v.float().numpy(), vs), vs)
    ref, ref_lse = oracle.causal_chunk_attention(to_np64(q[P:]), kq, vq, P)
    assert ref_lse[:, -1].max() / math.log(2) > 100
    assert_close(to_np64(out), ref)
    assert np.abs(to_np64(lse) - ref_lse).max() <= LSE_ABS
