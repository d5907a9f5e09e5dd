"""Decode rows of a mixed batch (split-KV decode kernel) against the oracle.

Contexts sit on both sides of the 16-token step, the 64-token block and the
1024-key range boundaries; shapes cover every head grouping the decode kernel
takes and two it hands to the chunk kernel.  The pool is NaN-filled, so a
read past a row's context would show.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from chunked_prefill_causal_gb300 import vpp
from tests.helpers import LSE_ABS, assert_close, to_np64

pytestmark = pytest.mark.gpu

DEV = "cuda"
CTX = [1, 2, 15, 16, 17, 63, 64, 65, 1000, 1023, 1024, 1025, 2048, 3001, 5000]


def _gen(shape, seed, std):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to(torch.bfloat16)


@pytest.mark.parametrize("Hq,Hkv,d", [(32, 8, 128), (8, 8, 128), (16, 8, 64), (64, 8, 64), (64, 8, 128),
                                      (8, 2, 128), (4, 1, 64), (128, 8, 128), (16, 16, 64)])
def test_decode_rows_match_oracle(Hq, Hkv, d):
    B = len(CTX)
    ctx = np.array(CTX, dtype=np.int32)
    cu = np.arange(B + 1, dtype=np.int32)
    need = [(c + 63) // 64 for c in CTX]
    maxb = max(need)
    pool = sum(need) + 3
    perm = np.random.default_rng(Hq * 100 + d).permutation(pool).astype(np.int32)
    table = np.full((B, maxb), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[off:off + n]
        off += n
    kc = torch.full((pool, 64, Hkv, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    vc = torch.full_like(kc, float("nan"))
    std = 1 / math.sqrt(d)
    ks, vs = [], []
    for b in range(B):
        k = _gen((CTX[b], Hkv, d), 10 + b, std)
        v = _gen((CTX[b], Hkv, d), 500 + b, std)
        ks.append(k)
        vs.append(v)
        vpp.vpp_kv_append(k.to(DEV), v.to(DEV), kc, vc, 0,
                          block_table=torch.from_numpy(table[b].copy()).to(DEV))
    q = _gen((B, Hq, d), 999, std)
    lse = torch.empty((Hq, B), dtype=torch.float32, device=DEV)
    out = vpp.vpp_mixed_attn(q.to(DEV), kc, vc, torch.from_numpy(table).to(DEV), cu, ctx, lse=lse)
    torch.cuda.synchronize()
    assert vpp.vpp_last_device_status() == 0
    ref, ref_lse = oracle.mixed_batch_attention(to_np64(q), [to_np64(x) for x in ks],
                                                [to_np64(x) for x in vs], cu, ctx)
    assert_close(to_np64(out), ref)
    assert np.abs(to_np64(lse) - ref_lse).max() <= LSE_ABS


def test_decode_workspace_is_sized_and_required():
    Hq, Hkv, d = 32, 8, 128
    cu = np.array([0, 1, 2], dtype=np.int32)
    ctx = np.array([5000, 300], dtype=np.int32)
    ws = vpp.mixed_attn_workspace_size(cu, ctx, Hq, Hkv, d, d)
    items = math.ceil(5000 / 1024) + 1
    assert ws >= items * Hq * (d + 1) * 4
    short = np.array([1000, 300], dtype=np.int32)
    assert vpp.mixed_attn_workspace_size(cu, short, Hq, Hkv, d, d) == 0
