"""The allocation-free chunk-attention entry point against the workspace one.

vpp_chunk_attn_noalloc serves callers that may not allocate device memory on
their execution path and have no scratch buffer to pass: it keeps the split
partials in the library's fixed 32 MiB device array.  Its results must match
vpp_chunk_attn_ex (caller workspace) within the parity tolerance, on two calls
in a row that reuse the shared array, and it must refuse calls whose partials
do not fit.  This file is collected last so that a run stopping at the first
failure has already run every other test.
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


def _inputs(Hq, Hkv, d, P, C, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    std = 1 / math.sqrt(d)
    q = (torch.randn((C, Hq, d), generator=g) * std).to(torch.bfloat16)
    k = (torch.randn((P + C, Hkv, d), generator=g) * std).to(torch.bfloat16)
    v = (torch.randn((P + C, Hkv, d), generator=g) * std).to(torch.bfloat16)
    return q, k, v


def _case(Hq, Hkv, d, P, C, seed, host=False):
    q, k, v = _inputs(Hq, Hkv, d, P, C, seed)
    need = (P + C + 63) // 64
    table = torch.from_numpy(random_table(need, need + 3, seed)).to(DEV)
    kc = torch.zeros((need + 3, 64, Hkv, d), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    vpp.vpp_kv_append(k.to(DEV), v.to(DEV), kc, vc, 0, block_table=table)
    if host:
        return q.to(DEV), kc, vc, table, (q, k, v)
    return q.to(DEV), kc, vc, table


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    cases = [(16, 4, 128, 3000, 100, 3, 11), (8, 2, 128, 900, 257, 2, 12)]
    for Hq, Hkv, d, P, C, splits, seed in cases:
        q, kc, vc, table = _case(Hq, Hkv, d, P, C, seed)
        assert vpp.chunk_attn_num_splits(P, C, Hq, Hkv, d, d, splits) == splits
        lse_a = torch.empty((Hq, C), dtype=torch.float32, device=DEV)
        lse_b = torch.empty((Hq, C), dtype=torch.float32, device=DEV)
        ref = vpp.vpp_chunk_attn_ex(q, kc, vc, P, block_table=table, lse=lse_a, num_splits=splits)
        got = vpp.vpp_chunk_attn_noalloc(q, kc, vc, P, block_table=table, lse=lse_b, num_splits=splits)
        torch.cuda.synchronize()
        assert vpp.vpp_last_device_status() == 0
        ma, rl = errors(to_np64(got), to_np64(ref))
        assert np.all(np.isfinite(to_np64(got)))
        assert ma <= 2e-2 and rl <= 5e-3, (ma, rl)
        assert np.abs(to_np64(lse_b) - to_np64(lse_a)).max() <= LSE_ABS


def test_noalloc_refuses_partials_larger_than_its_array():
    Hq, Hkv, d, P, C = 32, 8, 128, 8192, 4096
    q, kc, vc, table = _case(Hq, Hkv, d, P, C, 13)
    # 2 ranges x 4096 tokens x 32 heads x (128 + 1) x 4 bytes > 32 MiB
    with pytest.raises(vpp.VppError) as e:
        vpp.vpp_chunk_attn_noalloc(q, kc, vc, P, block_table=table, num_splits=2)
    assert e.value.code == vpp.VPP_ERR_WORKSPACE


def test_noalloc_matches_the_oracle_unsplit_split_and_library_chosen():
    # One range (no scratch used), an explicit split, and the library's own
    # choice, each against the fp64 oracle on the same inputs.
    Hq, Hkv, d, P, C = 16, 4, 128, 1500, 300
    q, kc, vc, table, (qh, kh, vh) = _case(Hq, Hkv, d, P, C, 21, host=True)
    ref, ref_lse = oracle.causal_chunk_attention(to_np64(qh), to_np64(kh), to_np64(vh), P)
    for splits in (1, 2, 0):
        lse = torch.empty((Hq, C), dtype=torch.float32, device=DEV)
        got = vpp.vpp_chunk_attn_noalloc(q, kc, vc, P, block_table=table, lse=lse, num_splits=splits)
        torch.cuda.synchronize()
        assert vpp.vpp_last_device_status() == 0
        assert_close(to_np64(got), ref, what=f"noalloc num_splits={splits}")
        assert np.abs(to_np64(lse) - ref_lse).max() <= LSE_ABS


def test_noalloc_lowers_the_library_split_choice_to_fit_its_array():
    # In both shapes the library would split the prefix for speed into ranges
    # whose partials exceed 32 MiB.  The call then takes the largest range
    # count that fits (three ranges in the first shape, none in the second)
    # instead of refusing, and its result is bit for bit the workspace entry
    # point's with that count.
    limit = 32 << 20
    Hq, Hkv, d = 32, 8, 128
    for P, C, expect, seed in ((40000, 512, 3, 22), (60000, 2048, 1, 23)):
        auto = vpp.chunk_attn_num_splits(P, C, Hq, Hkv, d, d, 0)
        assert vpp.chunk_attn_workspace_size(vpp.VPP_BF16, P, C, Hq, Hkv, d, d, 0) > limit
        fit = max(s for s in range(1, auto + 1)
                  if vpp.chunk_attn_workspace_size(vpp.VPP_BF16, P, C, Hq, Hkv, d, d, s) <= limit)
        assert fit == expect
        q, kc, vc, table = _case(Hq, Hkv, d, P, C, seed)
        lse_a = torch.empty((Hq, C), dtype=torch.float32, device=DEV)
        lse_b = torch.empty((Hq, C), dtype=torch.float32, device=DEV)
        ref = vpp.vpp_chunk_attn_ex(q, kc, vc, P, block_table=table, lse=lse_a, num_splits=fit)
        got = vpp.vpp_chunk_attn_noalloc(q, kc, vc, P, block_table=table, lse=lse_b, num_splits=0)
        torch.cuda.synchronize()
        assert vpp.vpp_last_device_status() == 0
        assert torch.equal(got, ref)
        assert torch.equal(lse_b, lse_a)


def test_noalloc_runs_the_library_heavy_tile_plan():
    # The library's own plan for this shape splits only the keys of the tokens
    # from 1152 on (3 ranges, 19 MB of partials): the allocation-free call runs
    # that same plan in its array and matches the workspace entry point bit
    # for bit, and both match the oracle.
    Hq, Hkv, d, P, C = 32, 8, 128, 4096, 1536
    assert vpp.chunk_attn_plan(P, C, Hq, Hkv, d, d) == (3, 1152)
    q, kc, vc, table, (qh, kh, vh) = _case(Hq, Hkv, d, P, C, 24, host=True)
    lse_a = torch.empty((Hq, C), dtype=torch.float32, device=DEV)
    lse_b = torch.empty((Hq, C), dtype=torch.float32, device=DEV)
    ref = vpp.vpp_chunk_attn_ex(q, kc, vc, P, block_table=table, lse=lse_a)
    got = vpp.vpp_chunk_attn_noalloc(q, kc, vc, P, block_table=table, lse=lse_b)
    torch.cuda.synchronize()
    assert vpp.vpp_last_device_status() == 0
    assert torch.equal(got, ref) and torch.equal(lse_b, lse_a)
    want, want_lse = oracle.causal_chunk_attention(to_np64(qh), to_np64(kh), to_np64(vh), P)
    assert_close(to_np64(got), want)
    assert np.abs(to_np64(lse_b) - want_lse).max() <= LSE_ABS
