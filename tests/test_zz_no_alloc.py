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

from chunked_prefill_causal_gb300 import vpp
from tests.helpers import LSE_ABS, errors, random_table, to_np64

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _case(Hq, Hkv, d, P, C, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    std = 1 / math.sqrt(d)
    q = (torch.randn((C, Hq, d), generator=g) * std).to(torch.bfloat16).to(DEV)
    k = (torch.randn((P + C, Hkv, d), generator=g) * std).to(torch.bfloat16).to(DEV)
    v = (torch.randn((P + C, Hkv, d), generator=g) * std).to(torch.bfloat16).to(DEV)
    need = (P + C + 63) // 64
    table = torch.from_numpy(random_table(need, need + 3, seed)).to(DEV)
    kc = torch.zeros((need + 3, 64, Hkv, d), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    vpp.vpp_kv_append(k, v, kc, vc, 0, block_table=table)
    return q, kc, vc, table


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
