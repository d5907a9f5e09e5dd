"""The C ABI library loads, exports every symbol include/vpp.h declares, and
rejects bad arguments on the host before touching a device (runs on CPU)."""

import ctypes
import os
import re

import numpy as np
import pytest

from chunked_prefill_causal_gb300 import vpp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "vpp.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return vpp.load()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(vpp_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_symbols()
    for n in ("vpp_kv_append", "vpp_chunk_attn", "vpp_chunk_attn_ex", "vpp_mixed_attn",
              "vpp_last_device_status"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_symbols() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(declared_symbols()) <= set(vpp.SIGNATURES)


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5):
        assert vpp.status_string(code)
    assert "unknown" in vpp.status_string(42)
    assert lib.vpp_version() >= 100


def test_host_validation_rejects_bad_arguments(lib):
    null = None
    fake = ctypes.c_void_p(0x100000)  # never dereferenced: validation fails first
    # null tensors
    assert lib.vpp_chunk_attn(null, fake, fake, 0, 16, 8, 2, 128, fake, null, null) == vpp.VPP_ERR_INVALID
    # unsupported head dim / grouping
    assert lib.vpp_chunk_attn(fake, fake, fake, 0, 16, 8, 2, 96, fake, null, null) == vpp.VPP_ERR_UNSUPPORTED
    assert lib.vpp_chunk_attn(fake, fake, fake, 0, 16, 24, 8, 128, fake, null, null) == vpp.VPP_ERR_UNSUPPORTED
    assert lib.vpp_chunk_attn(fake, fake, fake, 0, 16, 7, 2, 128, fake, null, null) == vpp.VPP_ERR_INVALID
    # misaligned pointer
    bad = ctypes.c_void_p(0x100004)
    assert lib.vpp_chunk_attn(bad, fake, fake, 0, 16, 8, 2, 128, fake, null, null) == vpp.VPP_ERR_INVALID
    # negative lengths
    assert lib.vpp_chunk_attn(fake, fake, fake, -1, 16, 8, 2, 128, fake, null, null) == vpp.VPP_ERR_INVALID
    # cache too small for prefix + chunk (paged: 2 blocks = 128 tokens)
    assert lib.vpp_chunk_attn_ex(fake, 0, fake, fake, fake, 2, 100, 29, 8, 2, 128, 128, 0.0, 0, fake,
                                 null, null, 0, null) == vpp.VPP_ERR_INVALID
    assert lib.vpp_kv_append(fake, fake, 0, fake, fake, fake, 2, 100, 29, 2, 128, 128, null) == vpp.VPP_ERR_INVALID
    assert lib.vpp_kv_append(fake, fake, 7, fake, fake, fake, 2, 0, 29, 2, 128, 128, null) == vpp.VPP_ERR_INVALID
    # varlen: cu_seqlens must start at 0 and ctx >= q_len
    cu = (ctypes.c_int32 * 3)(0, 5, 9)
    ctx = (ctypes.c_int32 * 2)(4, 10)
    assert lib.vpp_mixed_attn(fake, fake, fake, fake, 4, 16, cu, ctx, 2, 8, 2, 128, 128, 0.0, fake, null,
                              null, 0, null) == vpp.VPP_ERR_INVALID
    # at most 1024 sequences per mixed batch (the plan travels by value)
    n = 1025
    cu_big = (ctypes.c_int32 * (n + 1))(*range(n + 1))
    ctx_big = (ctypes.c_int32 * n)(*([1] * n))
    assert lib.vpp_mixed_attn(fake, fake, fake, fake, 4, 16, cu_big, ctx_big, n, 8, 2, 128, 128, 0.0, fake, null,
                              null, 0, null) == vpp.VPP_ERR_INVALID
    assert lib.vpp_kv_append_varlen(fake, fake, fake, fake, fake, 4, 16, cu_big, ctx_big, n, 2, 128, 128,
                                    null) == vpp.VPP_ERR_INVALID
    assert lib.vpp_selftest_wait_timeout(0, null) == vpp.VPP_ERR_INVALID
    # fp8 cache: scales are required and 4-byte aligned
    assert lib.vpp_kv_append_fp8(fake, fake, fake, fake, null, fake, fake, 2, 0, 29, 2, 128, 128,
                                 null) == vpp.VPP_ERR_INVALID
    assert lib.vpp_kv_append_fp8(fake, fake, fake, fake, bad, ctypes.c_void_p(0x100002), fake, 2, 0, 29, 2,
                                 128, 128, null) == vpp.VPP_ERR_INVALID
    assert lib.vpp_kv_append_fp8(fake, fake, fake, fake, fake, fake, fake, 2, 0, 29, 2, 96, 128,
                                 null) == vpp.VPP_ERR_UNSUPPORTED
    assert lib.vpp_chunk_attn_fp8(fake, fake, fake, null, fake, fake, 2, 0, 29, 8, 2, 128, 128, 0.0, 0,
                                  fake, null, fake, 1 << 30, null) == vpp.VPP_ERR_INVALID
    # fp8 chunk attention: an empty chunk is a no-op; unsupported dims are refused on the host
    assert lib.vpp_chunk_attn_fp8(null, null, null, null, null, null, 2, 0, 0, 8, 2, 128, 128, 0.0, 0,
                                  null, null, null, 0, null) == vpp.VPP_OK
    assert lib.vpp_chunk_attn_fp8(fake, fake, fake, fake, fake, fake, 2, 0, 29, 8, 2, 96, 96, 0.0, 0,
                                  fake, null, null, 0, null) == vpp.VPP_ERR_UNSUPPORTED
    assert lib.vpp_mixed_attn_fp8(fake, fake, fake, fake, null, fake, 4, 16, cu, ctx, 2, 8, 2, 128, 128,
                                  0.0, fake, null, null, 0, null) == vpp.VPP_ERR_INVALID


def test_topk_validation_and_workspace(lib):
    null = None
    fake = ctypes.c_void_p(0x100000)
    # no index list / unsupported shape (16 query heads per kv head) / bad topk
    assert lib.vpp_topk_chunk_attn(fake, fake, fake, fake, 64, 0, 16, null, fake, 2048, 8, 2, 128, 0.0, fake,
                                   null, null, 0, null) == vpp.VPP_ERR_INVALID
    assert lib.vpp_topk_chunk_attn(fake, fake, fake, fake, 64, 0, 16, fake, fake, 2048, 128, 8, 128, 0.0, fake,
                                   null, null, 0, null) == vpp.VPP_ERR_UNSUPPORTED
    assert lib.vpp_topk_chunk_attn(fake, fake, fake, fake, 64, 0, 16, fake, fake, 0, 8, 2, 128, 0.0, fake,
                                   null, null, 0, null) == vpp.VPP_ERR_INVALID
    # more than 1024 entries per list: key-range partials need a workspace
    assert lib.vpp_topk_chunk_attn(fake, fake, fake, fake, 64, 0, 16, fake, fake, 2048, 8, 2, 128, 0.0, fake,
                                   null, null, 0, null) == vpp.VPP_ERR_WORKSPACE
    assert vpp.topk_chunk_attn_workspace_size(16, 1024, 8, 128) == 0
    assert vpp.topk_chunk_attn_workspace_size(16, 2048, 8, 128) == 16 * 2 * 8 * 128 * 4 + 16 * 2 * 8 * 4
    assert lib.vpp_topk_chunk_attn_fp8(fake, fake, fake, null, fake, fake, 64, 0, 16, fake, fake, 1024, 8, 2, 128,
                                       0.0, fake, null, null, 0, null) == vpp.VPP_ERR_INVALID


def test_split_plan_is_host_side(lib):
    # No device needed: the planner falls back to 152 SMs for its model.
    assert vpp.chunk_attn_num_splits(0, 4096, 32, 8, 128, 128) == 1
    assert vpp.chunk_attn_num_splits(7 * 16384, 16384, 64, 8, 128, 128) == 1
    assert vpp.chunk_attn_num_splits(100000, 64, 8, 8, 128, 128, num_splits=4) == 4
    assert vpp.chunk_attn_num_splits(300, 64, 8, 8, 128, 128, num_splits=8) <= 3
    assert vpp.chunk_attn_num_splits(100000, 64, 8, 8, 128, 128, num_splits=1) == 1
    ws = vpp.chunk_attn_workspace_size(vpp.VPP_BF16, 100000, 64, 8, 8, 128, 128, 4)
    assert ws >= 4 * 64 * 8 * 128 * 4
    assert vpp.chunk_attn_workspace_size(vpp.VPP_BF16, 100000, 64, 8, 8, 128, 128, 1) == 0
    assert vpp.chunk_attn_workspace_size(vpp.VPP_FP32, 0, 64, 8, 8, 128, 128, 1) == 64 * 8 * 128 * 2


def test_plan_splits_heavy_query_tiles_only(lib):
    """The library's own plan for a gqa32k chunk (32/8 heads, C 4096, 512
    unsplit CTAs = 3.4 waves of 152) splits the keys of the heaviest query
    tiles only; an explicit request splits every token.  The workspace holds
    exactly the split group's float32 partials and LSEs, each part rounded to
    256 bytes."""
    def r256(x):
        return (x + 255) // 256 * 256
    H, Hkv, d, C = 32, 8, 128, 4096
    assert vpp.chunk_attn_plan(0, C, H, Hkv, d, d) == (1, 0)
    for k in range(3, 8):
        S, t0 = vpp.chunk_attn_plan(k * C, C, H, Hkv, d, d)
        assert S >= 2 and 0 < t0 < C and t0 % 64 == 0
        rows = S * (C - t0)
        want = r256(rows * H * d * 4) + r256(rows * H * 4)
        assert vpp.chunk_attn_workspace_size(vpp.VPP_BF16, k * C, C, H, Hkv, d, d) == want
        assert vpp.chunk_attn_num_splits(k * C, C, H, Hkv, d, d) == S
    assert vpp.chunk_attn_plan(5 * C, C, H, Hkv, d, d, num_splits=4) == (4, 0)
    assert vpp.chunk_attn_workspace_size(vpp.VPP_BF16, 5 * C, C, H, Hkv, d, d, 4) == \
        r256(4 * C * H * d * 4) + r256(4 * C * H * 4)
    # many waves of CTAs (long128k: 4096 per chunk) are never split
    assert vpp.chunk_attn_plan(7 * 16384, 16384, 64, 8, d, d) == (1, 0)
    with pytest.raises(vpp.VppError):
        vpp.chunk_attn_plan(0, C, 32, 5, d, d)


def test_noalloc_host_checks_run_before_any_device_call(lib):
    null = None
    fake = ctypes.c_void_p(0x100000)  # never dereferenced
    f = lib.vpp_chunk_attn_noalloc
    # an empty chunk is a no-op, even with NULL tensors
    assert f(null, null, null, null, 1, 100, 0, 8, 2, 128, 128, ctypes.c_float(0.0), 0, null, null, null) == vpp.VPP_OK
    # unsupported head dims and groupings
    assert f(fake, fake, fake, null, 256, 100, 16, 8, 2, 96, 96, ctypes.c_float(0.0), 0, fake, null, null) == \
        vpp.VPP_ERR_UNSUPPORTED
    assert f(fake, fake, fake, null, 256, 100, 16, 8, 2, 128, 192, ctypes.c_float(0.0), 0, fake, null, null) == \
        vpp.VPP_ERR_UNSUPPORTED
    assert f(fake, fake, fake, null, 256, 100, 16, 24, 8, 128, 128, ctypes.c_float(0.0), 0, fake, null, null) == \
        vpp.VPP_ERR_UNSUPPORTED
    # negative sizes and split requests
    assert f(fake, fake, fake, null, 256, -1, 16, 8, 2, 128, 128, ctypes.c_float(0.0), 0, fake, null, null) == \
        vpp.VPP_ERR_INVALID
    assert f(fake, fake, fake, null, 256, 100, 16, 8, 2, 128, 128, ctypes.c_float(0.0), -1, fake, null, null) == \
        vpp.VPP_ERR_INVALID


def test_fp8_workspace_does_not_grow_with_the_prefix(lib):
    # The fp8 kernels widen the codes themselves: the workspace holds only
    # key-split partials, whose size depends on the chunk, not on the prefix.
    from chunked_prefill_causal_gb300 import vpp as v
    C, H, Hkv, d = 4096, 32, 8, 128
    assert v.chunk_attn_fp8_workspace_size(100000, C, H, Hkv, d, d, 1) == 0
    a = v.chunk_attn_fp8_workspace_size(8192, C, H, Hkv, d, d, 2)
    b = v.chunk_attn_fp8_workspace_size(500000, C, H, Hkv, d, d, 2)
    assert a == b == v.chunk_attn_workspace_size(v.VPP_BF16, 8192, C, H, Hkv, d, d, 2) > 0
    cu = np.array([0, 2048, 2049], dtype=np.int32)
    for ctx in ([2048 + 16384, 900], [2048 + 122880, 900]):
        assert v.mixed_attn_fp8_workspace_size(cu, np.array(ctx, dtype=np.int32), H, Hkv, d, d) == \
            v.mixed_attn_workspace_size(cu, np.array(ctx, dtype=np.int32), H, Hkv, d, d) == 0
        # the optional bf16 copy of the prefill sequence's context does grow with it
        assert v.mixed_attn_fp8_widen_workspace_size(cu, np.array(ctx, dtype=np.int32), H, Hkv, d, d) == \
            2 * ((ctx[0] * Hkv * d * 2 + 255) // 256 * 256)
    n = 8192 + C
    assert v.chunk_attn_fp8_widen_workspace_size(8192, C, H, Hkv, d, d, 2) == \
        2 * ((n * Hkv * d * 2 + 255) // 256 * 256) + a
