"""Thin ctypes binding of libvpp.so (declared in include/vpp.h).

Argument marshalling only: every function takes torch CUDA tensors, checks
their dtype/shape/contiguity, passes raw pointers and the current stream to
the C ABI, and raises VppError on a non-zero status.  All computation runs
in the library's CUDA kernels; there is no CPU fallback.
"""

from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libvpp.so")

VPP_OK, VPP_ERR_INVALID, VPP_ERR_UNSUPPORTED, VPP_ERR_CUDA, VPP_ERR_TIMEOUT, VPP_ERR_WORKSPACE = (
    0, -1, -2, -3, -4, -5)
VPP_BF16, VPP_FP32 = 0, 1

# Every exported symbol of include/vpp.h with its C signature.
_c_void_p, _i32, _i64, _f32, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
_int = ctypes.c_int
SIGNATURES = {
    "vpp_status_string": ([_int], ctypes.c_char_p),
    "vpp_version": ([], _int),
    "vpp_kv_append": ([_c_void_p, _c_void_p, _int, _c_void_p, _c_void_p, _c_void_p, _i32, _i64, _i64,
                       _int, _int, _int, _c_void_p], _int),
    "vpp_chunk_attn": ([_c_void_p, _c_void_p, _c_void_p, _i64, _i64, _int, _int, _int, _c_void_p,
                        _c_void_p, _c_void_p], _int),
    "vpp_chunk_attn_ex": ([_c_void_p, _int, _c_void_p, _c_void_p, _c_void_p, _i32, _i64, _i64, _int,
                           _int, _int, _int, _f32, _int, _c_void_p, _c_void_p, _c_void_p, _sz,
                           _c_void_p], _int),
    "vpp_chunk_attn_noalloc": ([_c_void_p, _c_void_p, _c_void_p, _c_void_p, _i32, _i64, _i64, _int, _int,
                                _int, _int, _f32, _int, _c_void_p, _c_void_p, _c_void_p], _int),
    "vpp_chunk_attn_workspace_size": ([_int, _i64, _i64, _int, _int, _int, _int, _int], _sz),
    "vpp_chunk_attn_num_splits": ([_i64, _i64, _int, _int, _int, _int, _int], _int),
    "vpp_chunk_attn_plan": ([_i64, _i64, _int, _int, _int, _int, _int, ctypes.POINTER(_i64)], _int),
    "vpp_mixed_attn": ([_c_void_p, _c_void_p, _c_void_p, _c_void_p, _i32, _i32, _c_void_p, _c_void_p,
                        _i32, _int, _int, _int, _int, _f32, _c_void_p, _c_void_p, _c_void_p, _sz,
                        _c_void_p], _int),
    "vpp_mixed_attn_workspace_size": ([_c_void_p, _c_void_p, _i32, _int, _int, _int, _int], _sz),
    "vpp_kv_append_varlen": ([_c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _i32, _i32,
                              _c_void_p, _c_void_p, _i32, _int, _int, _int, _c_void_p], _int),
    "vpp_kv_append_fp8": ([_c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _i32,
                           _i64, _i64, _int, _int, _int, _c_void_p], _int),
    "vpp_kv_append_varlen_fp8": ([_c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                  _i32, _i32, _c_void_p, _c_void_p, _i32, _int, _int, _int, _c_void_p], _int),
    "vpp_chunk_attn_fp8": ([_c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _i32, _i64, _i64,
                            _int, _int, _int, _int, _f32, _int, _c_void_p, _c_void_p, _c_void_p, _sz,
                            _c_void_p], _int),
    "vpp_chunk_attn_fp8_workspace_size": ([_i64, _i64, _int, _int, _int, _int, _int], _sz),
    "vpp_chunk_attn_fp8_widen_workspace_size": ([_i64, _i64, _int, _int, _int, _int, _int], _sz),
    "vpp_mixed_attn_fp8": ([_c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _i32, _i32,
                            _c_void_p, _c_void_p, _i32, _int, _int, _int, _int, _f32, _c_void_p, _c_void_p,
                            _c_void_p, _sz, _c_void_p], _int),
    "vpp_mixed_attn_fp8_workspace_size": ([_c_void_p, _c_void_p, _i32, _int, _int, _int, _int], _sz),
    "vpp_mixed_attn_fp8_widen_workspace_size": ([_c_void_p, _c_void_p, _i32, _int, _int, _int, _int], _sz),
    "vpp_topk_chunk_attn": ([_c_void_p, _c_void_p, _c_void_p, _c_void_p, _i32, _i64, _i64, _c_void_p, _c_void_p,
                             _i32, _int, _int, _int, _f32, _c_void_p, _c_void_p, _c_void_p, _sz, _c_void_p], _int),
    "vpp_topk_chunk_attn_fp8": ([_c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _i32, _i64,
                                 _i64, _c_void_p, _c_void_p, _i32, _int, _int, _int, _f32, _c_void_p, _c_void_p,
                                 _c_void_p, _sz, _c_void_p], _int),
    "vpp_topk_chunk_attn_workspace_size": ([_i64, _i32, _int, _int], _sz),
    "vpp_last_device_status": ([_c_void_p, ctypes.POINTER(_int)], _int),
    "vpp_selftest_wait_timeout": ([_int, _c_void_p], _int),
}


class VppError(RuntimeError):
    def __init__(self, fn, code):
        self.code = code
        super().__init__(f"{fn} failed: {status_string(code)} ({code})")


_lib = None


def load(path: str | None = None):
    """Loads libvpp.so (raises if it was not built)."""
    global _lib
    if _lib is None:
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"libvpp.so not found at {p}: run __graft_entry__.build() first")
        lib = ctypes.CDLL(p)
        for name, (args, res) in SIGNATURES.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = res
        _lib = lib
    return _lib


def status_string(code: int) -> str:
    return load().vpp_status_string(int(code)).decode()


def _check(fn, code):
    if code != VPP_OK:
        raise VppError(fn, code)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return VPP_BF16
    if t.dtype == torch.float32:
        return VPP_FP32
    raise ValueError(f"unsupported dtype {t.dtype}")


def _i32_host(a):
    import numpy as np
    arr = np.ascontiguousarray(a, dtype=np.int32)
    return arr, arr.ctypes.data_as(ctypes.c_void_p)


# ----------------------------------------------------------------- a1
def vpp_kv_append(k_new, v_new, k_cache, v_cache, prefix_len, block_table=None, stream=None):
    """Append a chunk's K/V ([C, Hkv, d], bf16 or fp32) to a bf16 cache.

    Paged cache [num_blocks, 64, Hkv, d] with block_table (int32 CUDA tensor),
    or contiguous [capacity, Hkv, d] with block_table None.
    """
    _need_cuda(k_new, v_new, k_cache, v_cache, block_table)
    if k_cache.dtype != torch.bfloat16 or v_cache.dtype != torch.bfloat16:
        raise ValueError("cache must be bf16")
    C, Hkv, dq = k_new.shape
    dv = v_new.shape[2]
    nb = k_cache.shape[0]
    _check("vpp_kv_append", load().vpp_kv_append(
        _ptr(k_new), _ptr(v_new), _dtype_code(k_new), _ptr(k_cache), _ptr(v_cache),
        _ptr(block_table), nb, int(prefix_len), C, Hkv, dq, dv, _stream(stream)))


def vpp_kv_append_varlen(k_new, v_new, k_cache, v_cache, block_table, cu_seqlens_q, ctx_lens,
                         stream=None):
    """Varlen append: packed new K/V rows go to the last q_len_b positions of
    each sequence b (host cu_seqlens_q / ctx_lens, device block_table [B, maxb])."""
    _need_cuda(k_new, v_new, k_cache, v_cache, block_table)
    _, Hkv, dq = k_new.shape
    dv = v_new.shape[2]
    cu, cu_p = _i32_host(cu_seqlens_q)
    ctx, ctx_p = _i32_host(ctx_lens)
    _check("vpp_kv_append_varlen", load().vpp_kv_append_varlen(
        _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
        block_table.shape[1], k_cache.shape[0], cu_p, ctx_p, len(ctx), Hkv, dq, dv,
        _stream(stream)))


# ----------------------------------------------------------------- a2..a7
def vpp_chunk_attn(q, k_cache, v_cache, prefix_len, out=None, lse=None, stream=None):
    """Plain form: contiguous bf16 cache [P + C, Hkv, d], dq = dv, no splitting."""
    _need_cuda(q, k_cache, v_cache, out, lse)
    C, H, d = q.shape
    Hkv = k_cache.shape[1]
    if out is None:
        out = torch.empty((C, H, d), dtype=torch.bfloat16, device=q.device)
    _check("vpp_chunk_attn", load().vpp_chunk_attn(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), int(prefix_len), C, H, Hkv, d, _ptr(out), _ptr(lse),
        _stream(stream)))
    return out


def chunk_attn_workspace_size(q_dtype, prefix_len, chunk_len, heads, kv_heads, dq, dv, num_splits=0):
    return int(load().vpp_chunk_attn_workspace_size(q_dtype, int(prefix_len), int(chunk_len), heads,
                                                    kv_heads, dq, dv, num_splits))


def chunk_attn_num_splits(prefix_len, chunk_len, heads, kv_heads, dq, dv, num_splits=0):
    return int(load().vpp_chunk_attn_num_splits(int(prefix_len), int(chunk_len), heads, kv_heads,
                                                dq, dv, num_splits))


def chunk_attn_plan(prefix_len, chunk_len, heads, kv_heads, dq, dv, num_splits=0):
    """(key ranges S, first query token whose keys are split) of the plan
    vpp_chunk_attn_ex uses; raises on an invalid shape."""
    t0 = _i64(0)
    s = int(load().vpp_chunk_attn_plan(int(prefix_len), int(chunk_len), heads, kv_heads, dq, dv, num_splits,
                                       ctypes.byref(t0)))
    _check("vpp_chunk_attn_plan", VPP_OK if s >= 1 else s)
    return s, int(t0.value)


def vpp_chunk_attn_ex(q, k_cache, v_cache, prefix_len, block_table=None, out=None, lse=None,
                      softmax_scale=0.0, num_splits=0, workspace=None, stream=None):
    """Full form: paged or contiguous cache, fp32 or bf16 q, key splitting."""
    _need_cuda(q, k_cache, v_cache, block_table, out, lse, workspace)
    C, H, dq = q.shape
    Hkv = k_cache.shape[-2]
    dv = v_cache.shape[-1]
    qd = _dtype_code(q)
    if block_table is not None:
        nb = k_cache.shape[0]
    else:
        nb = k_cache.shape[0]  # contiguous: capacity in tokens
    if out is None:
        out = torch.empty((C, H, dv), dtype=torch.bfloat16, device=q.device)
    need = chunk_attn_workspace_size(qd, prefix_len, C, H, Hkv, dq, dv, num_splits)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("vpp_chunk_attn_ex", load().vpp_chunk_attn_ex(
        _ptr(q), qd, _ptr(k_cache), _ptr(v_cache), _ptr(block_table), nb, int(prefix_len), C, H, Hkv,
        dq, dv, float(softmax_scale), int(num_splits), _ptr(out), _ptr(lse), _ptr(workspace), wbytes,
        _stream(stream)))
    return out


def vpp_chunk_attn_noalloc(q, k_cache, v_cache, prefix_len, block_table=None, out=None, lse=None,
                           softmax_scale=0.0, num_splits=0, stream=None):
    """Chunk attention whose key-split partials use the library's fixed 32 MiB
    device array instead of a workspace (for callers that cannot allocate);
    bf16 q only.  Calls on one device must not overlap on the GPU."""
    _need_cuda(q, k_cache, v_cache, block_table, out, lse)
    C, H, dq = q.shape
    Hkv = k_cache.shape[-2]
    dv = v_cache.shape[-1]
    if q.dtype != torch.bfloat16:
        raise ValueError("vpp_chunk_attn_noalloc takes bf16 q")
    if out is None:
        out = torch.empty((C, H, dv), dtype=torch.bfloat16, device=q.device)
    _check("vpp_chunk_attn_noalloc", load().vpp_chunk_attn_noalloc(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), k_cache.shape[0], int(prefix_len), C, H,
        Hkv, dq, dv, float(softmax_scale), int(num_splits), _ptr(out), _ptr(lse), _stream(stream)))
    return out


# ----------------------------------------------------------------- a8..a9
def mixed_attn_workspace_size(cu_seqlens_q, ctx_lens, heads, kv_heads, dq, dv):
    cu, cu_p = _i32_host(cu_seqlens_q)
    ctx, ctx_p = _i32_host(ctx_lens)
    return int(load().vpp_mixed_attn_workspace_size(cu_p, ctx_p, len(ctx), heads, kv_heads, dq, dv))


def vpp_mixed_attn(q, k_cache, v_cache, block_table, cu_seqlens_q, ctx_lens, out=None, lse=None,
                   softmax_scale=0.0, workspace=None, stream=None):
    """Mixed micro-batch over a paged cache (host cu_seqlens_q / ctx_lens)."""
    _need_cuda(q, k_cache, v_cache, block_table, out, lse, workspace)
    T, H, dq = q.shape
    Hkv = k_cache.shape[2]
    dv = v_cache.shape[3]
    cu, cu_p = _i32_host(cu_seqlens_q)
    ctx, ctx_p = _i32_host(ctx_lens)
    if out is None:
        out = torch.empty((T, H, dv), dtype=torch.bfloat16, device=q.device)
    need = mixed_attn_workspace_size(cu, ctx, H, Hkv, dq, dv)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("vpp_mixed_attn", load().vpp_mixed_attn(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
        k_cache.shape[0], cu_p, ctx_p, len(ctx), H, Hkv, dq, dv, float(softmax_scale), _ptr(out),
        _ptr(lse), _ptr(workspace), wbytes, _stream(stream)))
    return out


# ----------------------------------------------------------------- fp8 (E4M3) KV cache
def _fp8_cache(*caches):
    for c in caches:
        if c.dtype != torch.uint8:
            raise ValueError("fp8 caches hold E4M3 codes as uint8")


def _scales(k_scale, v_scale, kv_heads):
    _need_cuda(k_scale, v_scale)
    for s in (k_scale, v_scale):
        if s.dtype != torch.float32 or s.numel() != kv_heads:
            raise ValueError("scales are float32 CUDA tensors with one entry per kv head")


def vpp_kv_append_fp8(k_new, v_new, k_cache, v_cache, k_scale, v_scale, prefix_len, block_table=None,
                      stream=None):
    """Quantise a chunk's bf16 K/V ([C, Hkv, d]) into an E4M3 cache (uint8),
    one float32 scale per kv head (code = E4M3(fl32(x / scale)))."""
    _need_cuda(k_new, v_new, k_cache, v_cache, block_table)
    _fp8_cache(k_cache, v_cache)
    if k_new.dtype != torch.bfloat16 or v_new.dtype != torch.bfloat16:
        raise ValueError("fp8 append takes bf16 K/V")
    C, Hkv, dq = k_new.shape
    dv = v_new.shape[2]
    _scales(k_scale, v_scale, Hkv)
    _check("vpp_kv_append_fp8", load().vpp_kv_append_fp8(
        _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
        _ptr(block_table), k_cache.shape[0], int(prefix_len), C, Hkv, dq, dv, _stream(stream)))


def vpp_kv_append_varlen_fp8(k_new, v_new, k_cache, v_cache, k_scale, v_scale, block_table, cu_seqlens_q,
                             ctx_lens, stream=None):
    """Varlen append into an E4M3 paged cache (see vpp_kv_append_varlen)."""
    _need_cuda(k_new, v_new, k_cache, v_cache, block_table)
    _fp8_cache(k_cache, v_cache)
    _, Hkv, dq = k_new.shape
    dv = v_new.shape[2]
    _scales(k_scale, v_scale, Hkv)
    cu, cu_p = _i32_host(cu_seqlens_q)
    ctx, ctx_p = _i32_host(ctx_lens)
    _check("vpp_kv_append_varlen_fp8", load().vpp_kv_append_varlen_fp8(
        _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
        _ptr(block_table), block_table.shape[1], k_cache.shape[0], cu_p, ctx_p, len(ctx), Hkv, dq, dv,
        _stream(stream)))


def chunk_attn_fp8_workspace_size(prefix_len, chunk_len, heads, kv_heads, dq, dv, num_splits=0):
    return int(load().vpp_chunk_attn_fp8_workspace_size(int(prefix_len), int(chunk_len), heads, kv_heads,
                                                        dq, dv, num_splits))


def chunk_attn_fp8_widen_workspace_size(prefix_len, chunk_len, heads, kv_heads, dq, dv, num_splits=0):
    return int(load().vpp_chunk_attn_fp8_widen_workspace_size(int(prefix_len), int(chunk_len), heads, kv_heads,
                                                              dq, dv, num_splits))


def vpp_chunk_attn_fp8(q, k_cache, v_cache, k_scale, v_scale, prefix_len, block_table=None, out=None,
                       lse=None, softmax_scale=0.0, num_splits=0, workspace=None, stream=None, widen=False):
    """Chunk attention over an E4M3 cache (bf16 q), paged or contiguous.  The
    kernel widens the codes itself unless the workspace also holds a bf16
    copy of the visible keys (widen=True allocates one when no workspace is
    given)."""
    _need_cuda(q, k_cache, v_cache, block_table, out, lse, workspace)
    _fp8_cache(k_cache, v_cache)
    C, H, dq = q.shape
    Hkv = k_cache.shape[-2]
    dv = v_cache.shape[-1]
    _scales(k_scale, v_scale, Hkv)
    if out is None:
        out = torch.empty((C, H, dv), dtype=torch.bfloat16, device=q.device)
    if workspace is None:
        size = chunk_attn_fp8_widen_workspace_size if widen else chunk_attn_fp8_workspace_size
        need = size(prefix_len, C, H, Hkv, dq, dv, num_splits)
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    wbytes = workspace.numel() * workspace.element_size()
    _check("vpp_chunk_attn_fp8", load().vpp_chunk_attn_fp8(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(block_table),
        k_cache.shape[0], int(prefix_len), C, H, Hkv, dq, dv, float(softmax_scale), int(num_splits),
        _ptr(out), _ptr(lse), _ptr(workspace), wbytes, _stream(stream)))
    return out


def mixed_attn_fp8_workspace_size(cu_seqlens_q, ctx_lens, heads, kv_heads, dq, dv):
    cu, cu_p = _i32_host(cu_seqlens_q)
    ctx, ctx_p = _i32_host(ctx_lens)
    return int(load().vpp_mixed_attn_fp8_workspace_size(cu_p, ctx_p, len(ctx), heads, kv_heads, dq, dv))


def mixed_attn_fp8_widen_workspace_size(cu_seqlens_q, ctx_lens, heads, kv_heads, dq, dv):
    cu, cu_p = _i32_host(cu_seqlens_q)
    ctx, ctx_p = _i32_host(ctx_lens)
    return int(load().vpp_mixed_attn_fp8_widen_workspace_size(cu_p, ctx_p, len(ctx), heads, kv_heads, dq, dv))


def vpp_mixed_attn_fp8(q, k_cache, v_cache, k_scale, v_scale, block_table, cu_seqlens_q, ctx_lens, out=None,
                       lse=None, softmax_scale=0.0, workspace=None, stream=None, widen=False):
    """Mixed micro-batch over an E4M3 paged cache (host cu_seqlens_q / ctx_lens);
    widen as for vpp_chunk_attn_fp8."""
    _need_cuda(q, k_cache, v_cache, block_table, out, lse, workspace)
    _fp8_cache(k_cache, v_cache)
    T, H, dq = q.shape
    Hkv = k_cache.shape[2]
    dv = v_cache.shape[3]
    _scales(k_scale, v_scale, Hkv)
    cu, cu_p = _i32_host(cu_seqlens_q)
    ctx, ctx_p = _i32_host(ctx_lens)
    if out is None:
        out = torch.empty((T, H, dv), dtype=torch.bfloat16, device=q.device)
    need = (mixed_attn_fp8_widen_workspace_size if widen else mixed_attn_fp8_workspace_size)(cu, ctx, H, Hkv, dq, dv)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("vpp_mixed_attn_fp8", load().vpp_mixed_attn_fp8(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(block_table),
        block_table.shape[1], k_cache.shape[0], cu_p, ctx_p, len(ctx), H, Hkv, dq, dv, float(softmax_scale),
        _ptr(out), _ptr(lse), _ptr(workspace), wbytes, _stream(stream)))
    return out


# ----------------------------------------------------------------- top-k sparse prefix
def topk_chunk_attn_workspace_size(chunk_len, topk, heads, head_dim):
    return int(load().vpp_topk_chunk_attn_workspace_size(int(chunk_len), int(topk), heads, head_dim))


def _topk_args(q, k_cache, topk_idx, topk_len, workspace):
    if topk_idx.dtype != torch.int32 or topk_len.dtype != torch.int32:
        raise ValueError("topk_idx and topk_len are int32")
    C, H, d = q.shape
    topk = topk_idx.shape[1]
    if topk_idx.shape[0] != C or topk_len.shape[0] != C:
        raise ValueError("one index row and one length per query token")
    if workspace is None:
        need = topk_chunk_attn_workspace_size(C, topk, H, d)
        if need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return C, H, d, topk, workspace, wbytes


def vpp_topk_chunk_attn(q, k_cache, v_cache, prefix_len, topk_idx, topk_len, block_table=None, out=None, lse=None,
                        softmax_scale=0.0, workspace=None, stream=None):
    """Top-k sparse prefix attention of a chunk (bf16 q and cache): query token i
    attends the key positions topk_idx[i, :topk_len[i]] (int32 CUDA tensors)."""
    _need_cuda(q, k_cache, v_cache, topk_idx, topk_len, block_table, out, lse, workspace)
    C, H, d, topk, workspace, wbytes = _topk_args(q, k_cache, topk_idx, topk_len, workspace)
    Hkv = k_cache.shape[-2]
    if out is None:
        out = torch.empty((C, H, d), dtype=torch.bfloat16, device=q.device)
    _check("vpp_topk_chunk_attn", load().vpp_topk_chunk_attn(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), k_cache.shape[0], int(prefix_len), C,
        _ptr(topk_idx), _ptr(topk_len), topk, H, Hkv, d, float(softmax_scale), _ptr(out), _ptr(lse),
        _ptr(workspace), wbytes, _stream(stream)))
    return out


def vpp_topk_chunk_attn_fp8(q, k_cache, v_cache, k_scale, v_scale, prefix_len, topk_idx, topk_len,
                            block_table=None, out=None, lse=None, softmax_scale=0.0, workspace=None, stream=None):
    """vpp_topk_chunk_attn over an E4M3 cache (uint8 codes, per-kv-head scales)."""
    _need_cuda(q, k_cache, v_cache, topk_idx, topk_len, block_table, out, lse, workspace)
    _fp8_cache(k_cache, v_cache)
    C, H, d, topk, workspace, wbytes = _topk_args(q, k_cache, topk_idx, topk_len, workspace)
    Hkv = k_cache.shape[-2]
    _scales(k_scale, v_scale, Hkv)
    if out is None:
        out = torch.empty((C, H, d), dtype=torch.bfloat16, device=q.device)
    _check("vpp_topk_chunk_attn_fp8", load().vpp_topk_chunk_attn_fp8(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(block_table), k_cache.shape[0],
        int(prefix_len), C, _ptr(topk_idx), _ptr(topk_len), topk, H, Hkv, d, float(softmax_scale), _ptr(out),
        _ptr(lse), _ptr(workspace), wbytes, _stream(stream)))
    return out


# ----------------------------------------------------------------- status
def vpp_last_device_status(stream=None) -> int:
    code = ctypes.c_int(0)
    _check("vpp_last_device_status", load().vpp_last_device_status(_stream(stream), ctypes.byref(code)))
    return code.value


def vpp_selftest_wait_timeout(timeout_us: int, stream=None):
    _check("vpp_selftest_wait_timeout", load().vpp_selftest_wait_timeout(int(timeout_us), _stream(stream)))
