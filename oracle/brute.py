"""ctypes wrapper and build step for ``brute.c`` (test infrastructure only)."""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "brute.c")
_LIB = os.path.join(_HERE, "_build", "libbrute.so")


def build(force: bool = False) -> str:
    """Compile brute.c with gcc into oracle/_build/libbrute.so."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        os.makedirs(os.path.dirname(_LIB), exist_ok=True)
        subprocess.check_call(["gcc", "-O2", "-shared", "-fPIC", "-o", _LIB, _SRC, "-lm"])
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        f = _lib.brute_causal_chunk_attention
        dp = ctypes.POINTER(ctypes.c_double)
        f.argtypes = [dp, dp, dp] + [ctypes.c_int] * 6 + [ctypes.c_double, dp, dp]
        f.restype = ctypes.c_int
    return _lib


def causal_chunk_attention(q, k, v, prefix_len, scale):
    """Long-double triple-loop attention; same contract as the NumPy oracle."""
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    C, Hq, dq = q.shape
    T, Hkv, _ = k.shape
    dv = v.shape[2]
    assert T == prefix_len + C
    out = np.zeros((C, Hq, dv))
    lse = np.zeros((Hq, C))
    dp = ctypes.POINTER(ctypes.c_double)
    rc = lib.brute_causal_chunk_attention(
        q.ctypes.data_as(dp), k.ctypes.data_as(dp), v.ctypes.data_as(dp),
        C, int(prefix_len), Hq, Hkv, dq, dv, float(scale),
        out.ctypes.data_as(dp), lse.ctypes.data_as(dp))
    if rc != 0:
        raise ValueError("brute_causal_chunk_attention rejected its arguments")
    return out, lse
