"""fp8 (E4M3) KV-cache codec and quantiser: exact CPU oracle.

TEST INFRASTRUCTURE ONLY.  Nothing in the product package imports, calls or
links this module; only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code, table or helper with the CUDA path.

Sources:

* [GLM PP note] "02 · 并行策略与 PP 切分" (deployment note), §1 and §3.2: the
  deployment keeps its KV cache in an fp8 format, 656 B per token and layer
  against 1152 B in bf16, which nearly doubles the tokens a GPU can hold.
  The pages give the byte counts only, not the element format or scaling.
* The element format is E4M3 of the OCP 8-bit floating point specification
  (OFP8): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent
  field 0 holds subnormals (m / 8) * 2^-6; there are no infinities; S.1111.111
  is NaN, so the largest finite magnitude is S.1111.110 = 448.

Readings:

* One float32 scale per kv head for K and one for V; an element's value is
  decode(code) * scale.
* Quantisation: code = E4M3 rounding of the float32 quotient fl32(x / scale)
  (x is a bf16 value, exact in float32; the quotient is rounded to nearest
  even in float32, the precision the kernel works in), to the nearest E4M3
  value with ties to the even mantissa; magnitudes above 448 clamp to 448
  (saturating to the largest finite value); the sign of zero is kept.

Everything else is exact (float64 holds every E4M3 value and every product
with a float32 scale exactly).
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E4M3_NAN_CODE = 0x7F


def e4m3_decode(code) -> np.ndarray:
    """Value of each 8-bit code (float64; NaN for S.1111.111)."""
    c = np.asarray(code, dtype=np.int64) & 0xFF
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    mag = np.where((c & 0x7F) == E4M3_NAN_CODE, np.nan, mag)
    return sign * mag


# The 127 non-negative finite values, ascending with their codes 0x00 .. 0x7E.
_POS_VALUES = e4m3_decode(np.arange(0x7F))


def e4m3_encode(x) -> np.ndarray:
    """Round-to-nearest-even E4M3 code of each value, saturating at 448.

    x is taken as exact (float64).  NaN maps to the NaN code with x's sign."""
    x = np.asarray(x, dtype=np.float64)
    neg = np.signbit(x)
    a = np.abs(x)
    nan = np.isnan(a)
    a = np.where(nan, 0.0, np.minimum(a, E4M3_MAX))
    hi = np.searchsorted(_POS_VALUES, a, side="left")     # first value >= a
    hi = np.minimum(hi, len(_POS_VALUES) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - _POS_VALUES[lo]
    d_hi = _POS_VALUES[hi] - a
    # nearest; on a tie the even code (even mantissa: the code's low bit)
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(take_hi, hi, lo)
    code = np.where(a == _POS_VALUES[hi], hi, code)
    code = np.where(nan, E4M3_NAN_CODE, code)
    return (code | np.where(neg, 0x80, 0)).astype(np.uint8)


def quantize_kv(x, scale, head_axis: int = -2) -> np.ndarray:
    """Codes of x (bf16 values, any layout) with one float32 scale per kv head.

    x: [..., Hkv, d] (head_axis selects the kv-head axis); scale: [Hkv].
    The quotient x / scale is formed in float32 (round to nearest even)."""
    x32 = np.asarray(x, dtype=np.float32)
    s = np.asarray(scale, dtype=np.float32)
    shape = [1] * x32.ndim
    shape[head_axis] = s.shape[0]
    q = (x32 / s.reshape(shape)).astype(np.float32)
    return e4m3_encode(q.astype(np.float64))


def dequantize_kv(codes, scale, head_axis: int = -2) -> np.ndarray:
    """decode(code) * scale, exact in float64."""
    v = e4m3_decode(codes)
    s = np.asarray(scale, dtype=np.float32).astype(np.float64)
    shape = [1] * v.ndim
    shape[head_axis] = s.shape[0]
    return v * s.reshape(shape)

