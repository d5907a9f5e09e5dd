"""Pins of the fp8 (E4M3) KV-cache oracle against things other than itself.

The codec is tied to the OCP 8-bit floating point specification's E4M3
format (bias 7, 3 mantissa bits, no infinities, max 448, NaN = S.1111.111)
through its published values, to torch's float8_e4m3fn conversion (a library
routine; round to nearest even, no saturation), to exact rational
arithmetic, and to the rounding error bound.  Mutation tests at the end
plant plausible mistakes in a copy of the module and check that a pin fails.
"""

import os
import types
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle.fp8 as fp8
from oracle import causal_chunk_attention


def _torch_codes(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


# ------------------------------------------------------------------- codec
PUBLISHED = {            # code: value (E4M3 of the OCP FP8 specification)
    0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0,
    0x3F: 1.875, 0x40: 2.0, 0x70: 128.0, 0x78: 256.0, 0x7E: 448.0, 0x81: -(2.0 ** -9), 0xB8: -1.0, 0xFE: -448.0,
}


def test_published_values():
    for code, val in PUBLISHED.items():
        assert fp8.e4m3_decode(code) == val, hex(code)
        assert fp8.e4m3_encode(val) == code, hex(code)
    assert np.isnan(fp8.e4m3_decode(0x7F)) and np.isnan(fp8.e4m3_decode(0xFF))
    assert np.signbit(fp8.e4m3_decode(0x80)) and fp8.e4m3_decode(0x80) == 0.0


def test_value_set_structure():
    v = fp8.e4m3_decode(np.arange(256))
    pos = v[:0x7F]
    assert np.all(np.diff(pos) > 0)                      # 127 ascending finite values
    assert np.array_equal(-pos, v[0x80:0xFF])             # sign bit mirrors
    assert np.isnan(v).sum() == 2
    # exponent binades: 8 values per binade, spacing 2^(e-10) (3 mantissa bits)
    for e in range(1, 16):
        b = pos[8 * e: 8 * e + 8] if 8 * e + 8 <= 0x7F else pos[8 * e:]
        assert np.allclose(np.diff(b), 2.0 ** (e - 10))


def test_decode_matches_torch_for_every_code():
    t = torch.from_numpy(np.arange(256, dtype=np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    o = fp8.e4m3_decode(np.arange(256))
    assert np.array_equal(np.isnan(t), np.isnan(o))
    assert np.array_equal(t[~np.isnan(t)], o[~np.isnan(o)])


def test_encode_matches_torch_in_range():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(100000) * 40, rng.standard_normal(50000) * 2.0 ** -7,
                        rng.uniform(-448, 448, 50000)]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    assert np.array_equal(fp8.e4m3_encode(x), _torch_codes(x))


def test_ties_go_to_the_even_code_and_neighbours_to_the_nearest():
    v = fp8.e4m3_decode(np.arange(0x7F))
    for i in range(0x7E):
        mid = (v[i] + v[i + 1]) / 2
        even = i if i % 2 == 0 else i + 1
        assert fp8.e4m3_encode(mid) == even
        assert fp8.e4m3_encode(-mid) == even | 0x80
        eps = (v[i + 1] - v[i]) * 1e-6
        assert fp8.e4m3_encode(mid - eps) == i
        assert fp8.e4m3_encode(mid + eps) == i + 1


def test_saturation_and_specials():
    assert fp8.e4m3_encode(448.0) == 0x7E
    assert fp8.e4m3_encode(464.0) == 0x7E           # would round past 448: clamps
    assert fp8.e4m3_encode(1e30) == 0x7E and fp8.e4m3_encode(np.inf) == 0x7E
    assert fp8.e4m3_encode(-1e30) == 0xFE and fp8.e4m3_encode(-np.inf) == 0xFE
    assert fp8.e4m3_encode(np.nan) & 0x7F == 0x7F
    assert fp8.e4m3_encode(-0.0) == 0x80 and fp8.e4m3_encode(0.0) == 0x00
    assert fp8.e4m3_encode(-(2.0 ** -11)) == 0x80     # rounds to zero, keeps the sign
    assert fp8.e4m3_encode(2.0 ** -10) == 0x00        # half the smallest subnormal: tie to even 0
    assert fp8.e4m3_encode(3 * 2.0 ** -11) == 0x01


def test_round_trip_of_every_finite_code():
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F])
    assert np.array_equal(fp8.e4m3_encode(fp8.e4m3_decode(codes)), codes)


def test_rounding_error_bound():
    """Round to nearest: error <= half the spacing, 2^(e-4) in binade
    [2^e, 2^(e+1)), and 2^-10 among subnormals."""
    rng = np.random.default_rng(4)
    x = np.concatenate([rng.uniform(-448, 448, 200000), rng.uniform(-2.0 ** -6, 2.0 ** -6, 50000)])
    err = np.abs(fp8.e4m3_decode(fp8.e4m3_encode(x)) - x)
    a = np.abs(x)
    bound = np.where(a < 2.0 ** -6, 2.0 ** -10, np.exp2(np.floor(np.log2(np.maximum(a, 2.0 ** -6))) - 4))
    assert np.all(err <= bound)


# Quotients rounded to float32 land exactly on an E4M3 midpoint although the
# exact quotient does not: x (bf16), s (float32), midpoint index i.  The
# exact quotient rounds to the odd neighbour; the float32 one ties to even.
QUOTIENT_TIES = [(3.328125, 200.4705810546875, 8), (2.296875, 123.78947448730469, 9),
                 (1.9296875, 94.0952377319336, 10), (0.671875, 29.913043975830078, 11)]


@pytest.mark.parametrize("x,s,i", QUOTIENT_TIES)
def test_quotient_is_rounded_in_float32_first(x, s, i):
    v = fp8.e4m3_decode(np.arange(0x7F))
    mid = Fraction((v[i] + v[i + 1]) / 2)
    exact = Fraction(x) / Fraction(float(np.float32(s)))
    assert exact != mid
    exact_code = i if exact < mid else i + 1
    even_code = i if i % 2 == 0 else i + 1
    assert exact_code != even_code
    got = fp8.quantize_kv(np.full((1, 1, 2), x), np.array([s], dtype=np.float32))
    assert np.all(got == even_code)


def test_quantize_uses_one_scale_per_kv_head():
    rng = np.random.default_rng(5)
    x = torch.from_numpy(rng.standard_normal((6, 3, 8)) * 0.1).to(torch.bfloat16).float().numpy()
    s = np.array([0.5 / 448, 0.25 / 448, 1.0 / 448], dtype=np.float32)
    codes = fp8.quantize_kv(x, s)
    for h in range(3):
        assert np.array_equal(codes[:, h, :], fp8.e4m3_encode((x[:, h, :] / s[h]).astype(np.float32)))
    deq = fp8.dequantize_kv(codes, s)
    for h in range(3):
        assert np.array_equal(deq[:, h, :], fp8.e4m3_decode(codes[:, h, :]) * float(s[h]))


def test_attention_over_dequantised_cache_is_close_to_bf16():
    """Sanity of the reading (not a parity bound): fp8 KV with per-head
    amax scales changes a chunk's attention output by a few percent at most."""
    rng = np.random.default_rng(6)
    P, C, Hq, Hkv, d = 200, 40, 4, 2, 64
    q = rng.standard_normal((C, Hq, d)) / 8
    k = rng.standard_normal((P + C, Hkv, d)) / 8
    v = rng.standard_normal((P + C, Hkv, d)) / 8
    ks = (np.abs(k).max(axis=(0, 2)) / 448).astype(np.float32)
    vs = (np.abs(v).max(axis=(0, 2)) / 448).astype(np.float32)
    kq = fp8.dequantize_kv(fp8.quantize_kv(k, ks), ks)
    vq = fp8.dequantize_kv(fp8.quantize_kv(v, vs), vs)
    o, _ = causal_chunk_attention(q, k, v, P)
    o8, _ = causal_chunk_attention(q, kq, vq, P)
    assert np.linalg.norm(o8 - o) / np.linalg.norm(o) < 0.05


# ----------------------------------------------------------- mutation tests
_SRC = open(os.path.join(os.path.dirname(fp8.__file__), "fp8.py")).read()

MUTANTS = {
    "ties_up": ("take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))",
                "take_hi = (d_hi <= d_lo)"),
    "bias_8": ("np.exp2(e.astype(np.float64) - 7.0)", "np.exp2(e.astype(np.float64) - 8.0)"),
    "subnormal_exp": ("m / 8.0 * 2.0 ** -6", "m / 8.0 * 2.0 ** -7"),
    "drop_sign": ("return (code | np.where(neg, 0x80, 0)).astype(np.uint8)", "return code.astype(np.uint8)"),
    "float64_quotient": ("q = (x32 / s.reshape(shape)).astype(np.float32)\n    return e4m3_encode(q.astype(np.float64))",
                         "q = x32.astype(np.float64) / s.reshape(shape).astype(np.float64)\n    return e4m3_encode(q)"),
    "truncate": ("take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))", "take_hi = d_hi < 0"),
}

_PINS = [test_published_values, test_value_set_structure, test_decode_matches_torch_for_every_code,
         test_encode_matches_torch_in_range, test_ties_go_to_the_even_code_and_neighbours_to_the_nearest,
         test_saturation_and_specials, test_round_trip_of_every_finite_code, test_rounding_error_bound,
         test_quantize_uses_one_scale_per_kv_head]


def _pins_pass(mod):
    global fp8
    saved = fp8
    fp8 = mod
    try:
        for t in _PINS:
            t()
        for x, s, i in QUOTIENT_TIES:
            test_quotient_is_rounded_in_float32_first(x, s, i)
    except AssertionError:
        return False
    finally:
        fp8 = saved
    return True


def _module(src, name):
    mod = types.ModuleType(name)
    exec(compile(src, name, "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    old, new = MUTANTS[name]
    assert _SRC.count(old) == 1, name
    assert not _pins_pass(_module(_SRC.replace(old, new), "fp8_mutant_" + name)), name


def test_unmutated_copy_passes_pins():
    assert _pins_pass(_module(_SRC, "fp8_copy"))


def test_every_e4m3_value_is_an_f16_value():
    # The fp8 attention kernels widen codes to f16 operands with a plain
    # conversion and multiply by the scales afterwards; that is exact only if
    # every finite E4M3 value (3 mantissa bits, exponents 2^-9 .. 2^8) is an
    # f16 value (10 mantissa bits, subnormals down to 2^-24), signed zeros
    # included.
    codes = np.arange(256, dtype=np.uint8)
    val = fp8.e4m3_decode(codes).astype(np.float64)
    finite = ~np.isnan(val)
    assert finite.sum() == 254
    as_f16 = val[finite].astype(np.float16)
    assert np.array_equal(as_f16.astype(np.float64), val[finite])
    assert np.array_equal(np.signbit(as_f16), np.signbit(val[finite]))
    assert np.abs(val[finite]).max() == 448.0 and np.abs(val[finite][val[finite] != 0]).min() == 2.0 ** -9
