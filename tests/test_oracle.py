"""Pins of the fp64 CPU oracle against things other than itself.

Each test ties the oracle to the VPP technical review's Eq. (1) (§2.2,
softmax(Q K^T / sqrt(d)) V with token i attending to tokens <= i) and to
chunked prefill (§2.3) through an independent route: a long-double brute
force, a library routine, closed forms, invariants, exact golden values.
The mutation tests at the end plant plausible mistakes in a copy of the
oracle and check that some pin fails for each.
"""

import os
import re
import types

import numpy as np
import pytest
import torch

import oracle
from oracle import brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_case(rng, C, P, Hq, Hkv, dq, dv):
    q = rng.standard_normal((C, Hq, dq))
    k = rng.standard_normal((P + C, Hkv, dq))
    v = rng.standard_normal((P + C, Hkv, dv))
    return q, k, v


SHAPES = [  # C, P, Hq, Hkv, dq, dv
    (1, 0, 1, 1, 4, 4),
    (5, 0, 2, 1, 8, 8),
    (7, 3, 4, 2, 6, 5),
    (16, 40, 4, 1, 16, 8),
    (9, 17, 8, 2, 12, 4),
    (3, 29, 4, 4, 8, 16),
]


@pytest.mark.parametrize("shape", SHAPES)
def test_brute_force_long_double_matches(shape):
    rng = np.random.default_rng(hash(shape) % 2**32)
    C, P, Hq, Hkv, dq, dv = shape
    q, k, v = rand_case(rng, *shape)
    scale = 1.0 / np.sqrt(dq)
    out, lse = oracle.causal_chunk_attention(q, k, v, P)
    bout, blse = brute.causal_chunk_attention(q, k, v, P, scale)
    np.testing.assert_allclose(out, bout, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, blse, rtol=0, atol=1e-12)


@pytest.mark.parametrize("shape", SHAPES)
def test_torch_sdpa_float64_matches(shape):
    """Library cross-check: torch SDPA (CPU, float64) with an explicit mask."""
    rng = np.random.default_rng(7 + hash(shape) % 1000)
    C, P, Hq, Hkv, dq, dv = shape
    q, k, v = rand_case(rng, *shape)
    G = Hq // Hkv
    tq = torch.from_numpy(q).permute(1, 0, 2)                       # [Hq, C, dq]
    tk = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(G, 0)
    tv = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(G, 0)
    mask = torch.arange(P + C)[None, :] <= (P + torch.arange(C))[:, None]
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask)
    out, _ = oracle.causal_chunk_attention(q, k, v, P)
    np.testing.assert_allclose(out, ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("chunk", [1, 3, 8, 13])
def test_chunks_in_order_equal_full_sequence(chunk):
    """§2.3: processing chunks in order reproduces full causal attention."""
    rng = np.random.default_rng(11)
    L, Hq, Hkv, dq, dv = 37, 4, 2, 8, 8
    q = rng.standard_normal((L, Hq, dq))
    k = rng.standard_normal((L, Hkv, dq))
    v = rng.standard_normal((L, Hkv, dv))
    full_out, full_lse = oracle.causal_chunk_attention(q, k, v, 0)
    for P in range(0, L, chunk):
        C = min(chunk, L - P)
        o, l = oracle.causal_chunk_attention(q[P:P + C], k[:P + C], v[:P + C], P)
        np.testing.assert_allclose(o, full_out[P:P + C], rtol=0, atol=1e-12)
        np.testing.assert_allclose(l, full_lse[:, P:P + C], rtol=0, atol=1e-12)


def test_softmax_rows_sum_to_one_and_respect_mask():
    rng = np.random.default_rng(3)
    C, P, Hq, Hkv, dq = 6, 9, 4, 2, 8
    q = rng.standard_normal((C, Hq, dq))
    k = rng.standard_normal((P + C, Hkv, dq))
    probs, lse = oracle.causal_attention_probs(q, k, P)
    np.testing.assert_allclose(probs.sum(axis=2), 1.0, rtol=0, atol=1e-12)
    for i in range(C):
        assert np.all(probs[i, :, P + i + 1:] == 0.0)      # keys after position P+i
        assert np.all(probs[i, :, :P + i + 1] > 0.0)
    v = rng.standard_normal((P + C, Hkv, 5))
    out, lse2 = oracle.causal_chunk_attention(q, k, v, P)
    np.testing.assert_allclose(lse, lse2, rtol=0, atol=1e-12)
    # lse is the log of the denominator: probs = exp(score - lse).
    s = 1.0 / np.sqrt(dq)
    for h in range(Hq):
        sc = s * q[:, h, :] @ k[:, h // 2, :].T
        for i in range(C):
            np.testing.assert_allclose(probs[i, h, :P + i + 1],
                                       np.exp(sc[i, :P + i + 1] - lse[h, i]), rtol=1e-12)


@pytest.mark.parametrize("P,C", [(0, 1), (0, 9), (5, 4), (130, 7)])
def test_zero_query_gives_running_mean_of_v(P, C):
    rng = np.random.default_rng(5)
    Hq, Hkv, dq, dv = 4, 2, 8, 6
    q = np.zeros((C, Hq, dq))
    k = rng.standard_normal((P + C, Hkv, dq))
    v = rng.standard_normal((P + C, Hkv, dv))
    out, lse = oracle.causal_chunk_attention(q, k, v, P)
    for i in range(C):
        p = P + i
        for h in range(Hq):
            np.testing.assert_allclose(out[i, h], v[:p + 1, h // 2].mean(axis=0), rtol=0, atol=1e-12)
            assert abs(lse[h, i] - np.log(p + 1)) < 1e-12


def test_single_visible_key_returns_that_value():
    rng = np.random.default_rng(6)
    q = rng.standard_normal((1, 2, 8))
    k = rng.standard_normal((1, 1, 8))
    v = rng.standard_normal((1, 1, 3))
    out, lse = oracle.causal_chunk_attention(q, k, v, 0)
    np.testing.assert_allclose(out[0, 0], v[0, 0], atol=1e-15)
    np.testing.assert_allclose(out[0, 1], v[0, 0], atol=1e-15)
    np.testing.assert_allclose(lse[:, 0], q[0] @ k[0, 0] / np.sqrt(8), atol=1e-14)


def test_gqa_equals_mha_with_repeated_kv_heads():
    rng = np.random.default_rng(8)
    C, P, Hq, Hkv, dq, dv = 5, 6, 8, 2, 8, 8
    q, k, v = rand_case(rng, C, P, Hq, Hkv, dq, dv)
    G = Hq // Hkv
    o1, l1 = oracle.causal_chunk_attention(q, k, v, P)
    o2, l2 = oracle.causal_chunk_attention(q, np.repeat(k, G, axis=1), np.repeat(v, G, axis=1), P)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


def load_bit_golden():
    rows = []
    with open(os.path.join(GOLDEN, "bit_prefix_means.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            p, c, cnt, den = map(int, line.split())
            rows.append((p, c, cnt, den))
    return rows


def test_mask_probe_matches_golden_bit_means():
    """Q = 0, V[j,c] = bit c of j: out at position p is an exact fraction."""
    rows = load_bit_golden()
    pmax = max(r[0] for r in rows)
    L = pmax + 1
    bits = 10
    j = np.arange(L)
    v = ((j[:, None] >> np.arange(bits)[None, :]) & 1).astype(np.float64)[:, None, :]
    k = np.random.default_rng(1).standard_normal((L, 1, 4))
    # A chunk that starts at prefix 100 and covers positions 100..pmax, and a
    # chunk from 0 that covers the small positions.
    for P in (0, 100):
        C = L - P
        q = np.zeros((C, 2, 4))
        out, _ = oracle.causal_chunk_attention(q, k, v, P)
        for p, c, cnt, den in rows:
            if p < P:
                continue
            assert abs(out[p - P, 1, c] - cnt / den) < 1e-13, (P, p, c)


@pytest.mark.parametrize("offset", [0, 1])
def test_needle_visible_only_when_causal(offset):
    """K = 0 except one key equal to a large multiple of q[i*]: the output
    row i* picks that key's value iff the key is at a position <= P + i*."""
    rng = np.random.default_rng(9)
    C, P, Hq, Hkv, d = 8, 20, 1, 1, 16
    q = rng.standard_normal((C, Hq, d))
    k = np.zeros((P + C, Hkv, d))
    v = rng.standard_normal((P + C, Hkv, d))
    i_star = 4
    j_star = P + i_star + offset
    k[j_star, 0] = 60.0 * q[i_star, 0] / np.linalg.norm(q[i_star, 0]) ** 2 * np.sqrt(d)
    out, _ = oracle.causal_chunk_attention(q, k, v, P)
    if offset == 0:
        np.testing.assert_allclose(out[i_star, 0], v[j_star, 0], atol=1e-12)
    else:
        np.testing.assert_allclose(out[i_star, 0], v[:P + i_star + 1, 0].mean(axis=0), atol=1e-12)


@pytest.mark.parametrize("bounds", [[0, 16, 40], [0, 8, 24, 32, 40], [0, 39, 40]])
def test_split_key_ranges_merge_to_full(bounds):
    """[GLM PP note] §7: partials over disjoint key ranges + LSE merge."""
    rng = np.random.default_rng(12)
    C, P, Hq, Hkv, dq, dv = 8, 32, 4, 2, 8, 8
    q, k, v = rand_case(rng, C, P, Hq, Hkv, dq, dv)
    parts = oracle.split_key_range_attention(q, k, v, P, bounds)
    out, lse = oracle.merge_partials(parts)
    ref_out, ref_lse = oracle.causal_chunk_attention(q, k, v, P)
    np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


def test_paged_gather_equals_contiguous_and_append_places_rows():
    rng = np.random.default_rng(13)
    Hkv, d, L, nb = 2, 8, 300, 9
    table = rng.permutation(nb)[: (L + 63) // 64]
    k = rng.standard_normal((L, Hkv, d))
    cache = np.full((nb, 64, Hkv, d), np.nan)
    # Append in three uneven chunks, then read back through the table.
    for P, C in ((0, 100), (100, 64), (164, 136)):
        oracle.kv_append(cache, table, k[P:P + C], P)
    np.testing.assert_array_equal(oracle.gather_paged(cache, table, L), k)
    # Slot of token j: block table[j//64], row j%64, checked by hand.
    for j in (0, 63, 64, 65, 127, 128, 299):
        np.testing.assert_array_equal(cache[table[j // 64], j % 64], k[j])


def test_mixed_batch_is_per_sequence_and_decode_rows_match_brute():
    rng = np.random.default_rng(14)
    Hq, Hkv, dq, dv = 4, 2, 8, 8
    ctx = [9, 17, 1, 30]
    qlen = [3, 1, 1, 5]
    cu = np.concatenate([[0], np.cumsum(qlen)])
    ks = [rng.standard_normal((n, Hkv, dq)) for n in ctx]
    vs = [rng.standard_normal((n, Hkv, dv)) for n in ctx]
    q = rng.standard_normal((cu[-1], Hq, dq))
    out, lse = oracle.mixed_batch_attention(q, ks, vs, cu, ctx)
    for b in range(4):
        a, e = cu[b], cu[b + 1]
        P = ctx[b] - qlen[b]
        bo, bl = brute.causal_chunk_attention(q[a:e], ks[b], vs[b], P, 1 / np.sqrt(dq))
        np.testing.assert_allclose(out[a:e], bo, atol=1e-12)
        np.testing.assert_allclose(lse[:, a:e], bl, atol=1e-12)


def test_attention_rows_match_full_chunk():
    rng = np.random.default_rng(15)
    C, P, Hq, Hkv, dq, dv = 12, 50, 8, 2, 16, 8
    q, k, v = rand_case(rng, C, P, Hq, Hkv, dq, dv)
    out, lse = oracle.causal_chunk_attention(q, k, v, P)
    toks = np.array([0, 3, 11, 11, 5, 0])
    heads = np.array([0, 7, 3, 4, 1, 5])
    ro, rl = oracle.attention_rows(q[toks, heads], heads, P + toks, k, v, Hq // Hkv)
    np.testing.assert_allclose(ro, out[toks, heads], atol=1e-13)
    np.testing.assert_allclose(rl, lse[heads, toks], atol=1e-13)


def test_chunk_flops_counts_visible_pairs():
    for P, C in ((0, 1), (0, 128), (37, 5), (4096, 4096)):
        pairs = sum(P + i + 1 for i in range(C))
        assert oracle.chunk_flops(P, C, 3, 192, 128) == 2 * (192 + 128) * 3 * pairs
    # long128k chunk 7 (P = 7 * 16384, C = 16384, 64 heads, d 128): 65.97 TFLOP
    assert abs(oracle.chunk_flops(7 * 16384, 16384, 64, 128, 128) / 1e12 - 65.97) < 0.01


# ----------------------------------------------------------- mutation tests
# A plausible mistake planted in a copy of the oracle must make a pin fail.

_SRC = open(os.path.join(os.path.dirname(oracle.__file__), "attention.py")).read()

MUTANTS = {
    "mask_strict": ("allowed = keys[None, :] <= pos[:, None]         # causal rule",
                    "allowed = keys[None, :] < pos[:, None]          # causal rule"),
    "mask_shift": ("pos = P + np.arange(r0, r1)", "pos = P + np.arange(r0, r1) + 1"),
    "scale_dv": ("s = default_scale(dq) if scale is None else float(scale)\n    out = np.zeros((C, Hq, dv))",
                 "s = default_scale(dv) if scale is None else float(scale)\n    out = np.zeros((C, Hq, dv))"),
    "gqa_modulo": ("g = h // G                                  # GQA",
                   "g = h % Hkv                                 # GQA"),
    "lse_drop_max": ("lse[h, r0:r1] = m[:, 0] + np.log(den)", "lse[h, r0:r1] = np.log(den)"),
    "no_normalise": ("out[r0:r1, h, :] = (e @ v[:n_keys, g, :]) / den[:, None]",
                     "out[r0:r1, h, :] = (e @ v[:n_keys, g, :])"),
    "kv_swap": ("scores = s * (q[r0:r1, h, :] @ k[:n_keys, g, :].T)",
                "scores = s * (q[r0:r1, h, :] @ v[:n_keys, g, :dq].T)"),
}


def _mutant(name):
    old, new = MUTANTS[name]
    assert _SRC.count(old) == 1, name
    mod = types.ModuleType("oracle_mutant_" + name)
    exec(compile(_SRC.replace(old, new), mod.__name__, "exec"), mod.__dict__)
    return mod


def _pins_pass(mod):
    """The pins above, re-run against a candidate oracle module."""
    rng = np.random.default_rng(21)
    for C, P, Hq, Hkv, dq, dv in [(9, 17, 8, 2, 12, 12), (4, 6, 4, 1, 16, 8)]:
        q, k, v = rand_case(rng, C, P, Hq, Hkv, dq, dv)
        out, lse = mod.causal_chunk_attention(q, k, v, P)
        bout, blse = brute.causal_chunk_attention(q, k, v, P, 1 / np.sqrt(dq))
        if not (np.allclose(out, bout, atol=1e-12) and np.allclose(lse, blse, atol=1e-12)):
            return False
    return True


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    assert not _pins_pass(_mutant(name)), f"mutant {name} slipped past the pins"


def test_unmutated_copy_passes_pins():
    mod = types.ModuleType("oracle_copy")
    exec(compile(_SRC, mod.__name__, "exec"), mod.__dict__)
    assert _pins_pass(mod)
