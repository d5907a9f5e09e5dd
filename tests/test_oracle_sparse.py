"""Pins of the top-k sparse prefix attention oracle (CPU).

Against the dense oracle when every earlier key is listed (itself pinned by
tests/test_oracle.py), a long-double brute force over the gathered keys,
closed forms (one listed key; a key listed twice), invariants (order of the
list, GQA head sharing) and planted mistakes.
"""

import os
import types

import numpy as np
import pytest

import oracle
import oracle.sparse as sp
from oracle import brute


def _case(rng, C, P, Hq, Hkv, d, dv=None):
    dv = dv or d
    q = rng.standard_normal((C, Hq, d))
    k = rng.standard_normal((P + C, Hkv, d))
    v = rng.standard_normal((P + C, Hkv, dv))
    return q, k, v


def _random_idx(rng, P, C, kmax):
    idx = np.full((C, kmax), -1, dtype=np.int64)
    lens = np.zeros(C, dtype=np.int64)
    for i in range(C):
        p = P + i
        n = min(p + 1, kmax)
        keys = np.concatenate([[p], rng.choice(p, size=n - 1, replace=False)]) if n > 1 else np.array([p])
        rng.shuffle(keys)
        idx[i, :n] = keys
        lens[i] = n
    return idx, lens


def test_all_earlier_keys_listed_equals_dense_causal():
    rng = np.random.default_rng(1)
    P, C = 37, 11
    q, k, v = _case(rng, C, P, 4, 2, 16)
    idx = np.full((C, P + C), -1)
    lens = np.zeros(C, dtype=np.int64)
    for i in range(C):
        idx[i, : P + i + 1] = rng.permutation(P + i + 1)
        lens[i] = P + i + 1
    out, lse = sp.topk_chunk_attention(q, k, v, P, idx, lens)
    ref, ref_lse = oracle.causal_chunk_attention(q, k, v, P)
    np.testing.assert_allclose(out, ref, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, atol=1e-12)


def test_matches_long_double_brute_force_on_gathered_keys():
    """The brute force's causal rule with prefix n-1 lets one query see all n
    gathered keys: plain indexing, no attention arithmetic in the gather."""
    rng = np.random.default_rng(2)
    P, C, Hq, Hkv, d, kmax = 60, 9, 6, 3, 8, 24
    q, k, v = _case(rng, C, P, Hq, Hkv, d, 12)
    idx, lens = _random_idx(rng, P, C, kmax)
    out, lse = sp.topk_chunk_attention(q, k, v, P, idx, lens)
    s = 1 / np.sqrt(d)
    for i in range(C):
        keys = idx[i, : lens[i]]
        n = len(keys)
        bo, bl = brute.causal_chunk_attention(q[i:i + 1], k[keys], v[keys], n - 1, s)
        np.testing.assert_allclose(out[i], bo[0], atol=1e-12)
        np.testing.assert_allclose(lse[:, i], bl[:, 0], atol=1e-12)


def test_single_listed_key_returns_its_value():
    rng = np.random.default_rng(3)
    P, C = 20, 5
    q, k, v = _case(rng, C, P, 4, 2, 8)
    idx = np.array([[3], [21], [0], [22], [24]])
    out, lse = sp.topk_chunk_attention(q, k, v, P, idx, np.ones(C, dtype=np.int64))
    s = 1 / np.sqrt(8)
    for i in range(C):
        for h in range(4):
            np.testing.assert_allclose(out[i, h], v[idx[i, 0], h // 2], atol=1e-15)
            np.testing.assert_allclose(lse[h, i], s * q[i, h] @ k[idx[i, 0], h // 2], atol=1e-12)


def test_key_listed_twice_counts_twice():
    rng = np.random.default_rng(4)
    P, C = 30, 3
    q, k, v = _case(rng, C, P, 2, 1, 8)
    idx = np.array([[5, 7, 9], [1, 2, 31], [0, 10, 32]])
    once, l1 = sp.topk_chunk_attention(q, k, v, P, idx, np.full(C, 3))
    dup = np.concatenate([idx, idx[:, :1]], axis=1)
    twice, l2 = sp.topk_chunk_attention(q, k, v, P, dup, np.full(C, 4))
    s = 1 / np.sqrt(8)
    for i in range(C):
        for h in range(2):
            sc = s * k[idx[i], 0] @ q[i, h]
            w = np.exp(sc - sc.max())
            w[0] *= 2
            np.testing.assert_allclose(twice[i, h], (w @ v[idx[i], 0]) / w.sum(), atol=1e-12)
            np.testing.assert_allclose(l2[h, i], sc.max() + np.log(w.sum()), atol=1e-12)
    assert not np.allclose(once, twice)


def test_list_order_and_padding_do_not_matter():
    rng = np.random.default_rng(5)
    P, C, kmax = 100, 6, 40
    q, k, v = _case(rng, C, P, 4, 4, 16)
    idx, lens = _random_idx(rng, P, C, kmax)
    out, lse = sp.topk_chunk_attention(q, k, v, P, idx, lens)
    idx2 = idx.copy()
    for i in range(C):
        idx2[i, : lens[i]] = rng.permutation(idx[i, : lens[i]])
        idx2[i, lens[i]:] = rng.integers(-5, 5, kmax - lens[i])   # entries past len are never read
    out2, lse2 = sp.topk_chunk_attention(q, k, v, P, idx2, lens)
    np.testing.assert_allclose(out, out2, atol=1e-12)
    np.testing.assert_allclose(lse, lse2, atol=1e-12)


def test_rejects_keys_after_the_query_and_bad_lengths():
    rng = np.random.default_rng(6)
    q, k, v = _case(rng, 2, 10, 2, 1, 8)
    with pytest.raises(ValueError):
        sp.topk_chunk_attention(q, k, v, 10, np.array([[11], [0]]), np.array([1, 1]))
    with pytest.raises(ValueError):
        sp.topk_chunk_attention(q, k, v, 10, np.array([[1], [0]]), np.array([0, 1]))


def test_flops_count():
    assert sp.topk_flops([3, 5], 4, 128, 128) == 2 * 256 * 4 * 8


# ----------------------------------------------------------- mutation tests
_SRC = open(os.path.join(os.path.dirname(sp.__file__), "sparse.py")).read()
MUTANTS = {
    "no_scale": ("scores = s * (kk[:, g, :] @ q_rows[r, h])", "scores = (kk[:, g, :] @ q_rows[r, h])"),
    "ignore_len": ("keys = idx_rows[r, :n]", "keys = idx_rows[r]"),
    "head_mod": ("g = h // kv_group", "g = h % k.shape[1]"),
    "lse_no_max": ("lse[h, r] = m + np.log(den)", "lse[h, r] = np.log(den)"),
    "value_of_key": ("vv = np.asarray(v[keys], dtype=np.float64)", "vv = np.asarray(v[np.sort(keys)], dtype=np.float64)"),
}


def _pins_pass(mod):
    saved = sp.topk_rows, sp.topk_chunk_attention
    try:
        globals()["sp"] = mod
        for t in (test_all_earlier_keys_listed_equals_dense_causal, test_matches_long_double_brute_force_on_gathered_keys,
                  test_single_listed_key_returns_its_value, test_key_listed_twice_counts_twice,
                  test_list_order_and_padding_do_not_matter):
            t()
    except (AssertionError, ValueError, IndexError):
        return False
    finally:
        import oracle.sparse as orig
        globals()["sp"] = orig
    return True


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    old, new = MUTANTS[name]
    assert _SRC.count(old) == 1, name
    mod = types.ModuleType("sparse_mutant_" + name)
    exec(compile(_SRC.replace(old, new), mod.__name__, "exec"), mod.__dict__)
    assert not _pins_pass(mod), name


def test_unmutated_copy_passes_pins():
    mod = types.ModuleType("sparse_copy")
    exec(compile(_SRC, mod.__name__, "exec"), mod.__dict__)
    assert _pins_pass(mod)
