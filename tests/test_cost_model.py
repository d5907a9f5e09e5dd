"""Pins of the micro-batch latency model (host code, runs on CPU)."""

import numpy as np
import pytest

from chunked_prefill_causal_gb300.cost_model import (LatencyModel, MicroBatch, attention_features, mape,
                                                     token_features)


def test_features_by_hand():
    b = MicroBatch(prefill=((100, 50), (0, 8)), decode=(10, 20, 30))
    assert b.n_tokens == 50 + 8 + 3
    f = attention_features(b) * np.array([2.0 ** 30, 2.0 ** 30, 2.0 ** 20])
    np.testing.assert_allclose(f, [100 * 50 + 0 * 8, 50 * 50 + 8 * 8, 60], rtol=0, atol=1e-9)
    np.testing.assert_allclose(token_features(b), [1.0, 61 / 1024])


def _random_batches(rng, n):
    out = []
    for _ in range(n):
        pre = tuple((int(rng.integers(0, 131072)), int(rng.integers(1, 16384))) for _ in range(rng.integers(0, 4)))
        dec = tuple(int(x) for x in rng.integers(1, 32768, size=rng.integers(0, 64)))
        out.append(MicroBatch(pre, dec))
    return out


def _truth(b, alpha, beta):
    return float(alpha @ token_features(b) + beta @ attention_features(b))


def test_offline_and_full_fits_recover_noiseless_coefficients():
    rng = np.random.default_rng(1)
    batches = _random_batches(rng, 60)
    alpha, beta = np.array([0.05, 0.3]), np.array([1.7, 0.9, 0.4])
    t = [_truth(b, alpha, beta) for b in batches]
    m = LatencyModel()
    theta = m.fit_all(batches, t)
    np.testing.assert_allclose(theta, np.concatenate([alpha, beta]), rtol=1e-9, atol=1e-12)
    # Token counts alone: exact when the attention part is zero.
    t0 = [float(alpha @ token_features(b)) for b in batches]
    m0 = LatencyModel()
    np.testing.assert_allclose(m0.fit_offline(batches, t0), alpha, rtol=1e-9)


def test_rls_without_forgetting_equals_regularised_least_squares():
    """RLS with forgetting 1 started from beta = 0 and covariance delta * I
    equals the closed form (X^T X + I / delta)^-1 X^T r on the same residuals
    (the standard RLS identity), here on noisy data."""
    rng = np.random.default_rng(2)
    batches = _random_batches(rng, 80)
    alpha, beta = np.array([0.02, 0.1]), np.array([1.1, 0.7, 0.2])
    t = [_truth(b, alpha, beta) * (1 + 0.05 * rng.standard_normal()) for b in batches]
    delta = 10.0
    m = LatencyModel(forgetting=1.0, delta=delta)
    m.alpha = alpha.copy()
    for b, y in zip(batches, t):
        m.update(b, y)
    X = np.stack([attention_features(b) for b in batches])
    r = np.array(t) - np.array([alpha @ token_features(b) for b in batches])
    ridge = np.linalg.solve(X.T @ X + np.eye(3) / delta, X.T @ r)
    np.testing.assert_allclose(m.beta, ridge, rtol=1e-9, atol=1e-12)
    # and it approaches ordinary least squares as delta grows
    m2 = LatencyModel(forgetting=1.0, delta=1e6)
    m2.alpha = alpha.copy()
    for b, y in zip(batches, t):
        m2.update(b, y)
    ls = np.linalg.lstsq(X, r, rcond=None)[0]
    np.testing.assert_allclose(m2.beta, ls, rtol=1e-3)


def test_forgetting_tracks_a_change_of_hardware_speed():
    rng = np.random.default_rng(3)
    first, second = _random_batches(rng, 100), _random_batches(rng, 100)
    alpha = np.array([0.02, 0.1])
    b1, b2 = np.array([1.0, 0.5, 0.3]), np.array([2.0, 1.0, 0.6])   # twice as slow after the change
    errs = {}
    for lam in (1.0, 0.9):
        m = LatencyModel(forgetting=lam)
        m.alpha = alpha.copy()
        for b in first:
            m.update(b, _truth(b, alpha, b1))
        preds, meas = [], []
        for b in second:
            preds.append(m.update(b, _truth(b, alpha, b2)))
            meas.append(_truth(b, alpha, b2))
        errs[lam] = mape(preds[-20:], meas[-20:])
    assert errs[0.9] < 0.1 * errs[1.0]
    assert errs[0.9] < 1e-3


def test_fixed_chunk_time_is_affine_in_chunk_index():
    """VPP technical review §4.1, Eq. (2): with a fixed chunk C the model's
    time grows by the same step per chunk index (L_past = k C)."""
    m = LatencyModel()
    m.alpha, m.beta = np.array([0.1, 0.2]), np.array([1.3, 0.4, 0.0])
    C = 16384
    t = [m.predict(MicroBatch(((k * C, C),))) for k in range(8)]
    steps = np.diff(t)
    np.testing.assert_allclose(steps, steps[0], rtol=1e-12)
    assert steps[0] > 0


def test_bad_forgetting_factor_is_rejected():
    with pytest.raises(ValueError):
        LatencyModel(forgetting=0.0)
