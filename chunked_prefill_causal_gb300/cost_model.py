"""Latency model of one attention micro-batch, for chunk-size schedulers.

"Revisiting Pipeline Parallelism for LLM Serving", §2.3 (the ALP latency
predictor): an iteration's time is an offline-profiled part linear in the
number of new tokens, alpha_0 + alpha_1 * N_tokens, plus an online part in
three attention features, each summed over the batch's requests:

    sum L_past * L_pre   attention of a new prefill chunk to its cached prefix
    sum L_pre^2          attention inside the chunk
    sum L_dec            decode rows reading their cached context

with L_past the prefix length, L_pre the chunk length and L_dec a decode
request's context length.  The online coefficients are adapted after every
iteration by recursive least squares (RLS) with a forgetting factor on the
gap between the measured time and the offline part.  The page's displayed
formulas were lost in extraction; the model above is the plain reading of its
text (linear in exactly these terms).

The VPP technical review's Eq. (2), tau_k = (k+1) t, is the special case of a
fixed chunk C: L_past = kC, so the time is affine in the chunk index k.
"""

from __future__ import annotations

import dataclasses

import numpy as np

# Feature units keep the normal equations well conditioned: pairs in units of
# 2^30, decode context in units of 2^20, tokens in units of 2^10.
_PAIR_UNIT = float(1 << 30)
_DEC_UNIT = float(1 << 20)
_TOK_UNIT = float(1 << 10)


@dataclasses.dataclass(frozen=True)
class MicroBatch:
    """Prefill chunks as (L_past, L_pre) pairs and decode context lengths."""

    prefill: tuple = ()
    decode: tuple = ()

    @property
    def n_tokens(self) -> int:
        return sum(int(c) for _, c in self.prefill) + len(self.decode)


def attention_features(batch: MicroBatch) -> np.ndarray:
    """[sum L_past*L_pre, sum L_pre^2, sum L_dec] in model units."""
    past_pre = sum(float(p) * float(c) for p, c in batch.prefill)
    pre_sq = sum(float(c) * float(c) for _, c in batch.prefill)
    dec = sum(float(d) for d in batch.decode)
    return np.array([past_pre / _PAIR_UNIT, pre_sq / _PAIR_UNIT, dec / _DEC_UNIT])


def token_features(batch: MicroBatch) -> np.ndarray:
    """[1, N_tokens] in model units."""
    return np.array([1.0, batch.n_tokens / _TOK_UNIT])


class LatencyModel:
    """alpha . [1, N] (offline least squares) + beta . features (online RLS)."""

    def __init__(self, forgetting: float = 0.98, delta: float = 1e4):
        if not 0.0 < forgetting <= 1.0:
            raise ValueError("forgetting factor must be in (0, 1]")
        self.lam = float(forgetting)
        self.alpha = np.zeros(2)
        self.beta = np.zeros(3)
        self.cov = np.eye(3) * float(delta)   # RLS inverse-correlation matrix

    # ------------------------------------------------------------- offline
    def fit_offline(self, batches, times):
        """Least-squares fit of alpha on token counts alone."""
        X = np.stack([token_features(b) for b in batches])
        self.alpha = np.linalg.lstsq(X, np.asarray(times, dtype=np.float64), rcond=None)[0]
        return self.alpha

    def fit_all(self, batches, times):
        """Least-squares fit of alpha and beta together (a full offline profile)."""
        X = np.stack([np.concatenate([token_features(b), attention_features(b)]) for b in batches])
        theta = np.linalg.lstsq(X, np.asarray(times, dtype=np.float64), rcond=None)[0]
        self.alpha, self.beta = theta[:2].copy(), theta[2:].copy()
        return theta

    # -------------------------------------------------------------- online
    def predict(self, batch: MicroBatch) -> float:
        return float(self.alpha @ token_features(batch) + self.beta @ attention_features(batch))

    def update(self, batch: MicroBatch, measured: float) -> float:
        """One RLS step on the residual after the offline part; returns the
        prediction made before the update."""
        pred = self.predict(batch)
        x = attention_features(batch)
        r = float(measured) - float(self.alpha @ token_features(batch))
        px = self.cov @ x
        gain = px / (self.lam + float(x @ px))
        self.beta = self.beta + gain * (r - float(self.beta @ x))
        self.cov = (self.cov - np.outer(gain, px)) / self.lam
        return pred


def mape(pred, meas) -> float:
    """Mean absolute percentage error."""
    pred = np.asarray(pred, dtype=np.float64)
    meas = np.asarray(meas, dtype=np.float64)
    return float(np.mean(np.abs(pred - meas) / np.abs(meas)))
