"""Shared helpers for the GPU parity tests (no attention arithmetic here)."""

from __future__ import annotations

import numpy as np
import torch

# Tolerances for bf16 inputs with fp32 accumulation: max-abs 2e-2, relative
# L2 5e-3 on the output; the LSE is compared to 1e-2 absolute.
MAX_ABS = 2e-2
REL_L2 = 5e-3
LSE_ABS = 1e-2


def to_np64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    max_abs = float(np.max(np.abs(got - ref))) if got.size else 0.0
    den = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(got - ref) / den) if den > 0 else float(np.linalg.norm(got - ref))
    return max_abs, rel


def assert_close(got, ref, max_abs=MAX_ABS, rel_l2=REL_L2, what="out"):
    ma, rl = errors(got, ref)
    assert np.all(np.isfinite(np.asarray(got))), f"{what}: non-finite values"
    assert ma <= max_abs and rl <= rel_l2, f"{what}: max_abs {ma:.3e} (<= {max_abs}), rel_l2 {rl:.3e} (<= {rel_l2})"
    return ma, rl


def paged_cache(num_blocks, kv_heads, d, device, fill=0.0):
    c = torch.empty((num_blocks, 64, kv_heads, d), dtype=torch.bfloat16, device=device)
    c.fill_(fill)
    return c


def random_table(n_needed, pool, seed):
    rng = np.random.default_rng(seed)
    return rng.permutation(pool)[:n_needed].astype(np.int32)
