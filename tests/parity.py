"""Shared helpers of the GPU parity tests: tolerance checks against the fp64
oracle, row sampling for workloads too large for the oracle to do in full, and
the seeded workload builders."""
from __future__ import annotations

import math

import numpy as np
import torch

import swa_inputs

# bf16 outputs against the fp64 oracle: element-wise max-abs and tensor rel-L2
MAX_ABS = 2e-2
REL_L2 = 5e-3


def compare(gpu_out: torch.Tensor, ref: np.ndarray, what: str = "",
            max_abs: float = MAX_ABS, rel_l2: float = REL_L2):
    g = gpu_out.detach().float().cpu().double().numpy()
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = g - ref
    ma = float(np.max(np.abs(err))) if err.size else 0.0
    rl = float(np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-300))
    assert ma <= max_abs and rl <= rel_l2, f"{what}: max-abs {ma:.3e} rel-L2 {rl:.3e}"
    return ma, rl


def sample_rows(L: int, w: int, s: int, n_random: int, seed: int,
                head_cap: int | None = None) -> np.ndarray:
    """All rows t < w + s + 128 (the rows whose window still reaches the first
    keys, including the switch from a merged sink range to a separate sink
    tile near t = w + s), the last 128 rows, and n_random random rows.
    head_cap bounds the first part for full-causal layers (w >= L), where every
    row reaches the first keys."""
    n_head = min(L, w + s + 128)
    if head_cap is not None:
        n_head = min(n_head, head_cap)
    head = np.arange(n_head)
    tail = np.arange(max(0, L - 128), L)
    rng = np.random.default_rng(seed)
    mid = rng.integers(0, L, size=n_random)
    return np.unique(np.concatenate([head, tail, mid])).astype(np.int64)


def prefill_case(B, L, Hq, Hkv, d, seed, sink_rows=0):
    q, k, v = swa_inputs.prefill_inputs(B, L, Hq, Hkv, d, seed, sink_rows=sink_rows)
    return q, k, v


def scale_for(d: int) -> float:
    return 1.0 / math.sqrt(d)
