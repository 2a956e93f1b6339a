"""Helpers for the GPU-vs-oracle parity tests (no layer arithmetic here:
only gathering inputs, calling the oracle and measuring differences)."""
from __future__ import annotations

import numpy as np
import torch

import oracle


def rel_max_err(got, ref) -> float:
    """max |got - ref| / rms(ref)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = np.sqrt(np.mean(ref ** 2))
    return float(np.abs(got - ref).max() / rms)


def err_quantiles(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = np.sqrt(np.mean(ref ** 2))
    e = np.abs(got - ref) / rms
    return {q: float(np.quantile(e, q)) for q in (0.5, 0.99, 1.0)}


def experts_for_tokens(idx: np.ndarray, weights: dict, mode: str, E: int):
    """Copy to the host only the experts the given routing rows use (plus the
    shared group E, kept last), and remap the indices onto that subset."""
    used = np.unique(idx.reshape(-1))
    groups = torch.as_tensor(np.concatenate([used, [E]]), dtype=torch.long)
    remap = {int(e): i for i, e in enumerate(used)}
    idx_sub = np.vectorize(lambda e: remap[int(e)])(idx).astype(np.int32)

    def take(name):
        t = weights[name]
        return t.index_select(0, groups.to(t.device)).cpu()

    if mode == "fp8":
        # fp32 originals, quantised by the oracle's own block codec
        ex = oracle.Experts.quantised(take("w_gate"), take("w_up"), take("w_down"))
    else:
        ex = oracle.Experts(mode, take("w_gate"), take("w_up"), take("w_down"))
    return ex, idx_sub


def sample_rows(T: int, n: int, seed: int = 0) -> np.ndarray:
    g = np.random.default_rng(seed)
    pick = {0, T - 1}
    while len(pick) < min(n, T):
        pick.add(int(g.integers(0, T)))
    return np.array(sorted(pick), np.int64)
