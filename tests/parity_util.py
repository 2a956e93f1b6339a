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


def full_size_rows(counts, offsets, T: int, k: int, n_largest: int = 5, max_out_largest: int = 256,
                   n_out: int = 64, seed: int = 0):
    """Rows to check at full size, from the GPU's own group counts/offsets.

    y rows (grouped layout): the first and last row of every touched routed
    group, every 128-row tile boundary (last row of one tile, first of the
    next) of the n_largest groups, every row of the largest group, and the
    first and last shared-expert row.  out rows (tokens): n_out sampled
    tokens plus the tokens routed to the largest group (a deterministic
    subsample of at most max_out_largest)."""
    E = len(counts) - 1
    c = np.asarray(counts[:E], np.int64)
    o = np.asarray(offsets[:E + 1], np.int64)
    y = set()
    for e in np.nonzero(c)[0]:
        y.update((int(o[e]), int(o[e] + c[e] - 1)))
    largest = np.argsort(-c, kind="stable")[:n_largest]
    for e in largest:
        for b in range(128, int(c[e]), 128):
            y.update((int(o[e] + b - 1), int(o[e] + b)))
    e0 = int(largest[0])
    y.update(range(int(o[e0]), int(o[e0] + c[e0])))
    y.update((T * k, T * k + T - 1))
    return np.array(sorted(y), np.int64), e0


def y_reference(y_rows, src_tok, offsets, T: int, k: int, x, weights: dict, mode: str, E: int):
    """Oracle expert outputs for grouped rows: a row of routed group e holds
    expert e applied to token src_tok[row]; a shared row T*k + t holds the
    shared expert applied to token t.  Each routed row is one oracle token
    with top_k = 1 (its expert, weight 1), whose second output slot is the
    shared expert of that token."""
    o = np.asarray(offsets[:E + 1], np.int64)
    rows = np.asarray(y_rows, np.int64)
    routed = rows[rows < T * k]
    shared = rows[rows >= T * k]
    tok = np.asarray(src_tok, np.int64)[routed]
    grp = np.searchsorted(o, routed, side="right") - 1
    # shared rows ride on a routed pair of the same token when there is one
    extra = [t for t in (shared - T * k) if t not in set(tok.tolist())]
    tok_all = np.concatenate([tok, np.asarray(extra, np.int64)])
    grp_all = np.concatenate([grp, np.zeros(len(extra), np.int64)])
    ex, idx_sub = experts_for_tokens(grp_all.reshape(-1, 1).astype(np.int32), weights, mode, E)
    xs = x[torch.as_tensor(tok_all, device=x.device)].cpu()
    _, yr = oracle.moe_tokens(xs, idx_sub, np.ones((len(tok_all), 1)), ex, want_y=True)
    ref = {}
    for i, r in enumerate(routed):
        ref[int(r)] = yr[i, 0]
    first = {}
    for i, t in enumerate(tok_all):
        first.setdefault(int(t), i)
    for r in shared:
        ref[int(r)] = yr[first[int(r - T * k)], 1]
    return ref
