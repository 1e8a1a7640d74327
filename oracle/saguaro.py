"""Saguaro speculation cache: geometric fan-out, cache keys and lookup (float64 / integer).

TEST INFRASTRUCTURE ONLY (see the package docstring).

SSD abstract page, "Method" (Theorem 12): with cache budget B_c = sum_k F_k, the fan-out
that maximises the hit probability under a power-law hit rate 1 - F^-r is
    F_k = F_0 * a^(k/(1+r))                         for k < K,
    F_K = F_0 * a^(K/(1+r)) * (1 - a)^(-1/(1+r)),
with a the draft acceptance rate.  SSD notes §5.1: at every depth k the cache holds the
top-F_k tokens of the draft logits, excluding the draft token already sent for
verification, as guesses for the bonus token; the cache maps outcomes (k, t*) to
speculations, and a lookup hits iff the actual outcome is a key (SSD abstract page).
"""
from __future__ import annotations

import math

import numpy as np

from .dist import order_desc


def fanout(budget: float, a: float, r: float, K: int):
    """Theorem 12 fan-out.  Returns (F_real [K+1] float64, F_int [K+1] int64).

    F_real sums to the budget.  F_int is the integer allocation used for the keys:
    floor(F_real) plus one extra slot for each of the largest remainders (ties to the
    smaller depth) until it sums to floor(budget).
    """
    e = 1.0 / (1.0 + r)
    shape = [a ** (k * e) for k in range(K)] + [a ** (K * e) * (1.0 - a) ** (-e)]
    f0 = budget / math.fsum(shape)
    f_real = np.array([f0 * s for s in shape], dtype=np.float64)
    f_int = np.floor(f_real).astype(np.int64)
    deficit = int(math.floor(budget)) - int(f_int.sum())
    rem = f_real - np.floor(f_real)
    by_rem = sorted(range(K + 1), key=lambda k: (-rem[k], k))
    for k in by_rem[:max(deficit, 0)]:
        f_int[k] += 1
    return f_real, f_int


def cache_keys(draft, tokens, f_int):
    """Cache keys per sequence, depth-major: keys[b, off_k + i] for i < F_k, off_k = sum_{j<k} F_j.

    Depth k < K: the top-(F_k) tokens of the draft row at position k+1 (ranked by raw
    draft logit, lowest id on ties) after removing s_{k+1}, the token that position
    proposed.  Depth K: the top-F_K tokens of the draft row at position K+1.
    draft: [B, K+1, V] raw draft logits; tokens: [B, K]; f_int: [K+1].
    Slots without a candidate (tiny V) hold -1.
    """
    draft = np.asarray(draft, dtype=np.float64)
    tokens = np.asarray(tokens, dtype=np.int64)
    f_int = [int(f) for f in f_int]
    B, _, V = draft.shape
    K = len(f_int) - 1
    keys = np.full((B, sum(f_int)), -1, dtype=np.int64)
    off = 0
    for k in range(K + 1):
        fk = f_int[k]
        order = order_desc(draft[:, k, :])
        for b in range(B):
            if k < K:
                cand = [int(t) for t in order[b, : fk + 1] if int(t) != int(tokens[b, k])][:fk]
            else:
                cand = [int(t) for t in order[b, :fk]]
            keys[b, off: off + len(cand)] = cand
        off += fk
    return keys


def cache_lookup(accept_len, out_tokens, keys, f_int):
    """hit[b] = 1 iff the outcome (k, t*) = (accept_len[b], out_tokens[b, k]) is a cache key,
    i.e. t* is among the depth-k keys of sequence b."""
    accept_len = np.asarray(accept_len, dtype=np.int64)
    out_tokens = np.asarray(out_tokens, dtype=np.int64)
    keys = np.asarray(keys, dtype=np.int64)
    f_int = [int(f) for f in f_int]
    offs = np.concatenate([[0], np.cumsum(f_int)])
    hit = np.zeros(len(accept_len), dtype=np.uint8)
    for b, k in enumerate(accept_len):
        t = out_tokens[b, k]
        seg = keys[b, offs[k]: offs[k] + f_int[k]]
        hit[b] = 1 if t in set(int(v) for v in seg) else 0
    return hit
