"""Forming the target distribution q and the draft distribution p from logits (float64).

TEST INFRASTRUCTURE ONLY (see the package docstring).

SpS notes §3 and §6: temperature, nucleus (top-p) and top-k act on the draft and the
target distributions separately, before the acceptance ratio and the residual are formed.
SSD abstract page, "Method", and SSD notes §4.4: the Saguaro scheme sigma_{F,C} scales the
draft probabilities of the top-F tokens by C in [0, 1] and renormalises.

All arrays carry the vocabulary on the last axis; leading axes are independent rows.
"""
from __future__ import annotations

import numpy as np


def argmax_first(x):
    """Index of the largest logit, lowest id on ties (greedy decoding, Mirror-SD notes §2)."""
    return np.argmax(x, axis=-1)


def order_desc(x):
    """Token ids sorted by (logit descending, id ascending)."""
    return np.argsort(-x, axis=-1, kind="stable")


def softmax_t(x, temperature):
    """q = softmax(x / T) and its log-normaliser LSE = log sum_v exp(x_v / T).

    x: [..., V] float64; temperature: [...] > 0.
    """
    z = x / np.asarray(temperature, dtype=np.float64)[..., None]
    m = np.max(z, axis=-1, keepdims=True)
    e = np.exp(z - m)
    s = np.sum(e, axis=-1, keepdims=True)
    return e / s, (m + np.log(s))[..., 0]


def nucleus(q, x, top_p):
    """Top-p filter: keep the shortest prefix of tokens, ordered by (probability descending,
    id ascending), whose cumulative mass reaches top_p; zero the rest and renormalise.

    The ordering uses the logits x, which order the tokens exactly as q does for T > 0.
    Returns (filtered q, kept-mass M, nucleus size n).
    """
    V = q.shape[-1]
    order = order_desc(x)
    q_sorted = np.take_along_axis(q, order, axis=-1)
    cum = np.cumsum(q_sorted, axis=-1)
    tp = np.asarray(top_p, dtype=np.float64)[..., None]
    n = np.minimum(np.sum(cum < tp, axis=-1) + 1, V)
    keep_sorted = np.arange(V) < n[..., None]
    keep = np.zeros(q.shape, dtype=bool)
    np.put_along_axis(keep, order, keep_sorted, axis=-1)
    mass = np.take_along_axis(cum, (n - 1)[..., None], axis=-1)[..., 0]
    return np.where(keep, q / mass[..., None], 0.0), mass, n


def top_k(q, x, k):
    """Top-k filter: keep the first k tokens in (probability descending, id ascending) order;
    zero the rest and renormalise.  k <= 0 or k >= V keeps every token.

    The ordering uses the logits x, which order the tokens exactly as q does for T > 0.
    Returns (filtered q, kept-mass M).
    """
    V = q.shape[-1]
    k = np.asarray(k, dtype=np.int64)[..., None]
    k = np.where((k <= 0) | (k >= V), V, k)
    order = order_desc(x)
    keep = np.zeros(q.shape, dtype=bool)
    np.put_along_axis(keep, order, np.arange(V) < k, axis=-1)
    mass = np.sum(np.where(keep, q, 0.0), axis=-1)
    return np.where(keep, q / mass[..., None], 0.0), mass


def row_distribution(x, temperature, top_p, top_k_=0):
    """The distribution a row of logits stands for, after temperature, top-k and top-p.

    temperature == 0 means greedy: the one-hot vector at the first argmax.
    top_k_ <= 0 or >= V means no top-k filter; top_p >= 1 means no nucleus filter.  With both
    on, top-k acts first and the nucleus is taken of the renormalised top-k distribution (the
    pages fix no order between the two filters; this is the common sampler order).
    Returns (dist [..., V], lse [...] (nan for greedy rows), kept mass [...] (the fraction of
    the unfiltered q that the filters keep)).
    """
    x = np.asarray(x, dtype=np.float64)
    T = np.broadcast_to(np.asarray(temperature, dtype=np.float64), x.shape[:-1])
    tp = np.broadcast_to(np.asarray(top_p, dtype=np.float64), x.shape[:-1])
    tk = np.broadcast_to(np.asarray(top_k_, dtype=np.int64), x.shape[:-1])
    greedy = T == 0.0
    safe_T = np.where(greedy, 1.0, T)
    q, lse = softmax_t(x, safe_T)
    mass = np.ones(x.shape[:-1])
    kf = (tk > 0) & (tk < x.shape[-1]) & ~greedy
    if np.any(kf):
        qk, mk = top_k(q, x, np.where(kf, tk, 0))
        q = np.where(kf[..., None], qk, q)
        mass = np.where(kf, mk, mass)
    filt = (tp < 1.0) & ~greedy
    if np.any(filt):
        qf, mf, _ = nucleus(q, x, np.where(filt, tp, 1.0))
        q = np.where(filt[..., None], qf, q)
        mass = np.where(filt, mass * mf, mass)
    if np.any(greedy):
        onehot = np.zeros(x.shape)
        np.put_along_axis(onehot, argmax_first(x)[..., None], 1.0, axis=-1)
        q = np.where(greedy[..., None], onehot, q)
        lse = np.where(greedy, np.nan, lse)
    return q, lse, mass


def saguaro_transform(p, x, F, C):
    """sigma_{F,C}: multiply the draft probabilities of the top-F tokens (ranked by draft
    logit, lowest id on ties) by C and renormalise (SSD notes §4.4, Theorem 15/19;
    SSD abstract page, "Method").  F = 0 or C = 1 is the identity.  When the scaled mass is
    zero (C = 0 and every token with mass lies in the top-F set) the transform is undefined
    and the row is left unchanged.

    Returns (p', P_D = mass of the top-F set before scaling, Z' = normaliser).
    """
    p = np.asarray(p, dtype=np.float64)
    lead = p.shape[:-1]
    if F <= 0 or C == 1.0:
        return p, np.zeros(lead), np.ones(lead)
    F = min(int(F), p.shape[-1])
    top = order_desc(x)[..., :F]
    factor = np.ones(p.shape)
    np.put_along_axis(factor, top, float(C), axis=-1)
    in_d = np.zeros(p.shape, dtype=bool)
    np.put_along_axis(in_d, top, True, axis=-1)
    p_d = np.sum(np.where(in_d, p, 0.0), axis=-1)
    scaled = p * factor
    z = np.sum(scaled, axis=-1)
    ok = z > 0.0
    out = np.where(ok[..., None], scaled / np.where(ok, z, 1.0)[..., None], p)
    return out, p_d, np.where(ok, z, 1.0)


def inverse_cdf(w, u):
    """Inverse-CDF draw in token-id order.

    t = the smallest id v with w_0 + ... + w_v > u * R, where R = w_0 + ... + w_{V-1} and
    both are running sums in id order.  If rounding leaves no such id, t is the last id
    with positive weight.  Returns (t, R).
    """
    w = np.asarray(w, dtype=np.float64)
    c = np.cumsum(w, axis=-1)
    r = c[..., -1]
    thr = np.asarray(u, dtype=np.float64) * r
    above = c > thr[..., None]
    t = np.argmax(above, axis=-1)
    none = ~np.any(above, axis=-1)
    if np.any(none):
        V = w.shape[-1]
        last = V - 1 - np.argmax((w > 0.0)[..., ::-1], axis=-1)
        t = np.where(none, last, t)
    return t, r
