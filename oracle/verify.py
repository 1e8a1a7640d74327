"""Speculative-decoding verification and draft sampling in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The rule (SSD notes §2.2 steps ①-④; SpS notes §3): the target scores K+1 positions.
Draft token s_i is accepted with probability min(1, q_i(s_i) / p_i(s_i)), in order; the
first rejection ends the scan.  At the first rejection, at position k+1, the bonus token t*
is drawn from the residual (q_{k+1} - p_{k+1})_+ normalised by its sum; if all K are
accepted, t* is drawn from q_{K+1}.  1..K+1 tokens are committed.

Greedy sequences (temperature 0; Mirror-SD notes §2 step 3): accept the longest prefix whose
tokens equal the target argmax; the correction (or the bonus) is the target argmax at the
next position.  No uniforms are consumed; their slots stay reserved.

Randomness is an input: uniforms u[b, i] (i < K) decide the accept tests (accept iff
u < min(1, q/p)) and u[b, K] the residual / bonus draw (``inverse_cdf``).
"""
from __future__ import annotations

import numpy as np

from .dist import argmax_first, inverse_cdf, row_distribution, saguaro_transform


def _acceptance_ratio(q_s, p_s):
    """min(1, q/p) with p = 0 read as ratio 1 when q > 0 and 0 when q = 0."""
    with np.errstate(divide="ignore", invalid="ignore"):
        raw = np.where(p_s > 0.0, q_s / np.where(p_s > 0.0, p_s, 1.0), np.where(q_s > 0.0, np.inf, 0.0))
    return raw, np.minimum(1.0, raw)


def verify(target, draft, tokens, uniforms, temperature, top_p, saguaro_F=0, saguaro_C=1.0, top_k=None):
    """Verify B sequences.

    target:  [B, K+1, V] float64 target logits for positions 1..K+1.
    draft:   [B, >=K, V] float64 draft logits (rows 1..K are used).
    tokens:  [B, K] draft tokens s_1..s_K.
    uniforms:[B, K+1] float64 in [0, 1): K accept tests then the residual draw.
    temperature, top_p: [B] per sequence, applied to both q and p.
    top_k: [B] per sequence or None (<= 0 or >= V: off), applied to both q and p before
      top-p (SpS notes §3: the filters act on each distribution before the correction).
    saguaro_F, saguaro_C: the draft-side sigma_{F,C} transform applied to every draft row
      (F = 0 or C = 1: none).  Verification must use the transformed p for losslessness
      (SSD notes §3.2).

    Returns a dict with accept_len [B], out_tokens [B, K+1] (-1 padded), and per-position
    debug values: lse_q [B, K+1], lse_p [B, K], q_s [B, K], p_s [B, K], ratio [B, K]
    (the unclipped q/p), residual_mass [B] (R of the draw), mass_q/mass_p (nucleus masses).
    """
    target = np.asarray(target, dtype=np.float64)
    draft = np.asarray(draft, dtype=np.float64)
    tokens = np.asarray(tokens, dtype=np.int64)
    u = np.asarray(uniforms, dtype=np.float64)
    B, K1, V = target.shape
    K = K1 - 1
    T = np.asarray(temperature, dtype=np.float64).reshape(B)
    tp = np.asarray(top_p, dtype=np.float64).reshape(B)
    tk = np.zeros(B, np.int64) if top_k is None else np.asarray(top_k, dtype=np.int64).reshape(B)
    greedy = T == 0.0

    q, lse_q, mass_q = row_distribution(target, T[:, None], tp[:, None], tk[:, None])
    p, lse_p, mass_p = row_distribution(draft[:, :K, :], T[:, None], tp[:, None], tk[:, None])
    if saguaro_F > 0 and saguaro_C != 1.0:
        p_sag, _, _ = saguaro_transform(p, draft[:, :K, :], saguaro_F, saguaro_C)
        p = np.where(greedy[:, None, None], p, p_sag)

    idx = tokens[:, :, None]
    q_s = np.take_along_axis(q[:, :K, :], idx, axis=-1)[..., 0]
    p_s = np.take_along_axis(p, idx, axis=-1)[..., 0]
    ratio, r = _acceptance_ratio(q_s, p_s)
    acc_sampled = u[:, :K] < r
    acc_greedy = tokens == argmax_first(target[:, :K, :])
    acc = np.where(greedy[:, None], acc_greedy, acc_sampled)
    # k = length of the accepted prefix (first rejection ends the scan)
    k = np.sum(np.cumprod(acc, axis=1), axis=1).astype(np.int64)

    rows = np.arange(B)
    q_next = q[rows, k, :]                                   # q_{k+1}
    p_next = p[rows, np.minimum(k, K - 1), :] if K > 0 else np.zeros((B, V))
    w = np.where((k < K)[:, None], np.maximum(q_next - p_next, 0.0), q_next)
    r_mass = np.sum(w, axis=-1)
    w = np.where((r_mass > 0.0)[:, None], w, q_next)         # degenerate residual: fall back to q
    t_draw, R = inverse_cdf(w, u[:, K])
    t_greedy = argmax_first(target[rows, k, :])
    t_star = np.where(greedy, t_greedy, t_draw)

    out = np.full((B, K + 1), -1, dtype=np.int64)
    for b in range(B):
        out[b, : k[b]] = tokens[b, : k[b]]
        out[b, k[b]] = t_star[b]
    return dict(accept_len=k, out_tokens=out, lse_q=lse_q, lse_p=lse_p, q_s=q_s, p_s=p_s,
                ratio=ratio, residual_mass=np.where(greedy, np.nan, R), mass_q=mass_q,
                mass_p=mass_p)


def draft_sample(draft, uniforms, temperature, top_p, saguaro_F=0, saguaro_C=1.0, top_k=None):
    """Sample one draft token per row: s = inverse_cdf(p', u), with p' the draft
    distribution after temperature, top-k, top-p and sigma_{F,C} (SSD notes §4.4; SSD abstract
    page, "Method").  Temperature 0 rows take the argmax.

    draft: [B, R, V]; uniforms: [B, R]; temperature, top_p: [B]; top_k: [B] or None.
    Returns dict(tokens [B, R], p_top [B, R] (P_D), z_prime [B, R], lse [B, R]).
    """
    draft = np.asarray(draft, dtype=np.float64)
    B, R, V = draft.shape
    T = np.asarray(temperature, dtype=np.float64).reshape(B)
    tp = np.asarray(top_p, dtype=np.float64).reshape(B)
    tk = np.zeros(B, np.int64) if top_k is None else np.asarray(top_k, dtype=np.int64).reshape(B)
    p, lse, _ = row_distribution(draft, T[:, None], tp[:, None], tk[:, None])
    p2, p_d, zp = saguaro_transform(p, draft, saguaro_F, saguaro_C)
    t, _ = inverse_cdf(p2, np.asarray(uniforms, dtype=np.float64))
    greedy = (T == 0.0)[:, None]
    t = np.where(greedy, argmax_first(draft), t)
    return dict(tokens=t.astype(np.int64), p_top=p_d, z_prime=zp, lse=lse)
