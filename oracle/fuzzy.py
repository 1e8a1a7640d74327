"""One verification stage of three-model speculative decoding, in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

"3-Model Speculative Decoding (PyramidSD)" notes, "Method" (key designs 1 and 2): a drafter's
tokens are checked by a verifier -- the qualifier for the draft model, the target for the
qualifier -- position by position, in one of two ways:

  * fuzzy acceptance (PSDF): position t passes while Div(P_verifier(x_t), P_drafter(x_t)) is at
    most a threshold tau (tau_Q for the first stage, tau_T for the second);
  * assisted acceptance (PSDA): the speculative-sampling test u < min(1, q/p) of SpS notes §3,
    but a rejected token is replaced by a sample of the verifier's own distribution rather
    than of the residual (q - p)+.

Readings taken where the page is silent:
  * Div is the Jensen-Shannon divergence with base-2 logarithms (values in [0, 1]): the page's
    thresholds (0.4, 0.5) lie in that range and tau = 0 then means the two distributions agree;
  * the first position that fails gets a token drawn from the verifier's distribution at that
    position (inverse CDF in id order with the last uniform, as in ``verify``), and when every
    position passes the verifier's next row gives the bonus token, as in speculative sampling;
  * temperature 0 makes both distributions one-hot (greedy), so Div is 0 when the two argmaxes
    agree and 1 when they do not.
"""
from __future__ import annotations

import numpy as np

from .dist import argmax_first, inverse_cdf, row_distribution


def jensen_shannon(q, p):
    """JS divergence in bits of distributions on the last axis: with m = (q + p) / 2,
    Div = (KL(q || m) + KL(p || m)) / 2, where 0 log 0 = 0."""
    q = np.asarray(q, dtype=np.float64)
    p = np.asarray(p, dtype=np.float64)
    m = 0.5 * (q + p)
    with np.errstate(divide="ignore", invalid="ignore"):
        tq = np.where(q > 0.0, q * np.log2(q / np.where(m > 0.0, m, 1.0)), 0.0)
        tp = np.where(p > 0.0, p * np.log2(p / np.where(m > 0.0, m, 1.0)), 0.0)
    return 0.5 * (np.sum(tq, axis=-1) + np.sum(tp, axis=-1))


def fuzzy_verify(verifier, drafter, tokens, uniforms, temperature, tau, mode="divergence"):
    """Verify B sequences of K drafted tokens against a verifier.

    verifier: [B, K+1, V] logits of the verifying model at positions 1..K+1.
    drafter:  [B, >=K, V] logits of the drafting model (rows 1..K are used).
    tokens:   [B, K] drafted tokens; uniforms: [B, K+1] (slot i < K: accept test of position
              i+1 in the assisted mode; slot K: the draw); temperature: [B] (0 = greedy).
    mode:     "divergence" (PSDF, threshold tau) or "assisted" (PSDA).

    Returns dict(accept_len [B], out_tokens [B, K+1] (-1 padded), div [B, K]).
    """
    verifier = np.asarray(verifier, dtype=np.float64)
    drafter = np.asarray(drafter, dtype=np.float64)
    tokens = np.asarray(tokens, dtype=np.int64)
    u = np.asarray(uniforms, dtype=np.float64)
    B, K1, V = verifier.shape
    K = K1 - 1
    T = np.asarray(temperature, dtype=np.float64).reshape(B)
    greedy = T == 0.0
    ones = np.ones((B, 1))
    q, _, _ = row_distribution(verifier, T[:, None], ones)
    p, _, _ = row_distribution(drafter[:, :K, :], T[:, None], ones)
    div = jensen_shannon(q[:, :K, :], p)
    if mode == "divergence":
        acc = div <= float(tau)
    elif mode == "assisted":
        idx = tokens[:, :, None]
        q_s = np.take_along_axis(q[:, :K, :], idx, axis=-1)[..., 0]
        p_s = np.take_along_axis(p, idx, axis=-1)[..., 0]
        with np.errstate(divide="ignore", invalid="ignore"):
            ratio = np.where(p_s > 0.0, q_s / np.where(p_s > 0.0, p_s, 1.0), np.where(q_s > 0.0, np.inf, 0.0))
        acc = np.where(greedy[:, None], tokens == argmax_first(verifier[:, :K, :]), u[:, :K] < np.minimum(1.0, ratio))
    else:
        raise ValueError(mode)
    k = np.sum(np.cumprod(acc, axis=1), axis=1).astype(np.int64)
    rows = np.arange(B)
    t_draw, _ = inverse_cdf(q[rows, k, :], u[:, K])
    t_star = np.where(greedy, argmax_first(verifier[rows, k, :]), t_draw)
    out = np.full((B, K + 1), -1, dtype=np.int64)
    for b in range(B):
        out[b, : k[b]] = tokens[b, : k[b]]
        out[b, k[b]] = t_star[b]
    return dict(accept_len=k, out_tokens=out, div=div)
