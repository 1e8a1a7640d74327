"""Mirror-SD style early-exit roots and branch reuse (float64 / integer).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Mirror-SD notes §3.1: at the early-exit layer the LM head gives a distribution whose top-kappa
tokens, with their log-probabilities, are sent to the draft as branch roots; the draft
rolls out a depth-gamma path under every root.  §3.2: the target verifies along the chosen
path; when fewer than gamma tokens are accepted the committed prefix (accepted tokens,
then the correction) is reused iff it is a path of the pre-built tree.
"""
from __future__ import annotations

import numpy as np

from .dist import order_desc, softmax_t


def topk_rows(x, temperature, kappa):
    """Top-kappa token ids per row (logit descending, lowest id on ties) and their
    log-probabilities log softmax(x / T).  x: [R, V]; temperature: scalar or [R]."""
    x = np.asarray(x, dtype=np.float64)
    T = np.broadcast_to(np.asarray(temperature, dtype=np.float64), x.shape[:-1])
    ids = order_desc(x)[..., :kappa]
    _, lse = softmax_t(x, T)
    logp = np.take_along_axis(x, ids, axis=-1) / T[..., None] - lse[..., None]
    return ids.astype(np.int64), logp


def mirror_reuse(branches, accept_len, out_tokens):
    """reuse[b] = 1 iff k < gamma and the committed prefix (s_1..s_k, t*) equals the first
    k+1 tokens of some branch.  branches: [B, kappa, gamma]."""
    branches = np.asarray(branches, dtype=np.int64)
    accept_len = np.asarray(accept_len, dtype=np.int64)
    out_tokens = np.asarray(out_tokens, dtype=np.int64)
    B, kappa, gamma = branches.shape
    reuse = np.zeros(B, dtype=np.uint8)
    for b in range(B):
        k = int(accept_len[b])
        if k >= gamma:
            continue
        prefix = out_tokens[b, : k + 1]
        reuse[b] = 1 if np.any(np.all(branches[b, :, : k + 1] == prefix[None, :], axis=1)) else 0
    return reuse
