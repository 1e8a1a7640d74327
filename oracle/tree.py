"""Verification of a tree of drafted tokens, and the reuse check against a drafted tree, in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Mirror-SD notes §1.1 (tree drafts: the draft is a candidate tree that the target verifies in one
pass), §3.1 (branch-complete trees of kappa roots and depth gamma) and §3.2-§3.3 (the committed
prefix reuses the tree when it is one of the tree's paths; a node at depth 2 may hold several
branches).

A tree of N drafted tokens: node i (1..N) holds token tokens[i-1] and hangs below node
parents[i-1] in [0, i-1] (node 0 is the committed context).  Row i of the target and of the draft
logits is the distribution that follows node i; a node's children were drafted from the draft
distribution of its row.

Readings taken where the pages are silent:
  * greedy (temperature 0): from the root, move to the first child (lowest index) whose token
    is the target's argmax at the current node; the target argmax where no child matches is the
    correction;
  * sampled: the children of the current node are tested in index order by the rule of SpS notes
    §3 applied again after every rejection: child i passes with probability min(1, w_i(t)/p(t))
    where w_1 = q and w_{i+1} = (w_i - p)+ normalised.  In closed form w_i = (q - c_i p)+ / R(c_i)
    with R(c) = sum_v (q_v - c p_v)+, c_1 = 0 and c_{i+1} = c_i + R(c_i).  A passing child becomes
    the current node; when every child fails (or there is none) the token is drawn from
    w_{m+1} by the inverse CDF in id order.  The residual after a rejection never vanishes in exact
    arithmetic; if it does after rounding the draw falls back to q;
  * uniforms: u[b, i] is node i's test, u[b, 0] the final draw.
"""
from __future__ import annotations

import numpy as np

from .dist import argmax_first, inverse_cdf, row_distribution


def children_of(parents):
    """children[u] = nodes whose parent is u, in increasing index order (nodes are 1-based)."""
    N = len(parents)
    ch = [[] for _ in range(N + 1)]
    for i in range(1, N + 1):
        ch[int(parents[i - 1])].append(i)
    return ch


def tree_verify(target, draft, parents, tokens, uniforms, temperature):
    """Verify B token trees.

    target, draft: [B, N+1, V] logits (row i follows node i; draft rows of leaves are unused);
    parents, tokens: [B, N]; uniforms: [B, N+1]; temperature: [B] (0 = greedy).
    Returns dict(accept_len [B], out_tokens [B, N+1] (path tokens then the correction / bonus,
    -1 padded), path [B, N] (accepted node ids, -1 padded), residual_scale [B] (c of the draw)).
    """
    target = np.asarray(target, dtype=np.float64)
    draft = np.asarray(draft, dtype=np.float64)
    B, N1, V = target.shape
    N = N1 - 1
    T = np.asarray(temperature, dtype=np.float64).reshape(B)
    u = np.asarray(uniforms, dtype=np.float64)
    out = np.full((B, N + 1), -1, dtype=np.int64)
    path = np.full((B, N), -1, dtype=np.int64)
    acc_len = np.zeros(B, dtype=np.int64)
    scale = np.zeros(B)
    for b in range(B):
        ch = children_of(parents[b])
        tok = [None] + [int(t) for t in tokens[b]]
        greedy = T[b] == 0.0
        if not greedy:
            q_all, _, _ = row_distribution(target[b], T[b], 1.0)
            p_all, _, _ = row_distribution(draft[b], T[b], 1.0)
        node, k = 0, 0
        while True:
            if greedy:
                am = int(argmax_first(target[b, node]))
                nxt = next((c for c in ch[node] if tok[c] == am), None)
                if nxt is None:
                    out[b, k] = am
                    break
                path[b, k], out[b, k] = nxt, tok[nxt]
                node, k = nxt, k + 1
                continue
            q, p = q_all[node], p_all[node]
            c_cur, R_cur, nxt = 0.0, 1.0, None
            for c in ch[node]:
                t = tok[c]
                w_t = max(q[t] - c_cur * p[t], 0.0) / R_cur
                ratio = w_t / p[t] if p[t] > 0.0 else (np.inf if w_t > 0.0 else 0.0)
                if u[b, c] < min(1.0, ratio):
                    nxt = c
                    break
                c_new = c_cur + R_cur
                R_new = float(np.sum(np.maximum(q - c_new * p, 0.0)))
                if not R_new > 0.0:          # empty residual after rounding: draw from q
                    c_cur, R_cur = 0.0, 1.0
                    break
                c_cur, R_cur = c_new, R_new
            if nxt is not None:
                path[b, k], out[b, k] = nxt, tok[nxt]
                node, k = nxt, k + 1
                continue
            w = np.maximum(q - c_cur * p, 0.0)
            t_star, _ = inverse_cdf(w, u[b, 0])
            out[b, k] = int(t_star)
            scale[b] = c_cur
            break
        acc_len[b] = k
    return dict(accept_len=acc_len, out_tokens=out, path=path, residual_scale=scale)


def tree_reuse(parents, tokens, accept_len, out_tokens):
    """Mirror-SD notes §3.2: the committed prefix (the accept_len accepted tokens and the
    correction) reuses a drafted tree when it spells a path from the tree's root.  Returns, per
    sequence, the node where that path ends (1..N), or -1.  At every depth the first child
    (lowest index) holding the committed token is followed."""
    B = len(parents)
    res = np.full(B, -1, dtype=np.int64)
    for b in range(B):
        ch = children_of(parents[b])
        node = 0
        for t in out_tokens[b, : int(accept_len[b]) + 1]:
            nxt = next((c for c in ch[node] if int(tokens[b][c - 1]) == int(t)), None)
            if nxt is None:
                node = -1
                break
            node = nxt
        res[b] = node if node > 0 else -1
    return res
