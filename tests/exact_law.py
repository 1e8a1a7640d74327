"""Exact outcome law of a verify function, found by treating it as a black box.

For one sequence with fixed logits and draft tokens, a verify rule is a function of its
uniforms.  Each accept test is a threshold rule in its own uniform, and the residual draw
is a non-decreasing step function of the last uniform.  This helper locates those
thresholds and steps by bisection on the uniforms, so the outcome probabilities it
returns are exact up to the bisection width (~1e-15) and come from the function's
behaviour, not from its formulas.
"""
from __future__ import annotations

from collections import defaultdict
from itertools import product

import numpy as np

_ITERS = 60


def _call(verify, target, draft, tokens, u, T, top_p, F, C):
    r = verify(target[None], draft[None], np.asarray(tokens)[None], np.asarray(u)[None],
               np.array([T]), np.array([top_p]), F, C)
    k = int(r["accept_len"][0])
    return k, tuple(int(t) for t in r["out_tokens"][0, : k + 1])


def _accept_threshold(verify, args, K, j):
    """Largest u_j (as a limit) for which position j (0-based) is accepted, with earlier
    positions forced to accept (u = 0) and later ones irrelevant."""
    def accepted(uj):
        u = [0.0] * K + [0.5]
        u[j] = uj
        k, _ = _call(verify, *args[:3], u, *args[3:])
        return k > j
    if not accepted(0.0):
        return 0.0
    lo, hi = 0.0, 1.0
    if accepted(np.nextafter(1.0, 0.0)):
        return 1.0
    for _ in range(_ITERS):
        mid = 0.5 * (lo + hi)
        if accepted(mid):
            lo = mid
        else:
            hi = mid
    return hi


def _draw_law(verify, args, K, k):
    """Law of the drawn token when exactly k tokens are accepted: {token: probability}."""
    u_base = [0.0] * K + [0.0]
    if k < K:
        u_base[k] = np.nextafter(1.0, 0.0)

    def token(ur):
        u = list(u_base)
        u[K] = ur
        kk, toks = _call(verify, *args[:3], u, *args[3:])
        assert kk == k, (kk, k)
        return toks[-1]

    law = {}
    lo_u = 0.0
    cur = token(0.0)
    top = np.nextafter(1.0, 0.0)
    while True:
        if token(top) == cur:
            law[cur] = law.get(cur, 0.0) + (1.0 - lo_u)
            break
        lo, hi = lo_u, top
        for _ in range(_ITERS):
            mid = 0.5 * (lo + hi)
            if token(mid) == cur:
                lo = mid
            else:
                hi = mid
        law[cur] = law.get(cur, 0.0) + (hi - lo_u)
        lo_u = hi
        cur = token(hi)
    return law


def outcome_law(verify, target, draft, draft_probs, T=1.0, top_p=1.0, F=0, C=1.0):
    """{(k, committed tokens): probability} for draft tokens s_j ~ draft_probs[j]
    independently and all uniforms i.i.d. U[0, 1).

    target: [K+1, V] logits; draft: [K or K+1, V] logits; draft_probs: [K, V] the law of
    the draft tokens (the draft distribution the verify rule is meant to correct).
    """
    K = target.shape[0] - 1
    V = target.shape[1]
    law = defaultdict(float)
    for s in product(range(V), repeat=K):
        w = float(np.prod([draft_probs[j][s[j]] for j in range(K)])) if K else 1.0
        if w == 0.0:
            continue
        args = (target, draft, s, T, top_p, F, C)
        thr = [_accept_threshold(verify, args, K, j) for j in range(K)]
        reach = 1.0
        for k in range(K + 1):
            p_k = reach * ((1.0 - thr[k]) if k < K else 1.0)
            if p_k > 0.0:
                for t, pt in _draw_law(verify, args, K, k).items():
                    law[(k, tuple(s[:k]) + (t,))] += w * p_k * pt
            if k < K:
                reach *= thr[k]
    return dict(law)


def position_marginals(law, K, V):
    """P(position i exists and holds token v) for i = 0..K, and P(position i exists)."""
    joint = np.zeros((K + 1, V))
    for (k, toks), pr in law.items():
        for i, t in enumerate(toks):
            joint[i, t] += pr
    return joint, joint.sum(axis=1)


def sample_law(sample, V):
    """Law of a one-uniform sampler u -> token id that is non-decreasing in u (an inverse-CDF
    draw in id order), found by bisection on u: {token: probability} as a length-V array."""
    law = np.zeros(V)
    lo_u = 0.0
    top = np.nextafter(1.0, 0.0)
    cur = sample(0.0)
    while True:
        if sample(top) == cur:
            law[cur] += 1.0 - lo_u
            return law
        lo, hi = lo_u, top
        for _ in range(_ITERS):
            mid = 0.5 * (lo + hi)
            if sample(mid) == cur:
                lo = mid
            else:
                hi = mid
        law[cur] += hi - lo_u
        lo_u = hi
        cur = sample(hi)
