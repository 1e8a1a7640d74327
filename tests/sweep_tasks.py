"""Oracle side of the stated-rounds sweep: one task per workload family, run in the spawned
workers of oracle.parallel.OraclePool on a unit of sequences (one or more rounds stacked along
the batch axis, or a share of one large round).

Every input the oracle sees is a seeded input (logits, uniforms, temperatures) or its own
output: the draft tokens come from the oracle's draft sampler, the cache keys from its own
tokens, the Mirror branches from its own roots and sampler.  Nothing comes from the library.
"""
from __future__ import annotations

import numpy as np

import oracle

GROUP = 4   # sequences per oracle call: keeps each float64 temporary to a few rows of logits


def _grouped(fn, store, **kw):
    """fn over groups of GROUP sequences of the unit, outputs concatenated along the batch axis
    (sequences are independent, so this equals one call over the whole unit)."""
    n = store["target"].shape[0]
    parts = [fn({k: v[lo:lo + GROUP] for k, v in store.items()}, **kw) for lo in range(0, n, GROUP)]
    return {k: np.concatenate([p[k] for p in parts]) for k in parts[0]}


def _verify_round(store, K, F=0, C=1.0):
    """Draft sampling then verification (SSD notes §2.2; SpS notes §3), with sigma_{F,C} on the
    draft side when F > 0 and C < 1 (SSD notes §4.4)."""
    T, tp = store["T"], store["top_p"]
    tk = store.get("top_k")
    toks = oracle.draft_sample(store["draft"][:, :K], store["u_draft"][:, :K], T, tp, F, C, top_k=tk)["tokens"]
    r = oracle.verify(store["target"], store["draft"][:, :K], toks, store["u"], T, tp, F, C, top_k=tk)
    return {"tokens": toks, "accept_len": r["accept_len"], "out_tokens": r["out_tokens"]}


def _saguaro_round(store, K, F, C, f_int):
    """The Saguaro round: sigma_{F,C} draft tokens, verification with p', the top-F_k cache keys
    of every depth and the lookup of (k, t*) (SSD notes §4.4, §5.1; SSD abstract page, "Method")."""
    out = _verify_round(store, K, F, C)
    keys = oracle.cache_keys(store["draft"], out["tokens"], f_int)
    out["keys"] = keys
    out["hit"] = oracle.cache_lookup(out["accept_len"], out["out_tokens"], keys, f_int)
    return out


def _mirror_round(store, kappa, gamma):
    """The Mirror round: top-kappa roots of the early-exit row with their log-probabilities,
    branches drawn below them from the early-exit rows, verification along branch 0 and the
    reuse check (Mirror-SD notes §3.1-§3.2)."""
    ee, T = store["draft"], store["T"]
    B = ee.shape[0]
    ones = np.ones(B)
    rid, rlp = oracle.topk_rows(ee[:, 0], T, kappa)
    branches = np.zeros((B, kappa, gamma), dtype=np.int64)
    branches[:, :, 0] = rid
    for i in range(kappa):
        ub = store["u_branch"][:, i * gamma:(i + 1) * gamma]
        branches[:, i, 1:] = oracle.draft_sample(ee[:, 1:], ub[:, 1:], T, ones)["tokens"]
    r = oracle.verify(store["target"], ee, branches[:, 0, :], store["u"], T, ones)
    reuse = oracle.mirror_reuse(branches, r["accept_len"], r["out_tokens"])
    return {"roots": rid, "root_logprobs": rlp, "branches": branches, "accept_len": r["accept_len"],
            "out_tokens": r["out_tokens"], "reuse": reuse}


def verify_round(store, **kw):
    return _grouped(_verify_round, store, **kw)


def saguaro_round(store, **kw):
    return _grouped(_saguaro_round, store, **kw)


def mirror_round(store, **kw):
    return _grouped(_mirror_round, store, **kw)
