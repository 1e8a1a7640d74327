"""Shared test helpers: workload inputs for both sides and oracle runs in chunks.

Inputs come from ``synth`` (seeded generators).  Draft tokens for the oracle comparison are
drawn by the oracle's own draft sampler, so nothing the oracle sees comes from the library.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from synth import workloads as W


def to_f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 copy of a float32 / bfloat16 tensor."""
    return t.detach().to("cpu").to(torch.float64).numpy()


def make_inputs(w: W.Workload, round_idx: int = 0, device="cuda", chunk: int = 32):
    """Logits (on `device`), uniforms, temperatures, top-p and oracle-drawn draft tokens."""
    tgt, drf = W.logits(w, round_idx, device=device)
    u_draft, u_ver, u_branch = W.round_uniforms(w, round_idx)
    T = W.temperatures(w)
    tp = W.top_ps(w)
    tk = W.top_ks(w)
    K = w.K
    toks = np.zeros((w.B, K), dtype=np.int64)
    for b0 in range(0, w.B, chunk):
        b1 = min(w.B, b0 + chunk)
        d64 = to_f64(drf[b0:b1, :K])
        r = oracle.draft_sample(d64, u_draft[b0:b1, :K], T[b0:b1], tp[b0:b1], w.saguaro_F, w.saguaro_C,
                                top_k=tk[b0:b1])
        toks[b0:b1] = r["tokens"]
    return dict(target=tgt, draft=drf, tokens=toks, u_draft=u_draft, u=u_ver, u_branch=u_branch, T=T, top_p=tp,
                top_k=tk)


def oracle_verify(inp, w: W.Workload, seqs=None, chunk: int = 16, F=None, C=None):
    """Run the oracle on the selected sequences (all by default); returns dict of arrays."""
    B = w.B
    seqs = np.arange(B) if seqs is None else np.asarray(seqs)
    F = w.saguaro_F if F is None else F
    C = w.saguaro_C if C is None else C
    parts = []
    for i in range(0, len(seqs), chunk):
        sel = seqs[i:i + chunk]
        tsel = torch.as_tensor(sel, device=inp["target"].device)
        t64 = to_f64(inp["target"].index_select(0, tsel))
        d64 = to_f64(inp["draft"].index_select(0, tsel)[:, : w.K])
        tk = inp["top_k"][sel] if "top_k" in inp else None
        parts.append(oracle.verify(t64, d64, inp["tokens"][sel], inp["u"][sel], inp["T"][sel], inp["top_p"][sel], F, C,
                                   top_k=tk))
    return {k: np.concatenate([p[k] for p in parts]) for k in parts[0]}


def gpu_args(inp, device="cuda"):
    return dict(draft_tokens=torch.as_tensor(inp["tokens"], dtype=torch.int32, device=device),
                uniforms=torch.as_tensor(inp["u"], dtype=torch.float64, device=device),
                temperature=torch.as_tensor(inp["T"], dtype=torch.float32, device=device))
