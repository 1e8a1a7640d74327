"""Seeded synthetic workloads for the five verification configurations.

The logit recipes are the ones the configurations state: i.i.d. normal target logits,
optionally with a Zipf-ranked bias on a random set of tokens, and a draft (or early-exit)
row formed as a scaled copy of the target row plus fresh normal noise.  Logits are drawn
in float32 by ``torch`` from a generator seeded through Philox, then rounded (RNE) to the
storage dtype.  The values therefore depend on the device they are drawn on; a test that
compares two implementations draws once and copies the tensor to the other side.

Nothing here computes a probability, a ratio or a sample: the uniforms that the method
consumes come from ``synth.philox`` and are passed to both sides as inputs.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

from . import philox

# Tags for bulk-generator seeds (one per tensor role).
_TAG_TARGET, _TAG_DRAFT, _TAG_BIAS_IDS, _TAG_BIAS_PERM, _TAG_DRAFT_SPREAD = 1, 2, 3, 4, 5


@dataclass(frozen=True)
class Workload:
    """One verification configuration.

    rows_target = K+1 target positions; rows_draft = K (or K+1 when the draft row at
    position K+1 is needed for the depth-K cache keys).
    """
    name: str
    B: int
    K: int
    V: int
    dtype: str                   # "f32" or "bf16"
    temperature: float
    top_p: float
    rounds: int
    seed: int
    sigma: float                 # target logit std
    draft_scale: float
    draft_sigma: float
    zipf_bias: bool = False      # +4 * i^-1.1 on 50 random distinct tokens per row
    greedy_even_rows: bool = False
    draft_rows_extra: int = 0    # 1 when the draft also has a row at position K+1
    saguaro_F: int = 0
    saguaro_C: float = 1.0
    budget: float = 0.0
    accept_rate: float = 0.0
    power_r: float = 0.0
    kappa: int = 0               # Mirror-style: root candidates
    top_k: int = 0               # top-k filter (0: off)
    draft_sigma_spread: float = 0.0   # per drafter row, the noise sigma times U[1 - s, 1 + s]
    extra: dict = field(default_factory=dict)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def rows_draft(self) -> int:
        return self.K + self.draft_rows_extra


# The five configurations (sizes and recipes as stated for the workloads).
PLAIN = Workload("plain-sd B=1 K=4 V=32000 f32", B=1, K=4, V=32000, dtype="f32",
                 temperature=1.0, top_p=1.0, rounds=1000, seed=0, sigma=2.0,
                 draft_scale=0.8, draft_sigma=1.0)
SAMPLED_TOPP = Workload("sampled-sd B=8 K=5 V=128256 bf16 T=0.8 top-p=0.9", B=8, K=5, V=128256,
                        dtype="bf16", temperature=0.8, top_p=0.9, rounds=200, seed=1, sigma=3.0,
                        draft_scale=0.7, draft_sigma=1.5, zipf_bias=True)
SAGUARO = Workload("saguaro B=16 K=5 V=128256 bf16 F=8 C=0.3 budget=64", B=16, K=5, V=128256,
                   dtype="bf16", temperature=1.0, top_p=1.0, rounds=200, seed=2, sigma=3.0,
                   draft_scale=0.7, draft_sigma=1.5, zipf_bias=True, draft_rows_extra=1,
                   saguaro_F=8, saguaro_C=0.3, budget=64.0, accept_rate=0.7, power_r=1.0)
MIRROR = Workload("mirror B=4 kappa=8 gamma=7 V=151936 bf16", B=4, K=7, V=151936, dtype="bf16",
                  temperature=1.0, top_p=1.0, rounds=200, seed=3, sigma=3.0,
                  draft_scale=0.6, draft_sigma=1.5, zipf_bias=True, kappa=8)
LARGE_BATCH = Workload("large-batch B=512 K=5 V=128256 bf16 half-greedy", B=512, K=5, V=128256,
                       dtype="bf16", temperature=1.0, top_p=1.0, rounds=50, seed=4, sigma=3.0,
                       draft_scale=0.7, draft_sigma=1.5, zipf_bias=True, greedy_even_rows=True)

CONFIGS = {1: PLAIN, 2: SAMPLED_TOPP, 3: SAGUARO, 4: MIRROR, 5: LARGE_BATCH}

# One verification stage of three-model speculative decoding (PyramidSD notes: LLaMA-3 family,
# V = 128256; the qualifier accumulates l_Q = 25 tokens for the target, the draft model about
# half as many for the qualifier; tau_T = 0.5, tau_Q = 0.4).  The page runs one stream; a batch
# of 64 independent streams stands in for a serving batch.  The drafter's logits are a scaled
# copy of the verifier's plus noise whose scale varies from row to row (x U[0.1, 1.9]), so
# that confident and uncertain positions mix: about 83% of positions pass tau_T = 0.5 in the
# qualifier -> target stage and about 75% pass tau_Q = 0.4 in the draft -> qualifier stage.
PYRAMID_QT = Workload("pyramid qualifier->target B=64 K=25 V=128256 bf16 tau=0.5", B=64, K=25, V=128256,
                      dtype="bf16", temperature=1.0, top_p=1.0, rounds=50, seed=6, sigma=3.0,
                      draft_scale=0.8, draft_sigma=1.5, zipf_bias=True, draft_sigma_spread=0.9,
                      extra={"tau": 0.5})
PYRAMID_DQ = Workload("pyramid draft->qualifier B=64 K=12 V=128256 bf16 tau=0.4", B=64, K=12, V=128256,
                      dtype="bf16", temperature=1.0, top_p=1.0, rounds=50, seed=7, sigma=3.0,
                      draft_scale=0.75, draft_sigma=1.5, zipf_bias=True, draft_sigma_spread=0.9,
                      extra={"tau": 0.4})

# The sampled recipe with a top-k filter ahead of top-p (k = 50 is a common sampler setting;
# the pages name top-k without a value).
SAMPLED_TOPK = Workload("sampled-sd-topk B=8 K=5 V=128256 bf16 T=0.8 top-k=50 top-p=0.9", B=8, K=5, V=128256,
                        dtype="bf16", temperature=0.8, top_p=0.9, rounds=200, seed=5, sigma=3.0,
                        draft_scale=0.7, draft_sigma=1.5, zipf_bias=True, top_k=50)


def scaled(w: Workload, **kw) -> Workload:
    """The same recipe at other sizes (for tests that must finish in seconds)."""
    d = dict(w.__dict__)
    d.update(kw)
    return Workload(**d)


def _gen(seed: int, stream: int, round_idx: int, tag: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(philox.seed_words(seed, 4 + stream, round_idx, tag))
    return g


def logits(w: Workload, round_idx: int = 0, device="cpu"):
    """Target logits [B, K+1, V] and draft logits [B, rows_draft, V] in the workload dtype.

    For the Mirror-style workload the "draft" tensor holds the early-exit rows for depths
    1..gamma (gamma = K), formed from the final (target) rows at the same positions.
    """
    B, K, V = w.B, w.K, w.V
    rows_t = K + 1
    rows_d = w.rows_draft
    g_t = _gen(w.seed, 0, round_idx, _TAG_TARGET, device)
    tgt = torch.randn((B, rows_t, V), generator=g_t, device=device, dtype=torch.float32)
    tgt.mul_(w.sigma)
    if w.zipf_bias:
        n_bias = min(50, V)
        g_b = _gen(w.seed, 0, round_idx, _TAG_BIAS_IDS, device)
        keys = torch.rand((B * rows_t, V), generator=g_b, device=device, dtype=torch.float32)
        ids = keys.topk(n_bias, dim=1).indices            # a uniformly random ordered subset
        del keys
        rank = torch.arange(1, n_bias + 1, device=device, dtype=torch.float32)
        bias = 4.0 * rank.pow(-1.1)
        tgt.view(B * rows_t, V).scatter_add_(1, ids, bias.expand(B * rows_t, n_bias).contiguous())
    g_d = _gen(w.seed, 0, round_idx, _TAG_DRAFT, device)
    noise = torch.randn((B, rows_d, V), generator=g_d, device=device, dtype=torch.float32)
    src = tgt[:, :rows_d, :] if rows_d <= rows_t else torch.cat(
        [tgt, tgt[:, -1:, :].expand(B, rows_d - rows_t, V)], dim=1)
    if w.draft_sigma_spread > 0.0:
        g_s = _gen(w.seed, 0, round_idx, _TAG_DRAFT_SPREAD, device)
        f = torch.rand((B, rows_d, 1), generator=g_s, device=device, dtype=torch.float32)
        noise.mul_(f.mul_(2.0 * w.draft_sigma_spread).add_(1.0 - w.draft_sigma_spread))
    drf = noise.mul_(w.draft_sigma).add_(src, alpha=w.draft_scale)
    return tgt.to(w.torch_dtype), drf.to(w.torch_dtype)


def temperatures(w: Workload) -> np.ndarray:
    t = np.full(w.B, w.temperature, dtype=np.float32)
    if w.greedy_even_rows:
        t[0::2] = 0.0
    return t


def top_ps(w: Workload) -> np.ndarray:
    return np.full(w.B, w.top_p, dtype=np.float32)


def top_ks(w: Workload) -> np.ndarray:
    return np.full(w.B, w.top_k, dtype=np.int32)


def round_uniforms(w: Workload, round_idx: int = 0):
    """(u_draft [B, rows_draft], u_verify [B, K+1], u_branch [B, kappa*K]) as float64.

    u_verify[:, :K] are the accept tests for positions 1..K and u_verify[:, K] the
    residual / bonus draw.
    """
    u_draft = philox.uniforms(w.seed, philox.STREAM_DRAFT, round_idx, w.B, w.rows_draft)
    u_acc = philox.uniforms(w.seed, philox.STREAM_ACCEPT, round_idx, w.B, w.K)
    u_res = philox.uniforms(w.seed, philox.STREAM_RESIDUAL, round_idx, w.B, 1)
    u_branch = philox.uniforms(w.seed, philox.STREAM_BRANCH, round_idx, w.B, max(w.kappa, 1) * w.K)
    return u_draft, np.concatenate([u_acc, u_res], axis=1), u_branch
