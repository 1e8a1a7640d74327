"""CPU checks of the oracle's process pool and of the stated-rounds sweep's bookkeeping.

The pool must return exactly what the oracle returns in-process (the rows reach the workers as
raw bits and are widened there), and the sweep must count a mismatch wherever the two sides
differ, whichever way it stacks rounds into units or splits a large round across workers.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.parallel import OraclePool, exact_f64, split_ranges
from synth import workloads as W
from tests import sweep_rounds as SR
from tests import sweep_tasks as ST


def test_exact_f64_widens_bf16_and_f32_bits_exactly():
    x = torch.randn(4096, dtype=torch.float32) * 30
    x[:4] = torch.tensor([float("-inf"), 0.0, -0.0, 3.0e38])
    b = x.to(torch.bfloat16)
    got = exact_f64(b.view(torch.int16).numpy().view(np.uint16), "bf16")
    np.testing.assert_array_equal(got, b.to(torch.float64).numpy())
    np.testing.assert_array_equal(exact_f64(x.numpy(), "f32"), x.to(torch.float64).numpy())


def test_split_ranges_cover_every_item_once():
    for n, parts in ((512, 16), (5, 16), (37, 4), (1, 1)):
        r = split_ranges(n, parts)
        assert r[0][0] == 0 and r[-1][1] == n and len(r) == min(n, parts)
        assert all(a[1] == b[0] for a, b in zip(r, r[1:]))


@pytest.fixture(scope="module")
def pool():
    with OraclePool(2) as p:
        yield p


def _store(w, r):
    tgt, drf = W.logits(w, r)
    u_draft, u, u_branch = W.round_uniforms(w, r)
    return {"target": SR.raw(tgt), "draft": SR.raw(drf), "u": (u, None), "T": (W.temperatures(w), None),
            "top_p": (W.top_ps(w), None), "u_draft": (u_draft, None), "u_branch": (u_branch, None)}


def _f64(store):
    return {k: exact_f64(a, kind) if kind else a for k, (a, kind) in store.items()}


def test_pool_verify_equals_the_oracle_in_process(pool):
    w = W.scaled(W.LARGE_BATCH, B=12, V=777)
    s = _store(w, 0)
    parts = [SR._slice(s, lo, hi) for lo, hi in split_ranges(w.B, 2)]
    pool.load(parts)
    pool.run("oracle.parallel:draft_tokens", {"K": w.K})
    outs, secs = pool.run("oracle.parallel:verify_chunk", {"K": w.K})
    assert secs > 0
    f = _f64(s)
    toks = oracle.draft_sample(f["draft"][:, :w.K], f["u_draft"][:, :w.K], f["T"], f["top_p"])["tokens"]
    ref = oracle.verify(f["target"], f["draft"], toks, f["u"], f["T"], f["top_p"])
    np.testing.assert_array_equal(np.concatenate([o["accept_len"] for o in outs]), ref["accept_len"])
    np.testing.assert_array_equal(np.concatenate([o["out_tokens"] for o in outs]), ref["out_tokens"])


def _fake_round(plant=None):
    """A stand-in for the GPU round: the same store, with "GPU" outputs computed by the oracle
    in this process (so they must match), optionally with one planted difference."""
    def fn(cfg, w, r, dev, ws, tally):
        s = _store(w, r)
        task, kw = SR._task(cfg, w)
        out = getattr(ST, task.split(":")[1])(_f64(s), **kw)
        if plant is not None and r == plant[0]:
            out[plant[1]] = out[plant[1]].copy()
            out[plant[1]].reshape(-1)[plant[2]] += 1
        for k in SR.STAT_KEYS:
            tally[k] = tally.get(k, 0)
        return out, s
    return fn


CASES = [(1, W.scaled(W.PLAIN, V=300)),                                  # many rounds stacked per unit
         (2, W.scaled(W.SAMPLED_TOPP, V=300)),                           # top-p, stacked
         (3, W.scaled(W.SAGUARO, B=4, V=300)),                           # sigma, keys, lookup
         (4, W.scaled(W.MIRROR, V=300)),                                 # roots, branches, reuse
         (5, W.scaled(W.LARGE_BATCH, B=80, V=300))]                      # one round split over units


@pytest.mark.parametrize("cfg,w", CASES, ids=[str(c) for c, _ in CASES])
def test_sweep_counts_no_mismatch_when_both_sides_agree(pool, cfg, w):
    res = SR.sweep_config(cfg, 7, pool, dev="cpu", w=w, round_fn=_fake_round())
    assert res["mismatches"] == 0, res
    assert res["sequences"] == 7 * w.B
    assert res["decisions_oracle"] > 0


@pytest.mark.parametrize("cfg,w,field", [(5, CASES[4][1], "accept_len"), (2, CASES[1][1], "out_tokens"),
                                         (3, CASES[2][1], "keys"), (4, CASES[3][1], "branches"),
                                         (1, CASES[0][1], "tokens")])
def test_sweep_counts_a_planted_mismatch(pool, cfg, w, field):
    res = SR.sweep_config(cfg, 5, pool, dev="cpu", w=w, round_fn=_fake_round(plant=(3, field, 1)))
    assert res["mismatches"] == 1, res
