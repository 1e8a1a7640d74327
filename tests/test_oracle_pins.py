"""Pins of the float64 oracle against facts the pages and the mathematics fix.

Each test checks the oracle's behaviour (not a retyped formula) against: a worked example
printed on the pages, a closed form or optimality condition, a library routine, an exact
enumeration of the outcome law, or a large-sample statistic.
"""
import math

import numpy as np
import pytest
import scipy.optimize
import scipy.special
import scipy.stats

import oracle
from synth import philox
from tests.exact_law import outcome_law, position_marginals, sample_law


def softmax(x, T=1.0):
    return scipy.special.softmax(np.asarray(x, dtype=np.float64) / T, axis=-1)


# --------------------------------------------------------------------------------------
# Input generator
# --------------------------------------------------------------------------------------

def test_philox_known_answers():
    """Philox4x32-10 known-answer vectors published with the Random123 library."""
    cases = [
        ([0, 0, 0, 0], [0, 0], [0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8]),
        ([0xFFFFFFFF] * 4, [0xFFFFFFFF] * 2, [0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD]),
        ([0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344], [0xA4093822, 0x299F31D0],
         [0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1]),
    ]
    for ctr, key, want in cases:
        got = philox.philox4x32_10(np.array([ctr]), np.array(key))[0]
        assert [int(v) for v in got] == want


def test_uniforms_range_and_moments():
    u = philox.uniforms(7, philox.STREAM_ACCEPT, 3, 1000, 100)
    assert u.min() >= 0.0 and u.max() < 1.0
    assert abs(u.mean() - 0.5) < 0.005 and abs(u.var() - 1 / 12) < 0.002
    # different streams / rounds give different numbers
    assert not np.array_equal(u, philox.uniforms(7, philox.STREAM_RESIDUAL, 3, 1000, 100))


# --------------------------------------------------------------------------------------
# Distributions
# --------------------------------------------------------------------------------------

def test_softmax_and_lse_match_scipy():
    rng = np.random.default_rng(0)
    x = rng.normal(0, 3, size=(5, 1000))
    for T in (0.5, 0.8, 1.0, 2.0):
        q, lse = oracle.softmax_t(x, np.full(5, T))
        np.testing.assert_allclose(lse, scipy.special.logsumexp(x / T, axis=-1), rtol=0, atol=1e-12)
        np.testing.assert_allclose(q, softmax(x, T), rtol=1e-12, atol=1e-300)


def test_greedy_row_is_first_argmax():
    x = np.array([[1.0, 3.0, 3.0, -2.0], [5.0, 5.0, 5.0, 5.0]])
    d, lse, _ = oracle.row_distribution(x, 0.0, 1.0)
    np.testing.assert_array_equal(d, [[0, 1, 0, 0], [1, 0, 0, 0]])
    assert np.all(np.isnan(lse))


def test_nucleus_hand_examples():
    p = np.array([0.1, 0.5, 0.05, 0.3, 0.05])
    x = np.log(p)
    d, _, _ = oracle.row_distribution(x, 1.0, 0.75)          # {1, 3}: .5 + .3 >= .75
    np.testing.assert_allclose(d, [0, 0.625, 0, 0.375, 0], atol=1e-15)
    d, _, _ = oracle.row_distribution(x, 1.0, 0.85)          # {1, 3, 0}
    np.testing.assert_allclose(d, np.array([0.1, 0.5, 0, 0.3, 0]) / 0.9, atol=1e-15)
    d, _, _ = oracle.row_distribution(x, 1.0, 0.3)           # the top token alone
    np.testing.assert_allclose(d, [0, 1, 0, 0, 0], atol=1e-15)
    # equal probabilities: the lowest ids are kept
    d, _, _ = oracle.row_distribution(np.zeros(5), 1.0, 0.5)
    np.testing.assert_allclose(d, [1 / 3, 1 / 3, 1 / 3, 0, 0], atol=1e-15)
    # top_p = 1 is no filter, bit for bit
    y = np.random.default_rng(1).normal(size=(3, 50))
    a, _, _ = oracle.row_distribution(y, 0.7, 1.0)
    np.testing.assert_array_equal(a, oracle.softmax_t(y, np.full(3, 0.7))[0])


def test_nucleus_stops_at_the_prefix_that_reaches_top_p_exactly():
    """SpS notes §6: the nucleus is the shortest prefix whose mass reaches top_p.  With the dyadic
    masses (1/4, 1/2, 1/4) the prefix {1, 0} holds exactly 3/4, so top_p = 3/4 keeps those two
    tokens (2/3 and 1/3) and not the third; a hair above 3/4 needs all three."""
    q = np.array([[0.25, 0.5, 0.25]])
    x = np.log(q)
    d, m, n = oracle.nucleus(q, x, np.array([0.75]))
    np.testing.assert_array_equal(d, [[1 / 3, 2 / 3, 0.0]])
    assert m[0] == 0.75 and n[0] == 2
    d, m, n = oracle.nucleus(q, x, np.array([np.nextafter(0.75, 1.0)]))
    np.testing.assert_array_equal(d, q)
    assert m[0] == 1.0 and n[0] == 3


def test_top_k_hand_examples():
    """SpS notes §3: top-k acts on each distribution before the correction.  Probabilities
    (0.1, 0.4, 0.2, 0.2, 0.1): the plateaus at 0.2 and 0.1 are cut at the lowest ids."""
    p = np.array([0.1, 0.4, 0.2, 0.2, 0.1])
    x = np.log(p)
    cases = {1: [0, 1, 0, 0, 0], 2: [0, 2 / 3, 1 / 3, 0, 0], 3: [0, 0.5, 0.25, 0.25, 0],
             4: np.array([0.1, 0.4, 0.2, 0.2, 0]) / 0.9}
    for k, want in cases.items():
        d, _, m = oracle.row_distribution(x, 1.0, 1.0, k)
        np.testing.assert_allclose(d, want, atol=1e-15)
        assert m == pytest.approx([0.4, 0.6, 0.8, 0.9][k - 1], abs=1e-15)
    base = oracle.softmax_t(x[None], np.ones(1))[0][0]
    for k in (0, -1, 5, 99):                                   # off: no filter, bit for bit
        d, _, m = oracle.row_distribution(x, 1.0, 1.0, k)
        np.testing.assert_array_equal(d, base)
        assert m == 1.0
    # temperature first: at T = 1/2 the kept pair {1, 2} weighs 0.4^2 : 0.2^2
    d, _, _ = oracle.row_distribution(x, 0.5, 1.0, 2)
    np.testing.assert_allclose(d, [0, 0.8, 0.2, 0, 0], atol=1e-14)
    # greedy rows ignore the filter
    d, _, _ = oracle.row_distribution(x, 0.0, 1.0, 3)
    np.testing.assert_array_equal(d, [0, 1, 0, 0, 0])


def test_top_k_then_top_p_hand_examples():
    """With both filters, the nucleus is taken of the renormalised top-k distribution, so the
    order of the two filters shows in the result."""
    x = np.log(np.array([0.1, 0.4, 0.2, 0.2, 0.1]))
    # top-4 = (1/9, 4/9, 2/9, 2/9, 0): cumulative 4/9, 6/9, 8/9 >= 0.85 keeps {1, 2, 3}
    d, _, m = oracle.row_distribution(x, 1.0, 0.85, 4)
    np.testing.assert_allclose(d, [0, 0.5, 0.25, 0.25, 0], atol=1e-15)
    assert m == pytest.approx(0.8, abs=1e-15)
    # the nucleus of the unfiltered row at 0.85 needs 0.4 + 0.2 + 0.2 + 0.1
    d, _, _ = oracle.row_distribution(x, 1.0, 0.85)
    np.testing.assert_allclose(d, np.array([0.1, 0.4, 0.2, 0.2, 0]) / 0.9, atol=1e-15)
    # top-2 = (0, 2/3, 1/3, 0, 0): 2/3 >= 0.55 keeps the top token alone
    d, _, m = oracle.row_distribution(x, 1.0, 0.55, 2)
    np.testing.assert_array_equal(d, [0, 1, 0, 0, 0])
    assert m == pytest.approx(0.4, abs=1e-15)
    d, _, _ = oracle.row_distribution(x, 1.0, 0.55)
    np.testing.assert_allclose(d, [0, 2 / 3, 1 / 3, 0, 0], atol=1e-15)


def test_top_k_invariants_on_plateau_rows():
    """Rows of rounded logits (many ties): the kept set has min(k, V) tokens, no dropped token
    outranks a kept one, ties at the cut keep the lowest ids, and the kept tokens keep their
    relative probabilities.  k = 1 is the greedy one-hot."""
    rng = np.random.default_rng(21)
    V = 40
    x = np.round(rng.normal(0, 1.5, size=(60, V)))
    ks = rng.integers(1, V + 3, size=60)
    T = rng.uniform(0.3, 2.0, size=60)
    d, _, m = oracle.row_distribution(x, T, 1.0, ks)
    q = softmax(x / T[:, None])
    for i in range(60):
        keep = d[i] > 0
        assert keep.sum() == min(ks[i], V)
        assert d[i].sum() == pytest.approx(1.0, abs=1e-14)
        assert m[i] == pytest.approx(q[i][keep].sum(), abs=1e-14)
        np.testing.assert_allclose(d[i][keep], q[i][keep] / q[i][keep].sum(), rtol=1e-13)
        if keep.all():
            continue
        lo, hi = x[i][keep].min(), x[i][~keep].max()
        assert lo >= hi
        if lo == hi:
            assert np.flatnonzero(keep & (x[i] == lo)).max() < np.flatnonzero(~keep & (x[i] == lo)).min()
    d1, _, _ = oracle.row_distribution(x, T, 1.0, 1)
    g, _, _ = oracle.row_distribution(x, 0.0, 1.0)
    np.testing.assert_array_equal(d1, g)


def test_saguaro_under_top_k_hand_example():
    """sigma_{F,C} acts on the filtered draft distribution.  Top-2 of (0.1, 0.4, 0.2, 0.2, 0.1)
    keeps {1, 2} at (2/3, 1/3).  With F=1, C=0.5 the top token is halved: (1/3, 1/3) / (2/3) =
    (1/2, 1/2).  With F=3, C=0 every kept token is scaled to zero: the transform is undefined and
    the filtered row is sampled unchanged."""
    x = np.log(np.array([[[0.1, 0.4, 0.2, 0.2, 0.1]]]))
    one, tk = np.ones(1), np.array([2])
    for u, want in [(0.0, 1), (0.49, 1), (0.51, 2), (0.99, 2)]:
        r = oracle.draft_sample(x, np.array([[u]]), one, one, 1, 0.5, top_k=tk)
        assert r["tokens"][0, 0] == want
        assert r["p_top"][0, 0] == pytest.approx(2 / 3, abs=1e-15)
        assert r["z_prime"][0, 0] == pytest.approx(2 / 3, abs=1e-15)
    for u, want in [(0.0, 1), (0.66, 1), (0.67, 2), (0.99, 2)]:
        r = oracle.draft_sample(x, np.array([[u]]), one, one, 3, 0.0, top_k=tk)
        assert r["tokens"][0, 0] == want and r["z_prime"][0, 0] == 1.0


def test_saguaro_under_top_p_hand_example():
    """sigma_{F,C} acts on the nucleus of the draft row (SSD notes §4.4 with SpS notes §3).  At
    top_p = 0.75 the row (0.1, 0.4, 0.2, 0.2, 0.1) keeps {1, 2, 3}, cumulative 0.4, 0.6, 0.8, at
    (1/2, 1/4, 1/4).  F=1, C=1/4 quarters the top token: (1/8, 1/4, 1/4) / (5/8) = (0.2, 0.4, 0.4),
    P_D = 1/2, Z' = 5/8.  Scaling first and filtering after would give a different row: the scaled
    row (1, 1, 2, 2, 1) / 7 reaches 0.75 only with token 0 as well, keeping (1, 1, 2, 2, 0) / 6.
    F=2, C=0 zeroes tokens 1 and 2 and leaves token 3 alone (P_D = 3/4, Z' = 1/4)."""
    x = np.log(np.array([[[0.1, 0.4, 0.2, 0.2, 0.1]]]))
    one, tp = np.ones(1), np.array([0.75])
    for u, want in [(0.0, 1), (0.19, 1), (0.21, 2), (0.59, 2), (0.61, 3), (0.99, 3)]:
        r = oracle.draft_sample(x, np.array([[u]]), one, tp, 1, 0.25)
        assert r["tokens"][0, 0] == want, (u, r["tokens"])
        assert r["p_top"][0, 0] == pytest.approx(0.5, abs=1e-15)
        assert r["z_prime"][0, 0] == pytest.approx(0.625, abs=1e-15)
    for u in (0.0, 0.5, 0.99):
        r = oracle.draft_sample(x, np.array([[u]]), one, tp, 2, 0.0)
        assert r["tokens"][0, 0] == 3
        assert r["p_top"][0, 0] == pytest.approx(0.75, abs=1e-15)
        assert r["z_prime"][0, 0] == pytest.approx(0.25, abs=1e-15)
    # verification divides by the same p': p'(s) for s = 1, 2, 3 and the nucleus mass of p
    tgt = np.zeros((1, 2, 5))
    for s, want in [(1, 0.2), (2, 0.4), (3, 0.4)]:
        r = oracle.verify(tgt, x, np.array([[s]]), np.array([[0.5, 0.5]]), one, tp, 1, 0.25)
        assert r["p_s"][0, 0] == pytest.approx(want, abs=1e-15)
        assert r["mass_p"][0, 0] == pytest.approx(0.8, abs=1e-15)


def test_inverse_cdf_hand_example():
    w = np.array([0.1, 0.0, 0.3, 0.6])
    for u, want in [(0.0, 0), (0.0999, 0), (0.1, 2), (0.3999, 2), (0.4, 3), (0.999, 3)]:
        t, R = oracle.inverse_cdf(w, u)
        assert int(t) == want, (u, t)
        assert R == pytest.approx(1.0)


# --------------------------------------------------------------------------------------
# Theorem 19 worked example (SSD notes §4.4): F=2, C=47/147
# --------------------------------------------------------------------------------------

P_T = np.array([0.48, 0.48, 0.02, 0.02])
P_D = np.array([0.49, 0.49, 0.01, 0.01])
C19 = 47.0 / 147.0


def test_theorem19_transformed_draft():
    p2, p_top, zp = oracle.saguaro_transform(P_D, np.log(P_D), 2, C19)
    np.testing.assert_allclose(p2, [0.47, 0.47, 0.03, 0.03], rtol=0, atol=1e-15)
    assert p_top == pytest.approx(0.98, abs=1e-15)
    # acceptance alpha = sum min(p, q) is 0.98 before and after
    assert np.minimum(P_D, P_T).sum() == pytest.approx(0.98, abs=1e-15)
    assert np.minimum(p2, P_T).sum() == pytest.approx(0.98, abs=1e-15)


def _hit_given_reject(F, C):
    """P(cache hit | first draft token rejected) for the Theorem 19 rows, K = 1.

    For each draft token s, the verify rule's exact outcome law (black-box bisection) gives
    P(k=0, t*=v | s); the cache is the oracle's depth-0 keys (top-2 draft tokens excluding s).
    """
    tgt = np.log(np.stack([P_T, P_T]))
    drf = np.log(np.stack([P_D, P_D]))
    p_draft = oracle.saguaro_transform(P_D, np.log(P_D), F, C)[0] if F else P_D
    f_int = [2, 2]
    num = den = 0.0
    for s in range(4):
        keys = oracle.cache_keys(drf[None], np.array([[s]]), f_int)
        law_s = outcome_law(oracle.verify, tgt, drf, [np.eye(4)[s]], F=F, C=C)
        for (k, toks), pr in law_s.items():
            if k == 0:
                hit = oracle.cache_lookup([0], np.array([[toks[0], -1]]), keys, f_int)[0]
                den += p_draft[s] * pr
                num += p_draft[s] * pr * hit
    return num / den


def test_theorem19_hit_rate_rises_from_half_to_one():
    assert _hit_given_reject(0, 1.0) == pytest.approx(0.5, abs=1e-12)
    assert _hit_given_reject(2, C19) == pytest.approx(1.0, abs=1e-12)


# --------------------------------------------------------------------------------------
# Verification: exact outcome law (lossless, mass identities, accept-length law)
# --------------------------------------------------------------------------------------

@pytest.mark.parametrize("seed", [0, 1, 2])
def test_exact_law_is_target_law_V3_K2(seed):
    """Brute force on V=3, K=2: committed tokens follow q position by position
    (SSD notes §2.2: output law equals the target's autoregressive law)."""
    rng = np.random.default_rng(seed)
    tgt = rng.normal(0, 1.5, size=(3, 3))
    drf = 0.5 * tgt[:2] + rng.normal(0, 1.0, size=(2, 3))
    q, p = softmax(tgt), softmax(drf)
    law = outcome_law(oracle.verify, tgt, drf, p)
    assert sum(law.values()) == pytest.approx(1.0, abs=1e-12)
    joint, exists = position_marginals(law, 2, 3)
    # position 1 always exists and follows q_1; later positions follow q_i when present
    np.testing.assert_allclose(joint[0], q[0], atol=1e-12)
    for i in (1, 2):
        np.testing.assert_allclose(joint[i], exists[i] * q[i], atol=1e-12)
    # independence of consecutive committed tokens (rows do not depend on context here)
    pair = np.zeros((3, 3))
    for (k, toks), pr in law.items():
        if len(toks) >= 2:
            pair[toks[0], toks[1]] += pr
    alpha1 = np.minimum(p[0], q[0]).sum()
    np.testing.assert_allclose(pair, np.outer(np.minimum(p[0], q[0]) / alpha1, q[1]) * exists[1],
                               atol=1e-12)


@pytest.mark.parametrize("seed", [0, 1])
def test_exact_law_under_top_k_V4_K2(seed):
    """Brute force on V=4, K=2 with top-2 on both models: the committed tokens follow the
    top-2 target distribution, and tokens outside the target's top two never appear."""
    import functools
    rng = np.random.default_rng(40 + seed)
    tgt = rng.normal(0, 1.5, size=(3, 4))
    drf = 0.5 * tgt[:2] + rng.normal(0, 1.0, size=(2, 4))

    def top2(x):
        keep = np.zeros(x.shape, bool)
        for i, row in enumerate(x):
            keep[i, np.argsort(row)[-2:]] = True
        w = np.where(keep, softmax(x), 0.0)
        return w / w.sum(axis=-1, keepdims=True)

    q2, p2 = top2(tgt), top2(drf)
    verify = functools.partial(oracle.verify, top_k=np.array([2]))
    law = outcome_law(verify, tgt, drf, p2)
    assert sum(law.values()) == pytest.approx(1.0, abs=1e-12)
    joint, exists = position_marginals(law, 2, 4)
    np.testing.assert_allclose(joint[0], q2[0], atol=1e-12)
    for i in (1, 2):
        np.testing.assert_allclose(joint[i], exists[i] * q2[i], atol=1e-12)


@pytest.mark.parametrize("seed", [0, 1])
def test_exact_law_under_top_p_and_saguaro_V4_K2(seed):
    """Brute force on V=4, K=2 with top-p on both models and sigma_{F,C} on the draft: draft
    tokens drawn by draft_sample (its law read off by bisection on its uniform) and verified
    with the same p' commit tokens whose law, position by position, is that of sampling the
    target with the same nucleus and no transform (SSD notes §3.2: losslessness needs the
    verifier to use p')."""
    import functools
    rng = np.random.default_rng(80 + seed)
    tgt = rng.normal(0, 1.5, size=(3, 4))
    drf = 0.5 * tgt[:2] + rng.normal(0, 1.0, size=(2, 4))
    tp, F, C = 0.8, 1, 0.3
    one, tpa = np.ones(1), np.array([tp])

    def law_of(rows, F, C):
        return np.stack([sample_law(lambda u, row=row: int(oracle.draft_sample(
            row[None, None], np.array([[u]]), one, tpa, F, C)["tokens"][0, 0]), 4) for row in rows])

    p_draw = law_of(drf, F, C)
    q_want = law_of(tgt, 0, 1.0)
    # the nucleus really cuts and sigma really moves mass, on at least one row each
    assert np.any(q_want == 0.0) and np.any(p_draw == 0.0)
    assert not np.allclose(p_draw, law_of(drf, 0, 1.0), atol=1e-6)
    law = outcome_law(oracle.verify, tgt, drf, p_draw, top_p=tp, F=F, C=C)
    assert sum(law.values()) == pytest.approx(1.0, abs=1e-12)
    joint, exists = position_marginals(law, 2, 4)
    np.testing.assert_allclose(joint[0], q_want[0], atol=1e-12)
    for i in (1, 2):
        np.testing.assert_allclose(joint[i], exists[i] * q_want[i], atol=1e-12)
    # a verifier that divides by the untransformed nucleus is not lossless for these drafts
    plain = functools.partial(oracle.verify, saguaro_F=0, saguaro_C=1.0)
    bad = outcome_law(lambda t, d, s, u, T, p, F_, C_: plain(t, d, s, u, T, p), tgt, drf, p_draw,
                      top_p=tp)
    jb, _ = position_marginals(bad, 2, 4)
    assert np.abs(jb[0] - q_want[0]).max() > 1e-3


def test_mass_identities_single_position():
    """SpS notes §3: accepting gives token x the mass min(p, q); the total rejection
    probability is sum (q - p)_+; the residual draw gives (q - p)_+ and the two add to q."""
    rng = np.random.default_rng(5)
    V = 5
    tgt = rng.normal(0, 2, size=(2, V))
    drf = rng.normal(0, 2, size=(1, V))
    q, p = softmax(tgt), softmax(drf)
    law = outcome_law(oracle.verify, tgt, drf, p)
    acc = np.zeros(V)
    res = np.zeros(V)
    for (k, toks), pr in law.items():
        if k == 1:
            acc[toks[0]] += pr
        else:
            res[toks[0]] += pr
    np.testing.assert_allclose(acc, np.minimum(p[0], q[0]), atol=1e-13)
    np.testing.assert_allclose(res, np.maximum(q[0] - p[0], 0.0), atol=1e-13)
    assert res.sum() == pytest.approx(np.maximum(q[0] - p[0], 0).sum(), abs=1e-13)
    np.testing.assert_allclose(acc + res, q[0], atol=1e-13)


def test_accept_length_geometric_law():
    """SSD notes §4.3: with every position accepting at rate a, exactly j tokens are
    accepted with probability a^j (1 - a) for j < K and a^K for j = K."""
    rng = np.random.default_rng(9)
    row_t = rng.normal(0, 1.5, size=3)
    row_d = rng.normal(0, 1.5, size=3)
    K = 3
    tgt = np.stack([row_t] * (K + 1))
    drf = np.stack([row_d] * K)
    p = softmax(drf)
    a = np.minimum(softmax(row_t), softmax(row_d)).sum()
    law = outcome_law(oracle.verify, tgt, drf, p)
    pk = np.zeros(K + 1)
    for (k, _), pr in law.items():
        pk[k] += pr
    want = [a ** j * (1 - a) for j in range(K)] + [a ** K]
    np.testing.assert_allclose(pk, want, atol=1e-12)


def test_identical_draft_accepts_everything():
    rng = np.random.default_rng(3)
    B, K, V = 64, 4, 50
    tgt = rng.normal(0, 2, size=(B, K + 1, V))
    u = rng.random((B, K + 1))
    toks = rng.integers(0, V, size=(B, K))
    r = oracle.verify(tgt, tgt[:, :K], toks, u, np.ones(B), np.ones(B))
    assert np.all(r["accept_len"] == K)
    # the bonus token is the inverse CDF of q_{K+1} at the residual uniform
    q = softmax(tgt[:, K])
    want = [int(np.searchsorted(np.cumsum(q[b]), u[b, K] * np.cumsum(q[b])[-1], side="right"))
            for b in range(B)]
    np.testing.assert_array_equal(r["out_tokens"][:, K], want)


def test_single_token_vocabulary():
    B, K = 5, 3
    tgt = np.zeros((B, K + 1, 1))
    r = oracle.verify(tgt, tgt[:, :K], np.zeros((B, K), int), np.random.default_rng(0).random((B, K + 1)),
                      np.ones(B), np.ones(B))
    assert np.all(r["accept_len"] == K) and np.all(r["out_tokens"] == 0)


def test_identity_transforms_are_plain_verify():
    rng = np.random.default_rng(4)
    B, K, V = 16, 3, 40
    tgt = rng.normal(0, 2, size=(B, K + 1, V))
    drf = rng.normal(0, 2, size=(B, K, V))
    toks = rng.integers(0, V, size=(B, K))
    u = rng.random((B, K + 1))
    base = oracle.verify(tgt, drf, toks, u, np.ones(B), np.ones(B))
    for F, C in [(0, 0.3), (8, 1.0)]:
        other = oracle.verify(tgt, drf, toks, u, np.ones(B), np.ones(B), F, C)
        np.testing.assert_array_equal(base["out_tokens"], other["out_tokens"])
        np.testing.assert_array_equal(base["ratio"], other["ratio"])


def test_greedy_verify_hand_example():
    """Mirror-SD notes §2 step 3: longest prefix equal to the target argmax, then the
    target argmax as the correction."""
    V = 6
    tgt = np.full((1, 4, V), -1.0)
    for j, a in enumerate([2, 4, 1, 5]):
        tgt[0, j, a] = 3.0
    drf = np.zeros((1, 3, V))
    u = np.full((1, 4), 0.5)
    r = oracle.verify(tgt, drf, np.array([[2, 4, 0]]), u, np.zeros(1), np.ones(1))
    assert r["accept_len"][0] == 2 and list(r["out_tokens"][0]) == [2, 4, 1, -1]
    r = oracle.verify(tgt, drf, np.array([[2, 4, 1]]), u, np.zeros(1), np.ones(1))
    assert r["accept_len"][0] == 3 and list(r["out_tokens"][0]) == [2, 4, 1, 5]
    r = oracle.verify(tgt, drf, np.array([[0, 4, 1]]), u, np.zeros(1), np.ones(1))
    assert r["accept_len"][0] == 0 and list(r["out_tokens"][0]) == [2, -1, -1, -1]


@pytest.mark.parametrize("K", [1, 3])
def test_chi_square_committed_tokens_V8(K):
    """SpS notes §6: check the distribution with large-sample token statistics.
    10^6 sequences on V=8; committed tokens at every position against q, and the
    accept-length histogram against the product of per-position acceptance rates."""
    rng = np.random.default_rng(100 + K)
    V = 8
    row_t = rng.normal(0, 1.5, size=(K + 1, V))
    row_d = 0.6 * row_t[:K] + rng.normal(0, 1.0, size=(K, V))
    q, p = softmax(row_t), softmax(row_d)
    n_total, chunk = 1_000_000, 100_000
    counts = np.zeros((K + 1, V))
    klen = np.zeros(K + 1)
    for c in range(n_total // chunk):
        u_d = philox.uniforms(11, philox.STREAM_DRAFT, c, chunk, K)
        u_v = np.concatenate([philox.uniforms(11, philox.STREAM_ACCEPT, c, chunk, K),
                              philox.uniforms(11, philox.STREAM_RESIDUAL, c, chunk, 1)], axis=1)
        tgt = np.broadcast_to(row_t, (chunk, K + 1, V))
        drf = np.broadcast_to(row_d, (chunk, K, V))
        toks = oracle.draft_sample(drf, u_d, np.ones(chunk), np.ones(chunk))["tokens"]
        r = oracle.verify(tgt, drf, toks, u_v, np.ones(chunk), np.ones(chunk))
        k = r["accept_len"]
        klen += np.bincount(k, minlength=K + 1)
        for i in range(K + 1):
            present = k >= i
            counts[i] += np.bincount(r["out_tokens"][present, i], minlength=V)
    for i in range(K + 1):
        n = counts[i].sum()
        stat, pval = scipy.stats.chisquare(counts[i], n * q[i])
        assert pval > 0.01, (i, pval)
    a = np.minimum(p, q[:K]).sum(axis=1)
    want = np.array([np.prod(a[:j]) * (1 - a[j]) for j in range(K)] + [np.prod(a)])
    stat, pval = scipy.stats.chisquare(klen, n_total * want)
    assert pval > 0.01, pval


# --------------------------------------------------------------------------------------
# Theorem 12 fan-out (SSD abstract page, "Method")
# --------------------------------------------------------------------------------------

def _optimal_fanout(budget, a, r, K):
    """Maximise the hit probability sum_k P(k) (1 - F_k^-r) under sum_k F_k = budget, with
    the geometric accept-length law P(k) = a^k (1-a) (k < K), a^K (k = K)."""
    P = np.array([a ** k * (1 - a) for k in range(K)] + [a ** K])
    obj = lambda f: -np.sum(P * (1.0 - np.power(f, -r)))
    res = scipy.optimize.minimize(obj, np.full(K + 1, budget / (K + 1)), method="SLSQP",
                                  bounds=[(1e-6, budget)] * (K + 1),
                                  constraints=[{"type": "eq", "fun": lambda f: f.sum() - budget}],
                                  options={"ftol": 1e-15, "maxiter": 1000})
    return res.x


@pytest.mark.parametrize("budget,a,r,K", [(64, 0.7, 1.0, 5), (23, 0.8, 1.0, 5), (100, 0.5, 2.0, 3),
                                          (40, 0.9, 0.5, 4)])
def test_fanout_is_the_optimum_of_the_power_law_model(budget, a, r, K):
    f_real, f_int = oracle.fanout(budget, a, r, K)
    np.testing.assert_allclose(f_real, _optimal_fanout(budget, a, r, K), rtol=2e-4)
    assert f_real.sum() == pytest.approx(budget, rel=1e-14)
    assert f_int.sum() == math.floor(budget)
    assert np.all(np.abs(f_int - f_real) < 1.0)


def test_fanout_remainder_ties_go_to_the_smaller_depth():
    """a = 1/2, r = 0: the shape is (1, 1/2^k ..., 1/2^K * 2), so budget 3 at K = 1 splits
    (1.5, 1.5) and budget 6 at K = 2 splits (3, 1.5, 1.5).  The floors leave one slot, and
    equal remainders hand it to the smaller depth."""
    f_real, f_int = oracle.fanout(3.0, 0.5, 0.0, 1)
    np.testing.assert_array_equal(f_real, [1.5, 1.5])
    assert list(f_int) == [2, 1]
    f_real, f_int = oracle.fanout(6.0, 0.5, 0.0, 2)
    np.testing.assert_array_equal(f_real, [3.0, 1.5, 1.5])
    assert list(f_int) == [3, 2, 1]


def test_fanout_budget64_values():
    f_real, f_int = oracle.fanout(64.0, 0.7, 1.0, 5)
    np.testing.assert_allclose(f_real, [14.676, 12.279, 10.273, 8.595, 7.191, 10.985], atol=5e-4)
    assert list(f_int) == [15, 12, 10, 9, 7, 11]


# --------------------------------------------------------------------------------------
# Theorem 15 monotonicity (SSD notes §4.4)
# --------------------------------------------------------------------------------------

@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_hit_probability_monotone_in_C(seed):
    """p_hit rises as C falls: the share of the residual draw landing in the down-weighted
    top-F set, given a rejection, is non-increasing in C on a 21-point grid."""
    rng = np.random.default_rng(seed)
    V, F = 6, 2
    tgt = rng.normal(0, 1.5, size=(2, V))
    drf = 0.5 * tgt[:1] + rng.normal(0, 1.0, size=(1, V))
    top = set(np.argsort(-drf[0], kind="stable")[:F].tolist())
    prev = -1.0
    for C in np.linspace(0.0, 1.0, 21)[::-1]:
        p_draft = oracle.saguaro_transform(softmax(drf[0]), drf[0], F, C)[0]
        law = outcome_law(oracle.verify, tgt, drf, [p_draft], F=F, C=C)
        rej = sum(pr for (k, _), pr in law.items() if k == 0)
        hit = sum(pr for (k, t), pr in law.items() if k == 0 and t[0] in top)
        share = hit / rej
        assert share >= prev - 1e-12, (C, share, prev)
        prev = share


# --------------------------------------------------------------------------------------
# Cache keys, lookup, Mirror roots and reuse: hand examples
# --------------------------------------------------------------------------------------

def test_cache_keys_and_lookup_hand_example():
    # depth 0 uses draft row 1, excluding s_1; depth 1 (=K) uses draft row 2
    drf = np.array([[[0.0, 5.0, 5.0, 1.0, 4.0],
                     [3.0, 0.0, 2.0, 2.0, 1.0]]])
    keys = oracle.cache_keys(drf, np.array([[1]]), [2, 3])
    assert list(keys[0]) == [2, 4, 0, 2, 3]           # ties at 5.0 and 2.0 go to the lowest id
    keys2 = oracle.cache_keys(drf, np.array([[3]]), [2, 3])
    assert list(keys2[0][:2]) == [1, 2]
    hit = oracle.cache_lookup([0, 1, 0], np.array([[4, -1], [1, 3], [1, -1]]),
                              np.repeat(keys, 3, axis=0), [2, 3])
    assert list(hit) == [1, 1, 0]
    # k = 0 and t* = 0, the first depth-1 key: the depth-0 keys (2, 4) decide, so no hit
    assert oracle.cache_lookup([0], np.array([[0, -1]]), keys, [2, 3])[0] == 0


def test_topk_rows_and_reuse_hand_example():
    x = np.array([[1.0, 4.0, 4.0, 2.0, -1.0]])
    ids, logp = oracle.topk_rows(x, 1.0, 3)
    assert list(ids[0]) == [1, 2, 3]
    np.testing.assert_allclose(logp[0], np.log(softmax(x[0])[[1, 2, 3]]), atol=1e-14)
    br = np.array([[[5, 6, 7], [5, 8, 9], [3, 1, 1]]])
    assert oracle.mirror_reuse(br, [1], np.array([[5, 8, -1, -1]]))[0] == 1
    assert oracle.mirror_reuse(br, [1], np.array([[5, 2, -1, -1]]))[0] == 0
    assert oracle.mirror_reuse(br, [0], np.array([[3, -1, -1, -1]]))[0] == 1
    assert oracle.mirror_reuse(br, [3], np.array([[5, 6, 7, 1]]))[0] == 0    # k = gamma
    assert oracle.mirror_reuse(br, [2], np.array([[5, 8, 9, -1]]))[0] == 1   # k = gamma - 1: a whole branch
    # temperature first: at T = 1/2 the probabilities go as the squares (.01, .16, .04, .04, .01) / .26
    y = np.log(np.array([[0.1, 0.4, 0.2, 0.2, 0.1]]))
    ids, logp = oracle.topk_rows(y, 0.5, 3)
    assert list(ids[0]) == [1, 2, 3]
    np.testing.assert_allclose(logp[0], np.log(np.array([0.16, 0.04, 0.04]) / 0.26), atol=1e-14)


# --------------------------------------------------------------------------------------
# PyramidSD stage verification: Jensen-Shannon divergence, fuzzy and assisted acceptance
# --------------------------------------------------------------------------------------
def test_jensen_shannon_matches_scipy():
    """The divergence against scipy's Jensen-Shannon distance (squared, base 2), including
    distributions with zeros; identities: 0 on equal inputs, 1 on disjoint supports, symmetry."""
    import scipy.spatial.distance as ssd
    rng = np.random.default_rng(30)
    for V in (2, 7, 300):
        for _ in range(20):
            q = rng.random(V) ** 3
            p = rng.random(V) ** 3
            q[rng.random(V) < 0.2] = 0.0
            p[rng.random(V) < 0.2] = 0.0
            q[0] += 1e-3
            p[-1] += 1e-3
            q /= q.sum()
            p /= p.sum()
            want = ssd.jensenshannon(q, p, base=2) ** 2
            assert oracle.jensen_shannon(q, p) == pytest.approx(want, rel=1e-12, abs=1e-15)
            assert oracle.jensen_shannon(p, q) == pytest.approx(oracle.jensen_shannon(q, p), abs=1e-15)
            assert oracle.jensen_shannon(q, q) == pytest.approx(0.0, abs=1e-15)
    assert oracle.jensen_shannon([1.0, 0.0, 0.0], [0.0, 0.5, 0.5]) == pytest.approx(1.0, abs=1e-15)


def test_fuzzy_verify_hand_example():
    """Position 1: verifier and drafter agree (Div 0); position 2: disjoint one-token rows
    (Div 1).  tau = 0.5 accepts position 1 only, and position 2 takes the verifier's token."""
    ninf = -np.inf
    ver = np.array([[[0.0, 0.0, ninf], [ninf, 0.0, ninf], [0.0, ninf, ninf]]])
    drf = np.array([[[0.0, 0.0, ninf], [0.0, ninf, ninf]]])
    toks = np.array([[1, 0]])
    u = np.array([[0.9, 0.9, 0.3]])
    r = oracle.fuzzy_verify(ver, drf, toks, u, np.ones(1), 0.5)
    np.testing.assert_allclose(r["div"], [[0.0, 1.0]], atol=1e-15)
    assert r["accept_len"][0] == 1 and list(r["out_tokens"][0]) == [1, 1, -1]
    r = oracle.fuzzy_verify(ver, drf, toks, u, np.ones(1), 1.0)        # everything passes: bonus from row 3
    assert r["accept_len"][0] == 2 and list(r["out_tokens"][0]) == [1, 0, 0]
    r = oracle.fuzzy_verify(ver, drf, toks, u, np.ones(1), -0.1)       # nothing passes: draw from row 1
    assert r["accept_len"][0] == 0 and r["out_tokens"][0, 0] == 0       # u = 0.3 < 1/2 -> id 0


@pytest.mark.parametrize("seed", [0, 1])
def test_fuzzy_first_token_law(seed):
    """Exact outcome law (bisection on the uniforms): when Div <= tau the first committed token
    follows the drafter's distribution p (its token is kept whatever it is); otherwise it
    follows the verifier's q."""
    import functools
    rng = np.random.default_rng(50 + seed)
    ver = rng.normal(0, 1.5, size=(2, 4))
    drf = 0.5 * ver[:1] + rng.normal(0, 1.0, size=(1, 4))
    q, p = softmax(ver), softmax(drf)
    d = oracle.jensen_shannon(q[0], p[0])
    for tau, want in ((d + 1e-9, p[0]), (d - 1e-9, q[0])):
        fv = functools.partial(_fuzzy_as_verify, tau=tau, mode="divergence")
        law = outcome_law(fv, ver, drf, p)
        joint, _ = position_marginals(law, 1, 4)
        np.testing.assert_allclose(joint[0], want, atol=1e-12)


@pytest.mark.parametrize("seed", [0, 1])
def test_assisted_first_token_law(seed):
    """Assisted acceptance: accepting gives min(p, q); a rejection (probability 1 - sum min(p, q))
    draws from q itself, so the first token's law is min(p, q) + (1 - alpha) q (not q)."""
    import functools
    rng = np.random.default_rng(60 + seed)
    ver = rng.normal(0, 1.5, size=(2, 5))
    drf = rng.normal(0, 1.5, size=(1, 5))
    q, p = softmax(ver), softmax(drf)
    alpha = np.minimum(p[0], q[0]).sum()
    fv = functools.partial(_fuzzy_as_verify, tau=0.0, mode="assisted")
    law = outcome_law(fv, ver, drf, p)
    joint, _ = position_marginals(law, 1, 5)
    np.testing.assert_allclose(joint[0], np.minimum(p[0], q[0]) + (1.0 - alpha) * q[0], atol=1e-12)


def test_fuzzy_greedy_rows():
    """Temperature 0: assisted acceptance is greedy verification; the divergence of one-hot rows is
    0 or 1, so any tau in [0, 1) accepts exactly where the two argmaxes agree."""
    rng = np.random.default_rng(70)
    B, K, V = 40, 4, 9
    ver = np.round(rng.normal(0, 1, (B, K + 1, V)) * 2) / 2
    drf = np.where(rng.random((B, K, V)) < 0.5, ver[:, :K], np.round(rng.normal(0, 1, (B, K, V)) * 2) / 2)
    toks = np.argmax(drf, axis=-1)
    u = rng.random((B, K + 1))
    T = np.zeros(B)
    a = oracle.fuzzy_verify(ver, drf, toks, u, T, 0.0, mode="assisted")
    g = oracle.verify(ver, drf, toks, u, T, np.ones(B))
    np.testing.assert_array_equal(a["out_tokens"], g["out_tokens"])
    f = oracle.fuzzy_verify(ver, drf, toks, u, T, 0.5)
    agree = np.argmax(ver[:, :K], axis=-1) == np.argmax(drf, axis=-1)
    np.testing.assert_array_equal(f["div"], np.where(agree, 0.0, 1.0))
    np.testing.assert_array_equal(f["accept_len"], np.sum(np.cumprod(agree, axis=1), axis=1))
    np.testing.assert_array_equal(f["out_tokens"], g["out_tokens"])   # tokens = argmax where they agree


def _fuzzy_as_verify(target, draft, tokens, u, T, top_p, F, C, tau, mode):
    """fuzzy_verify under the calling convention of tests.exact_law."""
    return oracle.fuzzy_verify(target, draft, tokens, u, T, tau, mode=mode)


# --------------------------------------------------------------------------------------
# Tree verification and tree reuse
# --------------------------------------------------------------------------------------
def _bisect_last_true(pred, lo=0.0, hi=None):
    """Largest u in [0, 1) (as a limit, to ~1e-15) with pred(u) true, given pred monotone
    (true then false); 0 if pred(0) is false, 1 if pred is true up to 1."""
    hi = np.nextafter(1.0, 0.0) if hi is None else hi
    if not pred(0.0):
        return 0.0
    if pred(hi):
        return 1.0
    a, b = 0.0, hi
    for _ in range(60):
        m = 0.5 * (a + b)
        if pred(m):
            a = m
        else:
            b = m
    return b


def _first_token_law_of_tree(tgt, drf, m, V):
    """Exact law of the first committed token when the root has m children drafted i.i.d.
    from the root's draft distribution: the tree rule is treated as a black box of its uniforms."""
    from itertools import product
    p = softmax(drf[0])
    law = np.zeros(V)
    one = np.nextafter(1.0, 0.0)
    parents = np.zeros((1, m), dtype=np.int64)
    for toks in product(range(V), repeat=m):
        wgt = float(np.prod([p[t] for t in toks]))
        tt = np.array([toks])

        def run(uvec):
            r = oracle.tree_verify(tgt[None], drf[None], parents, tt, np.array([uvec]), np.ones(1))
            return int(r["path"][0, 0]), int(r["out_tokens"][0, 0])
        reach = 1.0
        for i in range(1, m + 1):
            if reach == 0.0:
                break
            base = [0.5] + [one] * m

            def accepted(x, i=i, base=base):
                v = list(base)
                v[i] = x
                return run(v)[0] == i
            r_i = _bisect_last_true(accepted)
            law[toks[i - 1]] += wgt * reach * r_i
            reach *= (1.0 - r_i)
        if reach > 0.0:
            base = [0.0] + [one] * m
            lo_u, cur = 0.0, run(base)[1]
            while True:
                def same(x, cur=cur):
                    v = list(base)
                    v[0] = x
                    return run(v)[1] == cur
                if same(one):
                    law[cur] += wgt * reach * (1.0 - lo_u)
                    break
                hi_u = _bisect_last_true(lambda x: same(max(x, lo_u)))
                law[cur] += wgt * reach * (hi_u - lo_u)
                lo_u = hi_u
                v = list(base)
                v[0] = hi_u
                cur = run(v)[1]
    return law


@pytest.mark.parametrize("m,V,seed", [(1, 4, 0), (2, 3, 1), (2, 5, 3), (3, 5, 14)])
def test_tree_root_with_m_children_is_lossless(m, V, seed):
    """SpS notes §3's rule applied again after each rejection (the residual of the residual):
    with m children drafted i.i.d. from p, the first committed token follows q exactly.  The
    draft is made far from the target so that several tokens keep a positive residual after
    each rejection (otherwise every residual is the same one-hot vector)."""
    rng = np.random.default_rng(80 + seed)
    tgt = rng.normal(0, 1.5, size=(m + 1, V))
    drf = rng.normal(0, 1.5, size=(m + 1, V))
    q, p = softmax(tgt[0]), softmax(drf[0])
    assert (q > p).sum() >= (3 if V >= 5 else 1)
    law = _first_token_law_of_tree(tgt, drf, m, V)
    np.testing.assert_allclose(law, softmax(tgt[0]), atol=1e-12)


def test_tree_chain_is_plain_verification():
    """A chain (node i below node i-1) is a plain draft of K tokens: the tree rule equals
    speculative sampling (uniform slots mapped: node i <- position i, the draw <- slot K)."""
    rng = np.random.default_rng(90)
    B, K, V = 64, 5, 40
    tgt = rng.normal(0, 2, size=(B, K + 1, V))
    drf = 0.7 * tgt + rng.normal(0, 1, size=(B, K + 1, V))
    toks = oracle.draft_sample(drf[:, :K], rng.random((B, K)), np.ones(B), np.ones(B))["tokens"]
    u = rng.random((B, K + 1))
    T = np.where(np.arange(B) % 4 == 0, 0.0, 1.0)
    ref = oracle.verify(tgt, drf[:, :K], toks, u, T, np.ones(B))
    parents = np.tile(np.arange(K), (B, 1))
    ut = np.concatenate([u[:, K:], u[:, :K]], axis=1)
    got = oracle.tree_verify(tgt, drf, parents, toks, ut, T)
    np.testing.assert_array_equal(got["accept_len"], ref["accept_len"])
    np.testing.assert_array_equal(got["out_tokens"], ref["out_tokens"])


def test_tree_greedy_hand_example():
    """Root children 1 (tok 2), 2 (tok 5); node 2 has children 3 (tok 1), 4 (tok 4).  The target
    argmax is 5 at the root, 4 after node 2 and 0 after node 4: the path is 2 -> 4, then 0."""
    V = 6
    tgt = np.full((1, 5, V), -1.0)
    for row, a in [(0, 5), (2, 4), (4, 0), (1, 3), (3, 3)]:
        tgt[0, row, a] = 2.0
    r = oracle.tree_verify(tgt, np.zeros((1, 5, V)), np.array([[0, 0, 2, 2]]), np.array([[2, 5, 1, 4]]),
                           np.full((1, 5), 0.5), np.zeros(1))
    assert r["accept_len"][0] == 2 and list(r["path"][0]) == [2, 4, -1, -1]
    assert list(r["out_tokens"][0]) == [5, 4, 0, -1, -1]


def test_tree_greedy_takes_the_first_of_equal_siblings():
    """Root children 1 and 2 both hold token 5, the target's argmax at the root; the walk takes
    node 1 (the lower index).  After node 1 the argmax is 1 (its child 3), after node 3 it is 0
    (no child): path 1 -> 3, then 0.  Through node 2 it would have gone to node 4 (token 4)."""
    V = 6
    tgt = np.full((1, 5, V), -1.0)
    for row, a in [(0, 5), (1, 1), (2, 4), (3, 0), (4, 3)]:
        tgt[0, row, a] = 2.0
    par, tok = np.array([[0, 0, 1, 2]]), np.array([[5, 5, 1, 4]])
    r = oracle.tree_verify(tgt, np.zeros((1, 5, V)), par, tok, np.full((1, 5), 0.5), np.zeros(1))
    assert r["accept_len"][0] == 2 and list(r["path"][0]) == [1, 3, -1, -1]
    assert list(r["out_tokens"][0]) == [5, 1, 0, -1, -1]
    # reuse walks the same way: (5, 1) ends at node 3; (5, 4) follows node 1 too, which has no
    # child 4, so node 4 below the equal sibling 2 is not found (the reading that the walk and
    # the reuse check both take)
    assert list(oracle.tree_reuse(np.repeat(par, 2, 0), np.repeat(tok, 2, 0), [1, 1],
                                  np.array([[5, 1, -1, -1, -1], [5, 4, -1, -1, -1]]))) == [3, -1]


def test_tree_reuse_depth2_branching():
    """Mirror-SD notes §3.3: roots A, B; under A -> F the draft expanded two branches (Z and Q).
    The committed prefix A, F, Q reuses the tree (ending at Q's node); A, F, X does not."""
    A, B_, F, Z, Q, X = 10, 11, 12, 13, 14, 15
    parents = np.array([[0, 0, 1, 3, 3]])          # nodes: 1 A, 2 B, 3 F (under A), 4 Z, 5 Q (under F)
    tokens = np.array([[A, B_, F, Z, Q]])
    hit = oracle.tree_reuse(parents, tokens, np.array([2]), np.array([[A, F, Q, -1]]))
    miss = oracle.tree_reuse(parents, tokens, np.array([2]), np.array([[A, F, X, -1]]))
    root = oracle.tree_reuse(parents, tokens, np.array([0]), np.array([[B_, -1, -1, -1]]))
    assert hit[0] == 5 and miss[0] == -1 and root[0] == 2
