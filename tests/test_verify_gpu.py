"""GPU parity of sv_verify against the float64 oracle (called through the C ABI).

Accept lengths and tokens must match exactly (the float32 tier certifies its decisions and
hands the rest to the float-float tier); log-normalisers and probabilities within 1e-6.
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_gb300 as sv
from synth import workloads as W
from tests.helpers import gpu_args, make_inputs, oracle_verify, to_f64

pytestmark = pytest.mark.gpu
TOL = 1e-6


def run_gpu(inp, w, top_p=False, F=None, C=None, top_k=False):
    F = w.saguaro_F if F is None else F
    C = w.saguaro_C if C is None else C
    a = gpu_args(inp)
    tp = torch.as_tensor(inp["top_p"], dtype=torch.float32, device="cuda") if top_p else None
    tk = torch.as_tensor(inp["top_k"], dtype=torch.int32, device="cuda") if top_k else None
    al, ot, dbg, st = sv.sv_verify(inp["target"], inp["draft"], a["draft_tokens"], a["uniforms"], a["temperature"],
                                   top_p=tp, saguaro_F=F, saguaro_C=C, debug=True, top_k=tk)
    torch.cuda.synchronize()
    return al.cpu().numpy(), ot.cpu().numpy(), dbg.cpu().numpy(), sv.read_stats(st)


def compare(w, inp, ref, al, ot, dbg, stats, seqs=None):
    seqs = np.arange(w.B) if seqs is None else np.asarray(seqs)
    assert stats["status"] == 0, stats
    np.testing.assert_array_equal(al[seqs], ref["accept_len"])
    np.testing.assert_array_equal(ot[seqs], ref["out_tokens"])
    K = w.K
    d = dbg[seqs]
    greedy = inp["T"][seqs] == 0
    s = ~greedy
    np.testing.assert_allclose(d[s, :, 0], ref["lse_q"][s], atol=TOL, rtol=0)
    np.testing.assert_allclose(d[s, :K, 1], ref["lse_p"][s], atol=TOL, rtol=0)
    np.testing.assert_allclose(d[s, :K, 2], ref["q_s"][s], atol=TOL, rtol=0)
    np.testing.assert_allclose(d[s, :K, 3], ref["p_s"][s], atol=TOL, rtol=0)
    # ratio: compare where the reference is finite, relative (ratios are unbounded)
    rr, gr = ref["ratio"][s], d[s, :K, 4]
    fin = np.isfinite(rr) & (rr < 1e6)
    np.testing.assert_allclose(gr[fin], rr[fin], rtol=1e-5, atol=TOL)
    np.testing.assert_allclose(d[s, 0, 7], ref["residual_mass"][s], atol=TOL, rtol=0)


def test_fast_exp2_error_bound():
    """A sample of 2^26 inputs: the fast exponential stays below 2^-22 (the exhaustive test pins
    the constant the certification uses); both float-float exponentials, plain and with an
    integer offset folded into the exponent, stay near 2^-44."""
    from speculative_decoding_verification_gb300 import _abi
    # results below ~2^-100 are negligible next to row sums >= 1 (and their low word underflows)
    out = sv.sv_selftest_exp2(-100.0, 1.0, 1 << 26).cpu().numpy()
    assert out[0] < 2.0 ** -22, out
    assert out[1] < 1e-13, out


def _layout_constant(name):
    import os
    import re
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "speculative_decoding_verification_gb300", "csrc", "sv_layout.h")
    m = re.search(name + r"\s*=\s*([0-9.eE+-]+);", open(path).read())
    return float(m.group(1))


def test_fast_exp2_error_bound_exhaustive():
    """Every float32 input in [-125, 1]: the fast exponential's largest relative error stays
    within the constant the float32 tier's certification uses.  The float-float one is below
    1e-13 down to 2^-64; below that its low word meets the float32 underflow range, where its
    absolute error (under 1e-7 of a value below 2^-64) is irrelevant to any sum."""
    e_fast, e_ff, n = sv.sv_selftest_exp2_all(-125.0, 1.0)
    assert n > 2_000_000_000
    assert e_fast <= _layout_constant("kEx2RelErr"), e_fast
    assert e_ff < 1e-7, e_ff
    _, e_ff_hi, n_hi = sv.sv_selftest_exp2_all(-64.0, 1.0)
    assert n_hi > 1_000_000_000
    assert e_ff_hi < 1e-13, e_ff_hi


def test_bounded_wait_reports_timeout():
    st = sv.sv_selftest_timeout(200_000)
    torch.cuda.synchronize()
    assert sv.read_stats(st)["status"] == sv._abi.SV_ERR_TIMEOUT


@pytest.mark.parametrize("round_idx", [0, 1])
def test_plain_config_parity(round_idx):
    """B=1, K=4, V=32000 fp32: 128 rounds batched as 128 independent sequences."""
    w = W.scaled(W.PLAIN, B=128)
    inp = make_inputs(w, round_idx)
    ref = oracle_verify(inp, w)
    al, ot, dbg, st = run_gpu(inp, w)
    compare(w, inp, ref, al, ot, dbg, st)
    assert st["draws"] == 128 - st["reresolved"] + st["reresolved"]


def test_large_batch_recipe_small_B():
    """The B=512 recipe (bf16, V=128256, even rows greedy) at B=24."""
    w = W.scaled(W.LARGE_BATCH, B=24)
    inp = make_inputs(w, 0)
    ref = oracle_verify(inp, w)
    al, ot, dbg, st = run_gpu(inp, w)
    compare(w, inp, ref, al, ot, dbg, st)


def test_large_batch_full_size_sampled_sequences():
    """Full B=512 launch; the oracle checks a sample of sequences (greedy and sampled)."""
    w = W.LARGE_BATCH
    inp = make_inputs(w, 0, chunk=64)
    al, ot, dbg, st = run_gpu(inp, w)
    seqs = np.array([0, 1, 2, 3, 100, 101, 255, 256, 257, 400, 401, 510, 511])
    ref = oracle_verify(inp, w, seqs=seqs)
    compare(w, inp, ref, al, ot, dbg, st, seqs=seqs)
    assert st["rows"] == 512 * 6 + 256 * 5


@pytest.mark.parametrize("V,dtype,pitch", [(1, torch.float32, 4), (8, torch.float32, 8), (31, torch.float32, 32),
                                           (31, torch.bfloat16, 32), (1000, torch.bfloat16, 1000),
                                           (4099, torch.bfloat16, 4104)])
def test_ragged_vocabularies(V, dtype, pitch):
    rng = np.random.default_rng(V)
    B, K = 48, 3
    w = W.Workload("ragged", B=B, K=K, V=V, dtype="f32" if dtype == torch.float32 else "bf16", temperature=1.0,
                   top_p=1.0, rounds=1, seed=0, sigma=2.0, draft_scale=0.7, draft_sigma=1.0)
    tg = torch.zeros((B, K + 1, pitch), dtype=dtype, device="cuda")
    dr = torch.zeros((B, K, pitch), dtype=dtype, device="cuda")
    tg[..., :V] = torch.as_tensor(rng.normal(0, 2, (B, K + 1, V)), dtype=dtype, device="cuda")
    dr[..., :V] = 0.7 * tg[:, :K, :V] + torch.as_tensor(rng.normal(0, 1, (B, K, V)), dtype=dtype, device="cuda")
    T = np.where(np.arange(B) % 3 == 0, 0.0, np.where(np.arange(B) % 3 == 1, 1.0, 0.7)).astype(np.float32)
    u = rng.random((B, K + 1))
    d64 = to_f64(dr[..., :V])
    toks = oracle.draft_sample(d64, rng.random((B, K)), T, np.ones(B))["tokens"]
    inp = dict(target=tg[..., :V], draft=dr[..., :V], tokens=toks, u=u, T=T, top_p=np.ones(B, np.float32))
    ref = oracle.verify(to_f64(tg[..., :V]), d64, toks, u, T, np.ones(B))
    al, ot, dbg, st = run_gpu(inp, w)
    compare(w, inp, ref, al, ot, dbg, st)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_masked_logits(dtype):
    """-inf logits (masked tokens) in target and draft rows, at several temperatures."""
    rng = np.random.default_rng(11)
    B, K, V = 40, 3, 3000
    x = rng.normal(0, 2, (B, K + 1, V))
    y = 0.7 * x[:, :K] + rng.normal(0, 1, (B, K, V))
    x[rng.random(x.shape) < 0.3] = -np.inf
    y[rng.random(y.shape) < 0.3] = -np.inf
    tg = torch.as_tensor(x, dtype=dtype, device="cuda")
    dr = torch.as_tensor(y, dtype=dtype, device="cuda")
    T = np.where(np.arange(B) % 4 == 0, 0.0, np.where(np.arange(B) % 4 == 1, 1.0,
                 np.where(np.arange(B) % 4 == 2, 0.6, 1.7))).astype(np.float32)
    d64 = to_f64(dr)
    toks = oracle.draft_sample(d64, rng.random((B, K)), T, np.ones(B))["tokens"]
    u = rng.random((B, K + 1))
    w = W.Workload("masked", B=B, K=K, V=V, dtype="f32" if dtype == torch.float32 else "bf16", temperature=1.0,
                   top_p=1.0, rounds=1, seed=0, sigma=2.0, draft_scale=0.7, draft_sigma=1.0)
    inp = dict(target=tg, draft=dr, tokens=toks, u=u, T=T, top_p=np.ones(B, np.float32))
    ref = oracle.verify(to_f64(tg), d64, toks, u, T, np.ones(B))
    al, ot, dbg, st = run_gpu(inp, w)
    compare(w, inp, ref, al, ot, dbg, st)


def test_identical_draft_accepts_all_and_k0():
    rng = np.random.default_rng(7)
    B, K, V = 32, 4, 2048
    tg = torch.as_tensor(rng.normal(0, 2, (B, K + 1, V)), dtype=torch.float32, device="cuda")
    u = rng.random((B, K + 1))
    T = np.ones(B, np.float32)
    toks = rng.integers(0, V, (B, K))
    a = dict(draft_tokens=torch.as_tensor(toks, dtype=torch.int32, device="cuda"),
             uniforms=torch.as_tensor(u, device="cuda"), temperature=torch.as_tensor(T, device="cuda"))
    al, ot, _, st = sv.sv_verify(tg, tg[:, :K].clone(), a["draft_tokens"], a["uniforms"], a["temperature"])
    ref = oracle.verify(to_f64(tg), to_f64(tg[:, :K]), toks, u, T, np.ones(B))
    assert (al.cpu().numpy() == K).all()
    np.testing.assert_array_equal(ot.cpu().numpy(), ref["out_tokens"])
    # K = 0: the bonus token alone
    al0, ot0, _, st0 = sv.sv_verify(tg[:, :1].contiguous(), None, None, a["uniforms"][:, :1].contiguous(),
                                    a["temperature"])
    ref0 = oracle.verify(to_f64(tg[:, :1]), np.zeros((B, 0, V)), np.zeros((B, 0), int), u[:, :1], T, np.ones(B))
    np.testing.assert_array_equal(ot0.cpu().numpy(), ref0["out_tokens"])
    assert sv.read_stats(st0)["status"] == 0


def test_device_detected_errors():
    rng = np.random.default_rng(1)
    B, K, V = 6, 2, 256
    tg = torch.as_tensor(rng.normal(0, 1, (B, K + 1, V)), dtype=torch.bfloat16, device="cuda")
    dr = torch.as_tensor(rng.normal(0, 1, (B, K, V)), dtype=torch.bfloat16, device="cuda")
    toks = torch.zeros((B, K), dtype=torch.int32, device="cuda")
    u = torch.full((B, K + 1), 0.5, dtype=torch.float64, device="cuda")
    T = torch.ones(B, device="cuda")
    tg2 = tg.clone()
    tg2[3, 1, 17] = float("nan")
    _, _, _, st = sv.sv_verify(tg2, dr, toks, u, T)
    s = sv.read_stats(st)
    assert s["status"] == sv._abi.SV_ERR_NONFINITE and s["error_index"] == 3 * (K + 1) + 1
    toks2 = toks.clone()
    toks2[2, 0] = V
    _, _, _, st = sv.sv_verify(tg, dr, toks2, u, T)
    assert sv.read_stats(st)["status"] == sv._abi.SV_ERR_BAD_TOKEN
    T2 = T.clone()
    T2[4] = -1.0
    _, _, _, st = sv.sv_verify(tg, dr, toks, u, T2)
    assert sv.read_stats(st)["status"] == sv._abi.SV_ERR_INVALID_ARG
    tg3 = tg.clone()
    tg3[0, 0, :] = float("-inf")
    _, _, _, st = sv.sv_verify(tg3, dr, toks, u, T)
    assert sv.read_stats(st)["status"] == sv._abi.SV_ERR_NONFINITE


@pytest.mark.parametrize("K", [1, 3])
def test_chi_square_committed_tokens_V8_gpu(K):
    """10^6 sequences on V=8 through the library: committed tokens follow q at every position
    and accept lengths follow the product law (chi-square, p > 0.01)."""
    import scipy.stats
    from synth import philox
    rng = np.random.default_rng(100 + K)
    V, n = 8, 1_000_000
    row_t = rng.normal(0, 1.5, size=(K + 1, V))
    row_d = 0.6 * row_t[:K] + rng.normal(0, 1.0, size=(K, V))
    q = np.exp(row_t - row_t.max(1, keepdims=True)); q /= q.sum(1, keepdims=True)
    p = np.exp(row_d - row_d.max(1, keepdims=True)); p /= p.sum(1, keepdims=True)
    tg32 = torch.as_tensor(row_t, dtype=torch.float32)
    dr32 = torch.as_tensor(row_d, dtype=torch.float32)
    # draft tokens: inverse CDF of p (float64 of the float32 rows) at Philox uniforms
    pd = np.exp(to_f64(dr32) - to_f64(dr32).max(1, keepdims=True)); pd /= pd.sum(1, keepdims=True)
    u_d = philox.uniforms(21, philox.STREAM_DRAFT, 0, n, K)
    toks = np.stack([np.searchsorted(np.cumsum(pd[j]), u_d[:, j] * pd[j].sum(), side="right") for j in range(K)], 1)
    toks = np.minimum(toks, V - 1)
    u = np.concatenate([philox.uniforms(21, philox.STREAM_ACCEPT, 0, n, K),
                        philox.uniforms(21, philox.STREAM_RESIDUAL, 0, n, 1)], axis=1)
    tg = tg32.to("cuda").expand(n, K + 1, V).contiguous()
    dr = dr32.to("cuda").expand(n, K, V).contiguous()
    al, ot, _, st = sv.sv_verify(tg, dr, torch.as_tensor(toks, dtype=torch.int32, device="cuda"),
                                 torch.as_tensor(u, device="cuda"), torch.ones(n, device="cuda"))
    al = al.cpu().numpy()
    ot = ot.cpu().numpy()
    assert sv.read_stats(st)["status"] == 0
    qf = np.exp(to_f64(tg32) - to_f64(tg32).max(1, keepdims=True)); qf /= qf.sum(1, keepdims=True)
    for i in range(K + 1):
        present = al >= i
        cnt = np.bincount(ot[present, i], minlength=V)
        assert scipy.stats.chisquare(cnt, cnt.sum() * qf[i]).pvalue > 0.01
    a = np.minimum(pd, qf[:K]).sum(axis=1)
    want = np.array([np.prod(a[:j]) * (1 - a[j]) for j in range(K)] + [np.prod(a)])
    assert scipy.stats.chisquare(np.bincount(al, minlength=K + 1), n * want).pvalue > 0.01


@pytest.mark.parametrize("K", [13, 25, 31, 32])
@pytest.mark.parametrize("lazy", [False, True])
@pytest.mark.parametrize("close", [False, True])
def test_long_drafts(K, lazy, close):
    """K up to the library's maximum (32), greedy and sampled sequences mixed (the large-batch
    recipe at B=16, V=128256 bf16).  With close=True the draft is nearly the target, so runs of
    accepted tokens reach deep positions (often the whole draft); with close=False most
    sequences stop early.  sv_verify and sv_verify_lazy (which reads positions 0 and 1 one at a
    time and the rest in one batch) both against the oracle."""
    extra = dict(draft_scale=0.98, draft_sigma=0.12) if close else {}
    w = W.scaled(W.LARGE_BATCH, B=16, K=K, **extra)
    inp = make_inputs(w, 3 + K, chunk=4)
    ref = oracle_verify(inp, w, chunk=2)
    a = gpu_args(inp)
    al, ot, dbg, st = sv.sv_verify(inp["target"], inp["draft"], a["draft_tokens"], a["uniforms"], a["temperature"],
                                   debug=not lazy, lazy=lazy)
    torch.cuda.synchronize()
    al, ot, st = al.cpu().numpy(), ot.cpu().numpy(), sv.read_stats(st)
    if lazy:
        assert st["status"] == 0, st
        np.testing.assert_array_equal(al, ref["accept_len"])
        np.testing.assert_array_equal(ot, ref["out_tokens"])
    else:
        compare(w, inp, ref, al, ot, dbg.cpu().numpy(), st)
    if close:
        assert al.max() >= min(K, 12)                  # deep positions are reached


@pytest.mark.parametrize("lazy", [False, True])
def test_accept_test_too_close_goes_float_float(lazy):
    """u of position 1 set within 1e-9 (relative) of the oracle's own acceptance ratio, above it
    for some sequences and below for others: far inside the float32 tier's certified margin, so
    those sequences' accept tests are redone in the float-float tier (exact row sums, then the
    draw), and every output still equals the oracle's.  Greedy sequences are left as they are."""
    w = W.scaled(W.LARGE_BATCH, B=24, V=20000)
    inp = make_inputs(w, 5)
    ref0 = oracle_verify(inp, w)
    moved = 0
    for b in range(w.B):
        r = ref0["ratio"][b, 0]
        if inp["T"][b] > 0 and 1e-3 < r < 0.99:
            inp["u"][b, 0] = r * (1.0 + (1e-9 if b % 4 == 1 else -1e-9))
            moved += 1
    assert moved >= 3
    ref = oracle_verify(inp, w)
    a = gpu_args(inp)
    al, ot, dbg, st = sv.sv_verify(inp["target"], inp["draft"], a["draft_tokens"], a["uniforms"], a["temperature"],
                                   debug=not lazy, lazy=lazy)
    torch.cuda.synchronize()
    al, ot, st = al.cpu().numpy(), ot.cpu().numpy(), sv.read_stats(st)
    assert st["reresolved"] >= moved, st
    if lazy:
        assert st["status"] == 0 and st["unresolved"] == 0, st
        np.testing.assert_array_equal(al, ref["accept_len"])
        np.testing.assert_array_equal(ot, ref["out_tokens"])
    else:
        compare(w, inp, ref, al, ot, dbg.cpu().numpy(), st)
        assert st["unresolved"] == 0, st


def _inject_special_logits(x, rng):
    """Logits the float-float tier's bf16 weight tables do not cover (zero, |x| < 2^-9, |x| >=
    128, -inf) and large negative ones inside them, at a few random ids of every row."""
    B, R, V = x.shape
    for val in (0.0, 1e-4, -3e-4, -60.0, -100.0, -150.0, -300.0, float("-inf")):
        ids = torch.as_tensor(rng.integers(0, V, size=(B, R, 3)), device=x.device)
        x.scatter_(2, ids, torch.full(ids.shape, val, dtype=x.dtype, device=x.device))


@pytest.mark.parametrize("lazy", [False, True])
def test_draw_near_boundary_goes_float_float(lazy):
    """u of the residual draw set 1e-8 (relative) above or below a boundary of the oracle's
    own cumulative residual sum, so that the float32 tier cannot certify the draw and the
    float-float tier decides it, at temperatures from 0.15 to 3 (bf16 rows without filters:
    the tier's factored weight tables, with the direct exponential for the logits and
    temperatures they leave out).  Every output equals the oracle's."""
    w = W.scaled(W.LARGE_BATCH, B=30, K=3, V=20000, greedy_even_rows=False)
    inp = make_inputs(w, 2)
    rng = np.random.default_rng(7)
    _inject_special_logits(inp["target"], rng)
    _inject_special_logits(inp["draft"], rng)
    temps = np.array([0.0, 0.15, 0.3, 0.6, 1.0, 1.7, 3.0], np.float32)
    inp["T"] = temps[np.arange(w.B) % len(temps)]
    ref0 = oracle_verify(inp, w)
    K = w.K
    moved = 0
    drawn = {}
    for b in range(w.B):
        if inp["T"][b] == 0:
            continue
        k = int(ref0["accept_len"][b])
        T = float(inp["T"][b])
        q, _, _ = oracle.row_distribution(to_f64(inp["target"][b, k]), T, 1.0)
        if k < K:
            p, _, _ = oracle.row_distribution(to_f64(inp["draft"][b, k]), T, 1.0)
            wr = np.maximum(q - p, 0.0)
        else:
            wr = q
        c = np.cumsum(wr)
        R = c[-1]
        # a boundary C(t) between 5% and 95% of R, the one nearest the middle id whose draw
        # (t just below it, the next id whose sum passes u R just above it) lies at least
        # 5e-10 R from every boundary: the float-float tier resolves 2e-11
        cand = np.nonzero((c > 0.05 * R) & (c < 0.95 * R) & (wr > 0))[0]
        if R <= 0 or len(cand) == 0:
            continue
        found = None
        for t in cand[np.argsort(np.abs(cand - cand[len(cand) // 2]), kind="stable")][:400]:
            u_b = c[t] / R * (1.0 + (1e-8 if b % 2 else -1e-8))
            thr = u_b * R
            v = int(np.searchsorted(c, thr, side="right"))
            if v < len(c) and min(c[v] - thr, thr - (c[v - 1] if v > 0 else 0.0)) >= 5e-10 * R:
                found = (u_b, v)
                break
        if found is None:
            continue
        inp["u"][b, K], drawn[b] = found
        moved += 1
    assert moved >= 12, moved
    ref = oracle_verify(inp, w)
    for b, t in drawn.items():
        assert ref["out_tokens"][b, ref["accept_len"][b]] == t, (b, t)
    a = gpu_args(inp)
    al, ot, dbg, st = sv.sv_verify(inp["target"], inp["draft"], a["draft_tokens"], a["uniforms"], a["temperature"],
                                   debug=not lazy, lazy=lazy)
    torch.cuda.synchronize()
    al, ot, st = al.cpu().numpy(), ot.cpu().numpy(), sv.read_stats(st)
    assert st["reresolved"] >= moved, st
    assert st["status"] == 0 and st["unresolved"] == 0, st
    np.testing.assert_array_equal(al, ref["accept_len"])
    np.testing.assert_array_equal(ot, ref["out_tokens"])
