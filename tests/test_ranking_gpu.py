"""GPU parity of the ranking-based paths against the float64 oracle (through the C ABI):
nucleus (top-p) and top-k verification, the Saguaro transform in verification and in draft sampling,
cache keys and lookup, top-kappa roots and Mirror-style branch reuse."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_gb300 as sv
from synth import workloads as W
from tests.helpers import gpu_args, make_inputs, oracle_verify, to_f64
from tests.test_verify_gpu import compare, run_gpu

pytestmark = pytest.mark.gpu


# --------------------------------------------------------------------------------------
# top-p verification (the T=0.8, top-p 0.9 recipe)
# --------------------------------------------------------------------------------------
@pytest.mark.parametrize("round_idx", [0, 1])
def test_top_p_verify_parity(round_idx):
    w = W.scaled(W.SAMPLED_TOPP, B=8)
    inp = make_inputs(w, round_idx)
    ref = oracle_verify(inp, w)
    al, ot, dbg, st = run_gpu(inp, w, top_p=True)
    compare(w, inp, ref, al, ot, dbg, st)
    np.testing.assert_allclose(dbg[:, :, 5], ref["mass_q"], atol=1e-6)
    np.testing.assert_allclose(dbg[:, : w.K, 6], ref["mass_p"], atol=1e-6)


@pytest.mark.parametrize("tp", [1.0, 0.999, 0.5, 1e-6])
def test_top_p_values_small_vocab(tp):
    """top_p = 1 (off), close to 1, middling, and so small the nucleus is the top token."""
    w = W.scaled(W.SAMPLED_TOPP, B=32, V=4000, top_p=tp)
    inp = make_inputs(w, 3)
    ref = oracle_verify(inp, w)
    al, ot, dbg, st = run_gpu(inp, w, top_p=True)
    compare(w, inp, ref, al, ot, dbg, st)
    np.testing.assert_allclose(dbg[:, :, 5], ref["mass_q"], atol=1e-6)
    np.testing.assert_allclose(dbg[:, : w.K, 6], ref["mass_p"], atol=1e-6)
    assert st["unresolved"] == 0, st


def test_top_p_with_plateaus():
    """Equal logits straddling the cut: the nucleus keeps the lowest ids of the tie group."""
    rng = np.random.default_rng(5)
    B, K, V = 16, 3, 512
    base = np.round(rng.normal(0, 1, (B, K + 1, V)) * 2) / 2       # many ties (step 0.5)
    tg = torch.as_tensor(base, dtype=torch.bfloat16, device="cuda")
    dr = torch.as_tensor(np.round(0.7 * base[:, :K] * 2) / 2 + 0.25, dtype=torch.bfloat16, device="cuda")
    T = np.ones(B, np.float32)
    tp = np.full(B, 0.7, np.float32)
    d64 = to_f64(dr)
    toks = oracle.draft_sample(d64, rng.random((B, K)), T, tp)["tokens"]
    u = rng.random((B, K + 1))
    w = W.Workload("plateau", B=B, K=K, V=V, dtype="bf16", temperature=1.0, top_p=0.7, rounds=1, seed=0, sigma=1,
                   draft_scale=0.7, draft_sigma=1)
    inp = dict(target=tg, draft=dr, tokens=toks, u=u, T=T, top_p=tp)
    ref = oracle.verify(to_f64(tg), d64, toks, u, T, tp)
    al, ot, dbg, st = run_gpu(inp, w, top_p=True)
    compare(w, inp, ref, al, ot, dbg, st)


# --------------------------------------------------------------------------------------
# top-k verification, alone and ahead of top-p
# --------------------------------------------------------------------------------------
@pytest.mark.parametrize("round_idx,top_p", [(0, 1.0), (1, 1.0), (0, 0.9), (1, 0.9)])
def test_top_k_verify_parity(round_idx, top_p):
    w = W.scaled(W.SAMPLED_TOPK, top_p=top_p)
    inp = make_inputs(w, round_idx)
    ref = oracle_verify(inp, w)
    al, ot, dbg, st = run_gpu(inp, w, top_p=top_p < 1, top_k=True)
    compare(w, inp, ref, al, ot, dbg, st)
    np.testing.assert_allclose(dbg[:, :, 5], ref["mass_q"], atol=1e-6)
    np.testing.assert_allclose(dbg[:, : w.K, 6], ref["mass_p"], atol=1e-6)
    assert st["unresolved"] == 0, st


@pytest.mark.parametrize("k,tp", [(1, 1.0), (2, 1.0), (50, 1.0), (3999, 1.0), (4000, 1.0), (0, 1.0), (-3, 1.0),
                                  (1, 0.5), (7, 0.999), (300, 0.5), (300, 1e-6), (3999, 0.9)])
def test_top_k_values_small_vocab(k, tp):
    """k = 1 (the argmax), small, V - 1, V and <= 0 (off); with top-p close to 1, middling and
    tiny, where the nucleus of the top-k set may be the whole set or its first token."""
    w = W.scaled(W.SAMPLED_TOPK, B=32, V=4000, top_p=tp, top_k=k)
    inp = make_inputs(w, 3)
    ref = oracle_verify(inp, w)
    al, ot, dbg, st = run_gpu(inp, w, top_p=tp < 1, top_k=True)
    compare(w, inp, ref, al, ot, dbg, st)
    np.testing.assert_allclose(dbg[:, :, 5], ref["mass_q"], atol=1e-6)
    np.testing.assert_allclose(dbg[:, : w.K, 6], ref["mass_p"], atol=1e-6)
    assert st["unresolved"] == 0, st


@pytest.mark.parametrize("k,tp", [(5, 1.0), (37, 1.0), (37, 0.6), (200, 1.0), (200, 0.95)])
def test_top_k_with_plateaus_and_signed_zeros(k, tp):
    """Equal logits straddling the k-th place keep the lowest ids; -0 and +0 are one value."""
    rng = np.random.default_rng(6)
    B, K, V = 16, 3, 512
    base = np.round(rng.normal(0, 1, (B, K + 1, V)) * 2) / 2       # many ties (step 0.5)
    base[rng.random(base.shape) < 0.15] = 0.0
    neg0 = rng.random(base.shape) < 0.5
    base = np.where((base == 0.0) & neg0, -0.0, base)
    dr_np = np.round(0.7 * base[:, :K] * 2) / 2
    dr_np = np.where(dr_np == 0.0, np.where(neg0[:, :K], -0.0, 0.0), dr_np)
    tg = torch.as_tensor(base, dtype=torch.bfloat16, device="cuda")
    dr = torch.as_tensor(dr_np, dtype=torch.bfloat16, device="cuda")
    assert (torch.signbit(tg) & (tg == 0)).any() and ((~torch.signbit(tg)) & (tg == 0)).any()
    T = np.ones(B, np.float32)
    T[1] = 0.0
    tpa = np.full(B, tp, np.float32)
    tka = np.full(B, k, np.int32)
    d64 = to_f64(dr)
    toks = oracle.draft_sample(d64, rng.random((B, K)), T, tpa, top_k=tka)["tokens"]
    u = rng.random((B, K + 1))
    w = W.Workload("plateau", B=B, K=K, V=V, dtype="bf16", temperature=1.0, top_p=tp, rounds=1, seed=0, sigma=1,
                   draft_scale=0.7, draft_sigma=1, top_k=k)
    inp = dict(target=tg, draft=dr, tokens=toks, u=u, T=T, top_p=tpa, top_k=tka)
    ref = oracle.verify(to_f64(tg), d64, toks, u, T, tpa, top_k=tka)
    al, ot, dbg, st = run_gpu(inp, w, top_p=tp < 1, top_k=True)
    compare(w, inp, ref, al, ot, dbg, st)
    np.testing.assert_allclose(dbg[:, :, 5], ref["mass_q"], atol=1e-6)


def test_top_k_on_the_lazy_and_static_entry_points():
    """sv_verify_lazy runs the full pipeline under a filter, sv_verify_static passes top_k on:
    both equal sv_verify."""
    w = W.scaled(W.SAMPLED_TOPK, B=6, V=20000)
    inp = make_inputs(w, 0)
    a = gpu_args(inp)
    tp = torch.as_tensor(inp["top_p"], device="cuda")
    tk = torch.as_tensor(inp["top_k"], device="cuda")
    outs = []
    for mode in ("eager", "lazy", "static"):
        if mode == "static":
            al, ot, _, st = sv.sv_verify_static(inp["target"], inp["draft"], a["draft_tokens"], a["uniforms"],
                                                a["temperature"], top_p=tp, top_k=tk)
        else:
            al, ot, _, st = sv.sv_verify(inp["target"], inp["draft"], a["draft_tokens"], a["uniforms"],
                                         a["temperature"], top_p=tp, top_k=tk, lazy=mode == "lazy")
        torch.cuda.synchronize()
        assert sv.read_stats(st)["status"] == 0
        outs.append((al.cpu().numpy(), ot.cpu().numpy()))
    ref = oracle_verify(inp, w)
    for al, ot in outs:
        np.testing.assert_array_equal(al, ref["accept_len"])
        np.testing.assert_array_equal(ot, ref["out_tokens"])


# --------------------------------------------------------------------------------------
# Saguaro: verification with p' and the draft sampler
# --------------------------------------------------------------------------------------
@pytest.mark.parametrize("F,C", [(8, 0.3), (8, 0.0), (1, 0.5), (100, 0.5), (300, 0.1)])
def test_saguaro_verify_parity(F, C):
    w = W.scaled(W.SAGUARO, B=16, saguaro_F=F, saguaro_C=C)
    inp = make_inputs(w, 0)
    ref = oracle_verify(inp, w)
    al, ot, dbg, st = run_gpu(inp, w)
    compare(w, inp, ref, al, ot, dbg, st)


@pytest.mark.parametrize("F,C,top_p,top_k", [(0, 1.0, None, None), (8, 0.3, None, None), (8, 0.0, None, None),
                                             (8, 0.3, 0.9, None), (0, 1.0, None, 20), (8, 0.3, 0.9, 20),
                                             (8, 0.0, None, 5), (48, 0.3, None, None), (128, 0.2, 0.9, None),
                                             (129, 0.2, None, None)])
def test_saguaro_sample_parity(F, C, top_p, top_k):
    w = W.scaled(W.SAGUARO, B=16)
    tgt, drf = W.logits(w, 1, device="cuda")
    u_draft, _, _ = W.round_uniforms(w, 1)
    T = W.temperatures(w)
    T[3] = 0.0                    # one greedy row
    T[5] = 0.7
    tp = np.full(w.B, top_p if top_p else 1.0, np.float32)
    tk = np.full(w.B, top_k if top_k else 0, np.int32)
    toks, dbg, st = sv.sv_saguaro_sample(drf, torch.as_tensor(u_draft, device="cuda"), torch.as_tensor(T, device="cuda"),
                                         top_p=torch.as_tensor(tp, device="cuda") if top_p else None, F=F, C=C,
                                         debug=True, top_k=torch.as_tensor(tk, device="cuda") if top_k else None)
    torch.cuda.synchronize()
    s = sv.read_stats(st)
    assert s["status"] == 0, s
    ref = oracle.draft_sample(to_f64(drf), u_draft, T, tp, F, C, top_k=tk)
    np.testing.assert_array_equal(toks.cpu().numpy(), ref["tokens"])
    d = dbg.cpu().numpy()
    sampled = T > 0
    np.testing.assert_allclose(d[sampled, :, 0], ref["lse"][sampled], atol=1e-6)
    if F > 0 and C < 1:
        np.testing.assert_allclose(d[sampled, :, 1], ref["p_top"][sampled], atol=1e-6)
        np.testing.assert_allclose(d[sampled, :, 2], ref["z_prime"][sampled], atol=1e-6)


# --------------------------------------------------------------------------------------
# cache keys, lookup, top-kappa roots, reuse
# --------------------------------------------------------------------------------------
def test_cache_keys_and_lookup_parity():
    w = W.scaled(W.SAGUARO, B=16)
    inp = make_inputs(w, 2)
    f_real, f_int = sv.sv_fanout(w.budget, w.accept_rate, w.power_r, w.K)
    assert list(f_int) == [15, 12, 10, 9, 7, 11]
    toks = torch.as_tensor(inp["tokens"], dtype=torch.int32, device="cuda")
    keys, st = sv.sv_cache_keys(inp["draft"], toks, f_int)
    torch.cuda.synchronize()
    assert sv.read_stats(st)["status"] == 0
    ref_keys = oracle.cache_keys(to_f64(inp["draft"]), inp["tokens"], f_int)
    np.testing.assert_array_equal(keys.cpu().numpy(), ref_keys)
    # lookup on the verification outcome
    ref = oracle_verify(inp, w)
    al, ot, _, _ = run_gpu(inp, w)
    hit = sv.sv_cache_lookup(torch.as_tensor(al, device="cuda"), torch.as_tensor(ot, device="cuda"), keys, f_int)
    ref_hit = oracle.cache_lookup(ref["accept_len"], ref["out_tokens"], ref_keys, f_int)
    np.testing.assert_array_equal(hit.cpu().numpy(), ref_hit)


@pytest.mark.parametrize("V,dtype", [(151936, torch.bfloat16), (5000, torch.float32), (40, torch.bfloat16)])
def test_topk_rows_parity(V, dtype):
    rng = np.random.default_rng(V)
    N = 12
    x = rng.normal(0, 3, (N, V))
    x[3, :] = 1.0                          # a plateau: every token ties
    x[4, ::2] = x[4, 0]                    # half the row ties at one value
    t = torch.as_tensor(x, dtype=dtype, device="cuda")
    T = np.where(np.arange(N) % 2 == 0, 1.0, 0.8).astype(np.float32)
    kappa = min(8, V)
    ids, lp, st = sv.sv_topk_rows(t, kappa, torch.as_tensor(T, device="cuda"))
    torch.cuda.synchronize()
    assert sv.read_stats(st)["status"] == 0
    rid, rlp = oracle.topk_rows(to_f64(t), T, kappa)
    np.testing.assert_array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(lp.cpu().numpy(), rlp, atol=1e-6)


@pytest.mark.parametrize("N,V", [(1, 7), (33, 4099), (700, 32000), (1024, 128256)])
def test_topn_against_sorting(N, V):
    """Radix select vs a full (value desc, id asc) sort, with bf16 plateaus and ties."""
    rng = np.random.default_rng(N + V)
    x = np.round(rng.normal(0, 2, (6, V)) * 4) / 4
    x[2] = 0.0
    x[3] = -np.abs(x[3]) - 0.25                   # all negative: keys with low bits set
    pitch = (V + 7) // 8 * 8                      # 16-byte aligned rows
    buf = torch.zeros((6, pitch), dtype=torch.bfloat16, device="cuda")
    buf[:, :V] = torch.as_tensor(x, dtype=torch.bfloat16, device="cuda")
    t = buf[:, :V]
    ids, _, _ = sv.sv_topk_rows(t, N)
    torch.cuda.synchronize()
    xs = to_f64(t)
    want = np.argsort(-xs, axis=1, kind="stable")[:, :N]
    np.testing.assert_array_equal(ids.cpu().numpy(), want)


def overflow_rows(rng, n, V, S=8):
    """Rows whose largest values fill seven threads of every warp of the first block of a row's
    cluster (16-byte vectors dealt round-robin to S * 256 threads).  Every warp's 8th-largest
    thread maximum stays low, so thousands of elements clear the candidate bound, the first
    block's buffer overflows and the selection takes the single-block radix path.  The high
    values are bf16 steps of 1/32 above 5: many equal values, ordered by id."""
    x = rng.normal(0, 1, (n, V))
    t = (np.arange(V) // 8) % (S * 256)
    hot = (t < 256) & ((t % 32) < 7)
    x[:, hot] = 5.0 + rng.random((n, int(hot.sum())))
    return x


def test_topn_candidate_overflow():
    rng = np.random.default_rng(17)
    V = 151936
    x = overflow_rows(rng, 2, V)
    t = torch.as_tensor(x, dtype=torch.bfloat16, device="cuda")
    for kappa in (8, 16):
        ids, _, st = sv.sv_topk_rows(t, kappa)
        torch.cuda.synchronize()
        assert sv.read_stats(st)["status"] == 0
        want = np.argsort(-to_f64(t), axis=1, kind="stable")[:, :kappa]
        np.testing.assert_array_equal(ids.cpu().numpy(), want)


@pytest.mark.parametrize("C", [0.3, 0.0])
def test_saguaro_sample_candidate_overflow(C):
    """The Saguaro top-F set on rows that overflow the cluster's candidate buffer."""
    rng = np.random.default_rng(18)
    B, R, V = 2, 3, 151936
    drf = torch.as_tensor(overflow_rows(rng, B * R, V).reshape(B, R, V), dtype=torch.bfloat16, device="cuda")
    u = rng.random((B, R))
    T = np.ones(B, np.float32)
    toks, dbg, st = sv.sv_saguaro_sample(drf, torch.as_tensor(u, device="cuda"), torch.as_tensor(T, device="cuda"),
                                         F=8, C=C, debug=True)
    torch.cuda.synchronize()
    assert sv.read_stats(st)["status"] == 0
    ref = oracle.draft_sample(to_f64(drf), u, T, np.ones(B), 8, C)
    np.testing.assert_array_equal(toks.cpu().numpy(), ref["tokens"])
    d = dbg.cpu().numpy()
    np.testing.assert_allclose(d[:, :, 1], ref["p_top"], atol=1e-6)
    np.testing.assert_allclose(d[:, :, 2], ref["z_prime"], atol=1e-6)


def test_mirror_round_parity():
    """Roots from the early-exit row, branches, verification along branch 0, reuse."""
    w = W.scaled(W.MIRROR, B=4)
    tgt, ee = W.logits(w, 0, device="cuda")
    _, u, u_branch = W.round_uniforms(w, 0)
    T = W.temperatures(w)
    kappa, gamma = w.kappa, w.K
    ids, lp, st = sv.sv_topk_rows(ee[:, 0].contiguous(), kappa, torch.as_tensor(T, device="cuda"))
    ee64 = to_f64(ee)
    rid, rlp = oracle.topk_rows(ee64[:, 0], T, kappa)
    np.testing.assert_array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(lp.cpu().numpy(), rlp, atol=1e-6)
    # branch i: root i, then depths 2..gamma sampled from the early-exit rows (oracle sampler)
    branches = np.zeros((w.B, kappa, gamma), dtype=np.int64)
    branches[:, :, 0] = rid
    for i in range(kappa):
        ub = u_branch[:, i * gamma:(i + 1) * gamma]
        branches[:, i, 1:] = oracle.draft_sample(ee64[:, 1:], ub[:, 1:], T, np.ones(w.B))["tokens"]
    toks = branches[:, 0, :]
    ref = oracle.verify(to_f64(tgt), ee64, toks, u, T, np.ones(w.B))
    al, ot, _, st = sv.sv_verify(tgt, ee, torch.as_tensor(toks, dtype=torch.int32, device="cuda"),
                                 torch.as_tensor(u, device="cuda"), torch.as_tensor(T, device="cuda"))
    torch.cuda.synchronize()
    assert sv.read_stats(st)["status"] == 0
    np.testing.assert_array_equal(al.cpu().numpy(), ref["accept_len"])
    np.testing.assert_array_equal(ot.cpu().numpy(), ref["out_tokens"])
    br = torch.as_tensor(branches, dtype=torch.int32, device="cuda")
    reuse = sv.sv_mirror_reuse(br, al, ot)
    np.testing.assert_array_equal(reuse.cpu().numpy(), oracle.mirror_reuse(branches, ref["accept_len"],
                                                                             ref["out_tokens"]))


def test_reuse_and_lookup_hand_cases():
    br = torch.as_tensor([[[5, 6, 7], [5, 8, 9], [3, 1, 1]]] * 4, dtype=torch.int32, device="cuda")
    al = torch.as_tensor([1, 1, 0, 3], dtype=torch.int32, device="cuda")
    ot = torch.as_tensor([[5, 8, -1, -1], [5, 2, -1, -1], [3, -1, -1, -1], [5, 6, 7, 1]], dtype=torch.int32,
                         device="cuda")
    assert sv.sv_mirror_reuse(br, al, ot).cpu().tolist() == [1, 0, 1, 0]
    keys = torch.as_tensor([[2, 4, 0, 2, 3]] * 3, dtype=torch.int32, device="cuda")
    hit = sv.sv_cache_lookup(torch.as_tensor([0, 1, 0], dtype=torch.int32, device="cuda"),
                             torch.as_tensor([[4, -1], [1, 3], [1, -1]], dtype=torch.int32, device="cuda"), keys, [2, 3])
    assert hit.cpu().tolist() == [1, 1, 0]
    # k = gamma - 1: the whole of branch 1 is the committed prefix
    one = torch.as_tensor([2], dtype=torch.int32, device="cuda")
    assert sv.sv_mirror_reuse(br[:1], one, torch.as_tensor([[5, 8, 9, -1]], dtype=torch.int32,
                                                         device="cuda")).cpu().tolist() == [1]
    # t* = 0 is the first depth-1 key, not a depth-0 key: no hit at k = 0
    hit0 = sv.sv_cache_lookup(torch.as_tensor([0], dtype=torch.int32, device="cuda"),
                              torch.as_tensor([[0, -1]], dtype=torch.int32, device="cuda"), keys[:1], [2, 3])
    assert hit0.cpu().tolist() == [0]
