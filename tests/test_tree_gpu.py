"""sv_tree_verify and sv_tree_reuse on the GPU (through the C ABI) against the float64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_gb300 as sv
from synth import workloads as W
from tests.helpers import to_f64

pytestmark = pytest.mark.gpu


def random_trees(rng, B, N, spread=4):
    """parents [B, N]: node i hangs below one of the `spread` nodes before it (or the root)."""
    par = np.zeros((B, N), dtype=np.int64)
    for i in range(1, N + 1):
        par[:, i - 1] = rng.integers(max(0, i - spread), i, size=B)
    return par


def tree_inputs(w, N, rng, greedy_every=0, round_idx=0):
    """Target / draft logits with N+1 rows per sequence; each node's token drawn by the oracle's
    sampler from the draft row of its parent."""
    w = W.scaled(w, K=N, draft_rows_extra=1)
    tgt, drf = W.logits(w, round_idx, device="cuda")
    T = W.temperatures(w)
    if greedy_every:
        T[::greedy_every] = 0.0
    par = random_trees(rng, w.B, N)
    d64 = to_f64(drf)
    rows = np.take_along_axis(d64, par[:, :, None], axis=1)          # the parent's draft row per node
    toks = oracle.draft_sample(rows, rng.random((w.B, N)), T, np.ones(w.B))["tokens"]
    u = rng.random((w.B, N + 1))
    return w, tgt, drf, par, toks, u, T


def run(tgt, drf, par, toks, u, T):
    al, ot, path, st = sv.sv_tree_verify(tgt, drf, torch.as_tensor(par, dtype=torch.int32, device="cuda"),
                                         torch.as_tensor(toks, dtype=torch.int32, device="cuda"),
                                         torch.as_tensor(u, device="cuda"), torch.as_tensor(T, device="cuda"))
    torch.cuda.synchronize()
    return al.cpu().numpy(), ot.cpu().numpy(), path.cpu().numpy(), sv.read_stats(st)


def check(out, ref, unresolved_ok=False):
    al, ot, path, st = out
    assert st["status"] == 0, st
    if not unresolved_ok:
        assert st["unresolved"] == 0, st
    np.testing.assert_array_equal(al, ref["accept_len"])
    np.testing.assert_array_equal(ot, ref["out_tokens"])
    np.testing.assert_array_equal(path, ref["path"])


@pytest.mark.parametrize("N,greedy_every", [(16, 0), (16, 3), (40, 4)])
def test_tree_verify_bf16(N, greedy_every):
    rng = np.random.default_rng(100 + N + greedy_every)
    w, tgt, drf, par, toks, u, T = tree_inputs(W.scaled(W.SAMPLED_TOPP, B=12, top_p=1.0, temperature=1.0), N, rng,
                                               greedy_every)
    ref = oracle.tree_verify(to_f64(tgt), to_f64(drf), par, toks, u, T)
    out = run(tgt, drf, par, toks, u, T)
    check(out, ref)
    assert out[0].max() >= 2                                # some multi-level paths


def test_tree_verify_f32_close_draft():
    """A draft close to the target: long accepted paths, several rejections per node elsewhere."""
    rng = np.random.default_rng(7)
    base = W.scaled(W.PLAIN, B=24, V=3000, draft_scale=0.95, draft_sigma=0.5)
    w, tgt, drf, par, toks, u, T = tree_inputs(base, 20, rng, greedy_every=5)
    check(run(tgt, drf, par, toks, u, T), oracle.tree_verify(to_f64(tgt), to_f64(drf), par, toks, u, T))


def test_tree_chain_equals_sv_verify():
    """A chain tree is a plain draft: same outputs as sv_verify with the uniform slots mapped."""
    rng = np.random.default_rng(11)
    B, K = 16, 5
    w = W.scaled(W.LARGE_BATCH, B=B, K=K, draft_rows_extra=1, V=20000)
    tgt, drf = W.logits(w, 0, device="cuda")
    T = W.temperatures(w)
    toks = oracle.draft_sample(to_f64(drf[:, :K]), rng.random((B, K)), T, np.ones(B))["tokens"]
    u = rng.random((B, K + 1))
    toks_d = torch.as_tensor(toks, dtype=torch.int32, device="cuda")
    al, ot, _, st = sv.sv_verify(tgt, drf, toks_d, torch.as_tensor(u, device="cuda"), torch.as_tensor(T, device="cuda"))
    par = np.tile(np.arange(K), (B, 1))
    ut = np.concatenate([u[:, K:], u[:, :K]], axis=1)
    out = run(tgt, drf, par, toks, ut, T)
    np.testing.assert_array_equal(out[0], al.cpu().numpy())
    np.testing.assert_array_equal(out[1], ot.cpu().numpy())


def test_tree_decision_too_close_goes_float_float():
    """u of the root's first child set just above the oracle's own acceptance ratio (relative
    1e-9, far inside the float32 margin): the node is redone in float-float and the outputs still
    match the oracle."""
    rng = np.random.default_rng(21)
    w, tgt, drf, par, toks, u, T = tree_inputs(W.scaled(W.PLAIN, B=8, V=5000), 8, rng)
    t64, d64 = to_f64(tgt), to_f64(drf)
    moved = 0
    for b in range(w.B):
        first = int(np.flatnonzero(par[b] == 0)[0]) + 1
        q, _, _ = oracle.row_distribution(t64[b, 0], T[b], 1.0)
        p, _, _ = oracle.row_distribution(d64[b, 0], T[b], 1.0)
        t = toks[b, first - 1]
        if q[t] < 0.99 * p[t]:                   # a ratio below 1: u stays in [0, 1)
            u[b, first] = q[t] / p[t] * (1.0 + 1e-9)
            moved += 1
    assert moved >= 1
    out = run(tgt, drf, par, toks, u, T)
    check(out, oracle.tree_verify(t64, d64, par, toks, u, T))
    assert out[3]["reresolved"] >= 1, out[3]


def test_tree_reuse_matches_oracle():
    rng = np.random.default_rng(31)
    B, N, V, K = 64, 24, 50, 6
    par = random_trees(rng, B, N)
    toks = rng.integers(0, V, size=(B, N))
    al = rng.integers(0, K + 1, size=B)
    ot = np.full((B, K + 1), -1, dtype=np.int64)
    for b in range(B):                       # half of the prefixes walk down the tree
        node, seq = 0, []
        for j in range(al[b] + 1):
            ch = [i for i in range(1, N + 1) if par[b, i - 1] == node]
            if ch and b % 2 == 0:
                node = ch[rng.integers(len(ch))]
                seq.append(toks[b, node - 1])
            else:
                seq.append(rng.integers(0, V))
        ot[b, : al[b] + 1] = seq
    want = oracle.tree_reuse(par, toks, al, ot)
    got = sv.sv_tree_reuse(*(torch.as_tensor(x, dtype=torch.int32, device="cuda") for x in (par, toks, al, ot)))
    np.testing.assert_array_equal(got.cpu().numpy(), want)
    assert (want > 0).sum() >= 8


def test_tree_greedy_equal_siblings():
    """Root children 1 and 2 both hold token 5, the target's argmax at the root: the walk takes
    node 1, then its child 3 (the argmax after node 1 is 1), then stops with 0; reuse follows the
    same first child, so (5, 4) below node 2 is not found.  Outputs equal the oracle's."""
    V = 1024
    x = np.full((1, 5, V), -1.0)
    for row, am in [(0, 5), (1, 1), (2, 4), (3, 0), (4, 3)]:
        x[0, row, am] = 2.0
    par, tok = np.array([[0, 0, 1, 2]]), np.array([[5, 5, 1, 4]])
    u, T = np.full((1, 5), 0.5), np.zeros(1, np.float32)
    tgt = torch.as_tensor(x, dtype=torch.float32, device="cuda")
    al, ot, path, st = run(tgt, torch.zeros_like(tgt), par, tok, u, T)
    assert st["status"] == 0, st
    ref = oracle.tree_verify(x, np.zeros_like(x), par, tok, u, T)
    assert al[0] == 2 and list(path[0]) == [1, 3, -1, -1] and list(ot[0]) == [5, 1, 0, -1, -1]
    np.testing.assert_array_equal(ot, ref["out_tokens"])
    i32 = dict(dtype=torch.int32, device="cuda")
    got = sv.sv_tree_reuse(torch.as_tensor(np.repeat(par, 2, 0), **i32), torch.as_tensor(np.repeat(tok, 2, 0), **i32),
                           torch.as_tensor([1, 1], **i32), torch.as_tensor([[5, 1, -1, -1, -1], [5, 4, -1, -1, -1]], **i32))
    assert got.cpu().tolist() == [3, -1]


def test_tree_errors():
    rng = np.random.default_rng(41)
    w, tgt, drf, par, toks, u, T = tree_inputs(W.scaled(W.PLAIN, B=6, V=1000), 6, rng)
    bad = par.copy()
    bad[2, 3] = 5                              # node 4 below node 5: not a tree order
    al, ot, _, st = run(tgt, drf, bad, toks, u, T)
    assert st["status"] == sv._abi.SV_ERR_INVALID_ARG and st["error_index"] == 2
    assert (ot[2] == -1).all()
    bt = toks.copy()
    bt[4, 0] = 5000
    _, _, _, st = run(tgt, drf, par, bt, u, T)
    assert st["status"] == sv._abi.SV_ERR_BAD_TOKEN and st["error_index"] == 4


def branch_complete_parents(B, kappa, gamma):
    """parents [B, kappa * gamma] of the branch-complete tree the benchmark verifies: kappa roots
    below the context, each heading a chain of gamma drafted tokens (node = branch * gamma + depth)."""
    par = np.zeros((B, kappa * gamma), dtype=np.int64)
    for i in range(kappa):
        for d in range(1, gamma + 1):
            node = i * gamma + d
            par[:, node - 1] = 0 if d == 1 else node - 1
    return par


def branch_complete_inputs(B, rng, round_idx):
    """The benchmark's tree workload (Mirror recipe, kappa = 8 roots x depth gamma = 7, 56 nodes,
    V = 151936 bf16, T = 1): each node's token drawn by the oracle's sampler from its parent's draft
    row, the uniforms from rng."""
    base = W.MIRROR
    N = base.kappa * base.K
    w = W.scaled(base, B=B, K=N, draft_rows_extra=1)
    tgt, drf = W.logits(w, round_idx, device="cuda")
    T = W.temperatures(w)
    par = branch_complete_parents(B, base.kappa, base.K)
    toks = np.zeros((B, N), dtype=np.int64)
    ud = rng.random((B, N))
    for b0 in range(0, B, 4):
        d64 = to_f64(drf[b0:b0 + 4])
        rows = np.take_along_axis(d64, par[b0:b0 + 4, :, None], axis=1)
        toks[b0:b0 + 4] = oracle.draft_sample(rows, ud[b0:b0 + 4], T[b0:b0 + 4], np.ones(len(rows)))["tokens"]
    u = rng.random((B, N + 1))
    return tgt, drf, par, toks, u, T


def _tree_reference(tgt, drf, par, toks, u, T, chunk=4):
    parts = []
    for b0 in range(0, tgt.shape[0], chunk):
        s = slice(b0, b0 + chunk)
        parts.append(oracle.tree_verify(to_f64(tgt[s]), to_f64(drf[s]), par[s], toks[s], u[s], T[s]))
    return {k: np.concatenate([p[k] for p in parts]) for k in ("accept_len", "out_tokens", "path")}


@pytest.mark.parametrize("B,round_idx", [(4, 0), (64, 1)])
def test_branch_complete_tree(B, round_idx):
    """The benchmark's branch-complete tree (eight roots under the context, depth 7, V = 151936) at
    B = 4 and B = 64, every sequence against the oracle.  At B = 64 the residuals after several
    rejected roots cancel often enough that some sequences need the float-float redo; those must
    match too."""
    rng = np.random.default_rng(500 + B)
    tgt, drf, par, toks, u, T = branch_complete_inputs(B, rng, round_idx)
    out = run(tgt, drf, par, toks, u, T)
    check(out, _tree_reference(tgt, drf, par, toks, u, T))
    if B == 64:
        assert out[3]["reresolved"] > 0, out[3]
