"""Ragged vocabularies on the GPU: V not a multiple of a 16-byte word (a scalar tail in every
row), rows on a padded pitch, for the filter cuts, the divergence pass and the tree walk,
against the float64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_gb300 as sv
from synth import workloads as W
from tests.helpers import to_f64

pytestmark = pytest.mark.gpu

CASES = [("bf16", 3001), ("bf16", 20003), ("f32", 1003), ("f32", 4097)]


def padded(x, V, dtype):
    """x [B, R, V] float64 -> a CUDA tensor view of shape [B, R, V] on rows padded to 64 elements."""
    pad = (V + 63) // 64 * 64
    buf = torch.full((x.shape[0], x.shape[1], pad), float("nan"), dtype=dtype, device="cuda")
    buf[:, :, :V] = torch.as_tensor(x, dtype=dtype, device="cuda")
    return buf[:, :, :V]


def logits(rng, B, R, V, scale=2.0):
    return rng.normal(0, scale, size=(B, R, V))


@pytest.mark.parametrize("dt,V", CASES)
@pytest.mark.parametrize("tk,tp", [(7, 1.0), (0, 0.8), (40, 0.9)])
def test_ragged_filters(dt, V, tk, tp):
    rng = np.random.default_rng(V + tk)
    B, K = 12, 3
    dtype = torch.bfloat16 if dt == "bf16" else torch.float32
    x = logits(rng, B, K + 1, V)
    y = 0.7 * x[:, :K] + rng.normal(0, 1, (B, K, V))
    tg, dr = padded(x, V, dtype), padded(y, V, dtype)
    T = np.where(np.arange(B) % 4 == 0, 0.0, 0.9).astype(np.float32)
    tpa, tka = np.full(B, tp, np.float32), np.full(B, tk, np.int32)
    t64, d64 = to_f64(tg), to_f64(dr)
    toks = oracle.draft_sample(d64, rng.random((B, K)), T, tpa, top_k=tka)["tokens"]
    u = rng.random((B, K + 1))
    ref = oracle.verify(t64, d64, toks, u, T, tpa, top_k=tka)
    al, ot, _, st = sv.sv_verify(tg, dr, torch.as_tensor(toks, dtype=torch.int32, device="cuda"),
                                 torch.as_tensor(u, device="cuda"), torch.as_tensor(T, device="cuda"),
                                 top_p=torch.as_tensor(tpa, device="cuda") if tp < 1 else None,
                                 top_k=torch.as_tensor(tka, device="cuda") if tk else None)
    torch.cuda.synchronize()
    s = sv.read_stats(st)
    assert s["status"] == 0 and s["unresolved"] == 0, s
    np.testing.assert_array_equal(al.cpu().numpy(), ref["accept_len"])
    np.testing.assert_array_equal(ot.cpu().numpy(), ref["out_tokens"])


@pytest.mark.parametrize("dt,V", CASES)
@pytest.mark.parametrize("mode", ["divergence", "assisted"])
def test_ragged_fuzzy(dt, V, mode):
    rng = np.random.default_rng(2 * V + len(mode))
    B, K = 10, 5
    dtype = torch.bfloat16 if dt == "bf16" else torch.float32
    x = logits(rng, B, K + 1, V, 3.0)
    y = 0.8 * x[:, :K] + rng.normal(0, 1.0, (B, K, V)) * rng.uniform(0.1, 1.9, (B, K, 1))
    vr, dr = padded(x, V, dtype), padded(y, V, dtype)
    T = np.where(np.arange(B) % 3 == 0, 0.0, 1.0).astype(np.float32)
    d64 = to_f64(dr)
    toks = oracle.draft_sample(d64, rng.random((B, K)), T, np.ones(B))["tokens"]
    u = rng.random((B, K + 1))
    ref = oracle.fuzzy_verify(to_f64(vr), d64, toks, u, T, 0.3, mode=mode)
    al, ot, div, st = sv.sv_fuzzy_verify(vr, dr, torch.as_tensor(toks, dtype=torch.int32, device="cuda"),
                                         torch.as_tensor(u, device="cuda"), torch.as_tensor(T, device="cuda"),
                                         tau=0.3, mode=mode, divergence=mode == "divergence")
    torch.cuda.synchronize()
    s = sv.read_stats(st)
    assert s["status"] == 0 and s["unresolved"] == 0, s
    np.testing.assert_array_equal(al.cpu().numpy(), ref["accept_len"])
    np.testing.assert_array_equal(ot.cpu().numpy(), ref["out_tokens"])
    if div is not None:
        np.testing.assert_allclose(div.cpu().numpy(), ref["div"], atol=1e-5, rtol=0)


@pytest.mark.parametrize("dt,V", CASES)
def test_ragged_tree(dt, V):
    rng = np.random.default_rng(3 * V)
    B, N = 8, 12
    dtype = torch.bfloat16 if dt == "bf16" else torch.float32
    x = logits(rng, B, N + 1, V)
    y = 0.7 * x + rng.normal(0, 1.2, (B, N + 1, V))
    tg, dr = padded(x, V, dtype), padded(y, V, dtype)
    par = np.zeros((B, N), dtype=np.int64)
    for i in range(1, N + 1):
        par[:, i - 1] = rng.integers(max(0, i - 3), i, size=B)
    T = np.where(np.arange(B) % 4 == 1, 0.0, 1.0).astype(np.float32)
    d64 = to_f64(dr)
    rows = np.take_along_axis(d64, par[:, :, None], axis=1)
    toks = oracle.draft_sample(rows, rng.random((B, N)), T, np.ones(B))["tokens"]
    u = rng.random((B, N + 1))
    ref = oracle.tree_verify(to_f64(tg), d64, par, toks, u, T)
    al, ot, path, st = sv.sv_tree_verify(tg, dr, torch.as_tensor(par, dtype=torch.int32, device="cuda"),
                                         torch.as_tensor(toks, dtype=torch.int32, device="cuda"),
                                         torch.as_tensor(u, device="cuda"), torch.as_tensor(T, device="cuda"))
    torch.cuda.synchronize()
    s = sv.read_stats(st)
    assert s["status"] == 0 and s["unresolved"] == 0, s
    np.testing.assert_array_equal(al.cpu().numpy(), ref["accept_len"])
    np.testing.assert_array_equal(ot.cpu().numpy(), ref["out_tokens"])
    np.testing.assert_array_equal(path.cpu().numpy(), ref["path"])


def test_tree_without_nodes():
    """N = 0: every sequence draws its token from row 0 (or takes its argmax)."""
    rng = np.random.default_rng(5)
    B, V = 6, 2051
    x = logits(rng, B, 1, V)
    tg = padded(x, V, torch.bfloat16)
    T = np.where(np.arange(B) % 2 == 0, 0.0, 1.0).astype(np.float32)
    u = rng.random((B, 1))
    ref = oracle.tree_verify(to_f64(tg), to_f64(tg), np.zeros((B, 0), np.int64), np.zeros((B, 0), np.int64), u, T)
    empty = torch.zeros((B, 0), dtype=torch.int32, device="cuda")
    al, ot, _, st = sv.sv_tree_verify(tg, tg, empty, empty, torch.as_tensor(u, device="cuda"),
                                      torch.as_tensor(T, device="cuda"), path=False)
    torch.cuda.synchronize()
    assert sv.read_stats(st)["status"] == 0
    np.testing.assert_array_equal(ot.cpu().numpy(), ref["out_tokens"])
    assert (al.cpu().numpy() == 0).all()
