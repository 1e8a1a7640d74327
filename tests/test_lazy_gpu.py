"""sv_verify_lazy on the GPU: the outputs of sv_verify and of the oracle, reading only the rows up
to each sequence's first rejection."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_gb300 as sv
from synth import workloads as W
from tests.helpers import gpu_args, make_inputs, oracle_verify, to_f64

pytestmark = pytest.mark.gpu
TOL = 1e-6


def run(inp, w, lazy, top_p=False):
    a = gpu_args(inp)
    tp = torch.as_tensor(inp["top_p"], dtype=torch.float32, device="cuda") if top_p else None
    al, ot, dbg, st = sv.sv_verify(inp["target"], inp["draft"], a["draft_tokens"], a["uniforms"], a["temperature"],
                                   top_p=tp, saguaro_F=w.saguaro_F, saguaro_C=w.saguaro_C, debug=True, lazy=lazy)
    torch.cuda.synchronize()
    return al.cpu().numpy(), ot.cpu().numpy(), dbg.cpu().numpy(), sv.read_stats(st)


TAIL = 2   # from this position on, the lazy path reads all remaining positions at once


def expected_rows(al, T, K):
    """Rows the lazy path reads: positions 0..min(k, TAIL-1) one at a time (the target row, and
    the draft row of a sampled sequence below K); once a sequence reaches position TAIL, every
    remaining row of it."""
    n = 0
    for k, t in zip(al, T):
        sampled = t != 0
        for j in range(0, min(k, TAIL - 1) + 1):
            n += 1 + (sampled and j < K)
        if k >= TAIL:
            n += (K - TAIL + 1) + (K - TAIL if sampled else 0)
    return n


def check(w, inp, ref, out, seqs=None):
    al, ot, dbg, st = out
    seqs = np.arange(w.B) if seqs is None else np.asarray(seqs)
    assert st["status"] == 0, st
    np.testing.assert_array_equal(al[seqs], ref["accept_len"])
    np.testing.assert_array_equal(ot[seqs], ref["out_tokens"])
    K = w.K
    T = inp["T"][seqs]
    d = dbg[seqs]
    for i, b in enumerate(seqs):
        if T[i] == 0:
            assert np.isnan(d[i, :, 0]).all()
            continue
        k = al[b]
        # read positions: 0..k; beyond them the debug fields stay NaN
        np.testing.assert_allclose(d[i, :k + 1, 0], ref["lse_q"][i, :k + 1], atol=TOL, rtol=0)
        assert np.isnan(d[i, k + 1:, 0]).all()
        m = min(k, K - 1) + 1 if K > 0 else 0
        np.testing.assert_allclose(d[i, :m, 1], ref["lse_p"][i, :m], atol=TOL, rtol=0)
        np.testing.assert_allclose(d[i, :m, 2], ref["q_s"][i, :m], atol=TOL, rtol=0)
        np.testing.assert_allclose(d[i, :m, 3], ref["p_s"][i, :m], atol=TOL, rtol=0)
        np.testing.assert_allclose(d[i, 0, 7], ref["residual_mass"][i], atol=TOL, rtol=0)


@pytest.mark.parametrize("round_idx", [0, 1])
def test_lazy_plain_config(round_idx):
    w = W.scaled(W.PLAIN, B=128)
    inp = make_inputs(w, round_idx)
    ref = oracle_verify(inp, w)
    out = run(inp, w, lazy=True)
    check(w, inp, ref, out)
    assert out[3]["rows"] == expected_rows(out[0], inp["T"], w.K)


def test_lazy_large_batch_small_B():
    w = W.scaled(W.LARGE_BATCH, B=24)
    inp = make_inputs(w, 0)
    ref = oracle_verify(inp, w)
    out = run(inp, w, lazy=True)
    check(w, inp, ref, out)


def test_lazy_full_batch_equals_eager_and_reads_fewer_rows():
    """B=512 workload: identical outputs to sv_verify for every sequence; a sample against the
    oracle; fewer rows read, exactly as many as the first rejections imply."""
    w = W.LARGE_BATCH
    inp = make_inputs(w, 2, chunk=64)
    lz = run(inp, w, lazy=True)
    eg = run(inp, w, lazy=False)
    np.testing.assert_array_equal(lz[0], eg[0])
    np.testing.assert_array_equal(lz[1], eg[1])
    seqs = np.array([0, 1, 2, 3, 254, 255, 256, 257, 510, 511])
    check(w, inp, oracle_verify(inp, w, seqs=seqs), lz, seqs=seqs)
    assert lz[3]["rows"] == expected_rows(lz[0], inp["T"], w.K)
    assert lz[3]["rows"] < 0.5 * eg[3]["rows"]
    assert lz[3]["draws"] == eg[3]["draws"] == 256


def test_lazy_repeated_calls_reuse_the_workspace():
    w = W.scaled(W.LARGE_BATCH, B=64)
    inp = make_inputs(w, 3)
    ref = oracle_verify(inp, w)
    for _ in range(3):
        check(w, inp, ref, run(inp, w, lazy=True))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_lazy_masked_logits(dtype):
    rng = np.random.default_rng(12)
    B, K, V = 40, 3, 3000
    x = rng.normal(0, 2, (B, K + 1, V))
    y = 0.7 * x[:, :K] + rng.normal(0, 1, (B, K, V))
    x[rng.random(x.shape) < 0.3] = -np.inf
    y[rng.random(y.shape) < 0.3] = -np.inf
    tg = torch.as_tensor(x, dtype=dtype, device="cuda")
    dr = torch.as_tensor(y, dtype=dtype, device="cuda")
    T = np.where(np.arange(B) % 3 == 0, 0.0, np.where(np.arange(B) % 3 == 1, 1.0, 0.7)).astype(np.float32)
    d64 = to_f64(dr)
    toks = oracle.draft_sample(d64, rng.random((B, K)), T, np.ones(B))["tokens"]
    u = rng.random((B, K + 1))
    w = W.Workload("masked", B=B, K=K, V=V, dtype="f32" if dtype == torch.float32 else "bf16", temperature=1.0,
                   top_p=1.0, rounds=1, seed=0, sigma=2.0, draft_scale=0.7, draft_sigma=1.0)
    inp = dict(target=tg, draft=dr, tokens=toks, u=u, T=T, top_p=np.ones(B, np.float32))
    ref = oracle.verify(to_f64(tg), d64, toks, u, T, np.ones(B))
    check(w, inp, ref, run(inp, w, lazy=True))


def test_lazy_all_accepted_and_k0():
    """Draft equal to target: every test accepts, so every row is read and the bonus draw comes
    from row K; K = 0: only the bonus draw."""
    rng = np.random.default_rng(8)
    B, K, V = 32, 4, 2048
    tg = torch.as_tensor(rng.normal(0, 2, (B, K + 1, V)), dtype=torch.float32, device="cuda")
    u = rng.random((B, K + 1))
    T = np.ones(B, np.float32)
    toks = rng.integers(0, V, (B, K))
    a = dict(draft_tokens=torch.as_tensor(toks, dtype=torch.int32, device="cuda"),
             uniforms=torch.as_tensor(u, device="cuda"), temperature=torch.as_tensor(T, device="cuda"))
    al, ot, _, st = sv.sv_verify(tg, tg[:, :K].clone(), a["draft_tokens"], a["uniforms"], a["temperature"],
                                 lazy=True)
    ref = oracle.verify(to_f64(tg), to_f64(tg[:, :K]), toks, u, T, np.ones(B))
    assert (al.cpu().numpy() == K).all()
    np.testing.assert_array_equal(ot.cpu().numpy(), ref["out_tokens"])
    assert sv.read_stats(st)["rows"] == B * (2 * K + 1)
    al0, ot0, _, st0 = sv.sv_verify(tg[:, :1].contiguous(), None, None, a["uniforms"][:, :1].contiguous(),
                                    a["temperature"], lazy=True)
    ref0 = oracle.verify(to_f64(tg[:, :1]), np.zeros((B, 0, V)), np.zeros((B, 0), int), u[:, :1], T, np.ones(B))
    np.testing.assert_array_equal(ot0.cpu().numpy(), ref0["out_tokens"])
    assert sv.read_stats(st0)["status"] == 0


def test_lazy_top_p_runs_the_full_pipeline():
    w = W.scaled(W.SAMPLED_TOPP, B=8)
    inp = make_inputs(w, 0)
    lz = run(inp, w, lazy=True, top_p=True)
    eg = run(inp, w, lazy=False, top_p=True)
    np.testing.assert_array_equal(lz[0], eg[0])
    np.testing.assert_array_equal(lz[1], eg[1])
    assert lz[3]["rows"] == eg[3]["rows"]


def test_lazy_device_errors():
    w = W.scaled(W.PLAIN, B=8)
    inp = make_inputs(w, 0)
    a = gpu_args(inp)
    bad = a["draft_tokens"].clone()
    bad[3, 2] = w.V + 5
    al, ot, _, st = sv.sv_verify(inp["target"], inp["draft"], bad, a["uniforms"], a["temperature"], lazy=True)
    torch.cuda.synchronize()
    s = sv.read_stats(st)
    assert s["status"] == sv._abi.SV_ERR_BAD_TOKEN and s["error_index"] == 3
    assert (ot.cpu().numpy()[3] == -1).all()
    T = a["temperature"].clone()
    T[5] = -1.0
    al, ot, _, st = sv.sv_verify(inp["target"], inp["draft"], a["draft_tokens"], a["uniforms"], T, lazy=True)
    torch.cuda.synchronize()
    s = sv.read_stats(st)
    assert s["status"] == sv._abi.SV_ERR_INVALID_ARG and s["error_index"] == 5
