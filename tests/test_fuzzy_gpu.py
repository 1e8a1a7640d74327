"""sv_fuzzy_verify on the GPU (through the C ABI) against the float64 oracle: one verification
stage of three-model speculative decoding, fuzzy (divergence threshold) and assisted modes."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_gb300 as sv
from synth import workloads as W
from tests.helpers import to_f64

pytestmark = pytest.mark.gpu
DIV_TOL = 1e-5   # the float32 divergence's certified bound is a few 1e-6


def stage_inputs(w, round_idx=0, greedy_every=0):
    """Verifier / drafter logits from the workload generator, drafted tokens from the oracle's
    sampler of the drafter's distribution, uniforms, temperatures."""
    ver, drf = W.logits(w, round_idx, device="cuda")
    u_draft, u, _ = W.round_uniforms(w, round_idx)
    T = W.temperatures(w)
    if greedy_every:
        T[::greedy_every] = 0.0
    toks = np.zeros((w.B, w.K), dtype=np.int64)
    for b0 in range(0, w.B, 16):
        d64 = to_f64(drf[b0:b0 + 16, : w.K])
        toks[b0:b0 + 16] = oracle.draft_sample(d64, u_draft[b0:b0 + 16, : w.K], T[b0:b0 + 16],
                                               np.ones(len(d64)))["tokens"]
    return ver, drf, toks, u, T


def run(ver, drf, toks, u, T, tau, mode="divergence"):
    al, ot, div, st = sv.sv_fuzzy_verify(ver, drf, torch.as_tensor(toks, dtype=torch.int32, device="cuda"),
                                         torch.as_tensor(u, device="cuda"), torch.as_tensor(T, device="cuda"),
                                         tau=tau, mode=mode, divergence=mode == "divergence")
    torch.cuda.synchronize()
    return (al.cpu().numpy(), ot.cpu().numpy(), None if div is None else div.cpu().numpy(), sv.read_stats(st))


def reference(ver, drf, toks, u, T, tau, mode="divergence", seqs=None, chunk=8):
    seqs = np.arange(ver.shape[0]) if seqs is None else np.asarray(seqs)
    parts = []
    for i in range(0, len(seqs), chunk):
        sel = torch.as_tensor(seqs[i:i + chunk], device=ver.device)
        K = toks.shape[1]
        parts.append(oracle.fuzzy_verify(to_f64(ver.index_select(0, sel)), to_f64(drf.index_select(0, sel)[:, :K]),
                                         toks[seqs[i:i + chunk]], u[seqs[i:i + chunk]], T[seqs[i:i + chunk]], tau,
                                         mode=mode))
    return {k: np.concatenate([p[k] for p in parts]) for k in parts[0]}


def check(out, ref, seqs=None):
    al, ot, div, st = out
    seqs = np.arange(len(al)) if seqs is None else np.asarray(seqs)
    assert st["status"] == 0, st
    assert st["unresolved"] == 0, st
    np.testing.assert_array_equal(al[seqs], ref["accept_len"])
    np.testing.assert_array_equal(ot[seqs], ref["out_tokens"])
    if div is not None:
        K = div.shape[1]
        for i, b in enumerate(seqs):
            n = min(int(al[b]) + 1, K)          # positions the stage reached
            np.testing.assert_allclose(div[b, :n], ref["div"][i, :n], atol=DIV_TOL, rtol=0)


@pytest.mark.parametrize("tau", [0.5, 0.3, 1.0, -0.1])
def test_divergence_mode_qualifier_to_target(tau):
    w = W.scaled(W.PYRAMID_QT, B=12)
    ver, drf, toks, u, T = stage_inputs(w, 0, greedy_every=4)
    check(run(ver, drf, toks, u, T, tau), reference(ver, drf, toks, u, T, tau))


def test_divergence_mode_draft_to_qualifier_f32():
    w = W.scaled(W.PYRAMID_DQ, B=16, V=5000, dtype="f32")
    ver, drf, toks, u, T = stage_inputs(w, 1, greedy_every=3)
    tau = w.extra["tau"]
    check(run(ver, drf, toks, u, T, tau), reference(ver, drf, toks, u, T, tau))


def test_divergence_mode_full_stage_sampled_check():
    """B=64, K=25 (the qualifier -> target stage): every sequence's accept length and tokens
    against the oracle on a sample of sequences, and the rows-read count."""
    w = W.PYRAMID_QT
    ver, drf, toks, u, T = stage_inputs(w, 2)
    out = run(ver, drf, toks, u, T, w.extra["tau"])
    seqs = [0, 1, 31, 32, 62, 63]
    check(out, reference(ver, drf, toks, u, T, w.extra["tau"], seqs=seqs), seqs=seqs)
    assert out[3]["rows"] == w.B * (2 * w.K + 1)
    assert 0 < out[0].mean() < w.K                     # a real mix of acceptance lengths


def test_divergence_too_close_to_tau_goes_float_float():
    """tau set to the oracle's own divergence of one position (rounded to float32): the float32
    bound cannot place that position, the float-float pass decides it, and the outputs still
    equal the oracle's."""
    w = W.scaled(W.PYRAMID_QT, B=4, K=6, V=20000)
    ver, drf, toks, u, T = stage_inputs(w, 3)
    ref0 = reference(ver, drf, toks, u, T, 2.0)            # every position reached: all divergences
    tau = float(np.float32(ref0["div"][1, 0]))
    out = run(ver, drf, toks, u, T, tau)
    assert out[3]["reresolved"] >= 1, out[3]
    check(out, reference(ver, drf, toks, u, T, tau))


def test_greedy_sequences_compare_argmaxes():
    w = W.scaled(W.PYRAMID_DQ, B=16, V=3000)
    ver, drf, toks, u, T = stage_inputs(w, 4)
    T[:] = 0.0
    for tau in (0.0, 0.5, 1.0):
        out = run(ver, drf, toks, u, T, tau)
        ref = reference(ver, drf, toks, u, T, tau)
        check(out, ref)
        assert set(np.unique(out[2][~np.isnan(out[2])])) <= {0.0, 1.0}


@pytest.mark.parametrize("greedy_every", [0, 3])
def test_assisted_mode(greedy_every):
    w = W.scaled(W.PYRAMID_DQ, B=24)
    ver, drf, toks, u, T = stage_inputs(w, 5, greedy_every=greedy_every)
    check(run(ver, drf, toks, u, T, 0.0, mode="assisted"), reference(ver, drf, toks, u, T, 0.0, mode="assisted"))


def test_k0_and_errors():
    w = W.scaled(W.PYRAMID_DQ, B=8, K=4, V=2048)
    ver, drf, toks, u, T = stage_inputs(w, 6)
    al, ot, _, st = run(ver[:, :1].contiguous(), drf, toks[:, :0], u[:, :1].copy(), T, 0.5)
    ref = reference(ver[:, :1].contiguous(), drf, toks[:, :0], u[:, :1].copy(), T, 0.5)
    np.testing.assert_array_equal(ot, ref["out_tokens"])
    bad = toks.copy()
    bad[2, 1] = w.V + 7
    _, ot, _, st = run(ver, drf, bad, u, T, 0.5)
    assert st["status"] == sv._abi.SV_ERR_BAD_TOKEN and st["error_index"] == 2
    assert (ot[2] == -1).all()
    T2 = T.copy()
    T2[5] = -2.0
    _, _, _, st = run(ver, drf, toks, u, T2, 0.5)
    assert st["status"] == sv._abi.SV_ERR_INVALID_ARG and st["error_index"] == 5


@pytest.mark.parametrize("greedy_every", [0, 4])
def test_assisted_mode_full_stage_k25(greedy_every):
    """The assisted mode at the qualifier -> target stage's full size (B=64, K=25, V=128256 bf16),
    as the benchmark runs it: every sequence against the oracle.  With greedy_every=4 a quarter of
    the sequences are greedy."""
    w = W.PYRAMID_QT
    ver, drf, toks, u, T = stage_inputs(w, 7, greedy_every=greedy_every)
    out = run(ver, drf, toks, u, T, 0.0, mode="assisted")
    check(out, reference(ver, drf, toks, u, T, 0.0, mode="assisted", chunk=4))
    assert out[0].max() >= 3                           # positions deep into the 25 are reached
