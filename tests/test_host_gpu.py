"""sv_verify_host (inputs and outputs in host memory) on the GPU: the same outputs as sv_verify on
device copies and as the float64 oracle; only the rows the verification reads are copied."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_gb300 as sv
from tests.helpers import to_f64

pytestmark = pytest.mark.gpu


def on_device(t):
    """A CUDA copy of [B, R, V] logits on rows padded to 64 elements (16-byte rows for any V)."""
    B, R, V = t.shape
    buf = torch.zeros((B, R, (V + 63) // 64 * 64), dtype=t.dtype, device="cuda")
    buf[:, :, :V] = t.cuda()
    return buf[:, :, :V]


def case(rng, B, K, V, dt, extra_rows=0, greedy_every=3):
    x = rng.normal(0, 2.5, (B, K + 1, V))
    y = 0.7 * x[:, : K + extra_rows if K else 1] + rng.normal(0, 1.3, (B, K + extra_rows if K else 1, V))
    tg = torch.as_tensor(x, dtype=dt)
    dr = torch.as_tensor(y, dtype=dt)
    T = np.where(np.arange(B) % greedy_every == 0, 0.0, 0.9).astype(np.float32)
    d64 = to_f64(dr)
    toks = oracle.draft_sample(d64[:, :K], rng.random((B, K)), T, np.ones(B))["tokens"] if K else np.zeros((B, 0))
    u = rng.random((B, K + 1))
    return tg, dr, toks.astype(np.int32), u, T


@pytest.mark.parametrize("dt,V,pinned,extra", [(torch.bfloat16, 5003, True, 0), (torch.float32, 4097, False, 1),
                                               (torch.bfloat16, 128256, True, 0)])
def test_host_entry_matches_device_entry_and_oracle(dt, V, pinned, extra):
    rng = np.random.default_rng(V)
    B, K = 12, 4
    tg, dr, toks, u, T = case(rng, B, K, V, dt, extra)
    host = [torch.as_tensor(a) for a in (toks, u, T)]
    args = [tg, dr] + host
    if pinned:
        args = [a.pin_memory() for a in args]
    al_h, ot_h, st, moved = sv.sv_verify_host(*args)
    torch.cuda.synchronize()
    s = sv.read_stats(st)
    assert s["status"] == 0, s
    # device entry on device copies
    al_d, ot_d, _, _ = sv.sv_verify(on_device(tg), on_device(dr), *(torch.as_tensor(a).cuda() for a in (toks, u, T)))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(al_h.numpy(), al_d.cpu().numpy())
    np.testing.assert_array_equal(ot_h.numpy(), ot_d.cpu().numpy())
    ref = oracle.verify(to_f64(tg), to_f64(dr), toks, u, T, np.ones(B))
    np.testing.assert_array_equal(al_h.numpy(), ref["accept_len"])
    np.testing.assert_array_equal(ot_h.numpy(), ref["out_tokens"])
    es = tg.element_size()
    sampled = int((T != 0).sum())
    want = (B * (K + 1) + sampled * K) * V * es + B * K * 4 + B * (K + 1) * 8 + B * 4
    assert moved == want, (moved, want)


def test_host_entry_with_filters():
    rng = np.random.default_rng(9)
    B, K, V = 8, 3, 3001
    tg, dr, toks, u, T = case(rng, B, K, V, torch.bfloat16, greedy_every=4)
    tp = np.full(B, 0.85, np.float32)
    tk = np.full(B, 40, np.int32)
    al_h, ot_h, st, _ = sv.sv_verify_host(tg.pin_memory(), dr.pin_memory(), torch.as_tensor(toks), torch.as_tensor(u),
                                          torch.as_tensor(T), top_p=torch.as_tensor(tp), top_k=torch.as_tensor(tk))
    torch.cuda.synchronize()
    assert sv.read_stats(st)["status"] == 0
    ref = oracle.verify(to_f64(tg), to_f64(dr), toks, u, T, tp, top_k=tk)
    np.testing.assert_array_equal(al_h.numpy(), ref["accept_len"])
    np.testing.assert_array_equal(ot_h.numpy(), ref["out_tokens"])


def test_host_entry_without_draft_tokens():
    rng = np.random.default_rng(10)
    B, V = 5, 2000
    tg = torch.as_tensor(rng.normal(0, 2, (B, 1, V)), dtype=torch.float32)
    T = np.where(np.arange(B) % 2 == 0, 0.0, 1.0).astype(np.float32)
    u = rng.random((B, 1))
    al_h, ot_h, st, moved = sv.sv_verify_host(tg, tg, torch.zeros((B, 0), dtype=torch.int32), torch.as_tensor(u),
                                              torch.as_tensor(T))
    torch.cuda.synchronize()
    assert sv.read_stats(st)["status"] == 0
    ref = oracle.verify(to_f64(tg), to_f64(tg), np.zeros((B, 0), np.int64), u, T, np.ones(B))
    np.testing.assert_array_equal(ot_h.numpy(), ref["out_tokens"])
    assert (al_h.numpy() == 0).all()
    assert moved == B * V * 4 + B * 8 + B * 4


def test_host_entry_rejects_device_tensors():
    t = torch.zeros((2, 2, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(TypeError):
        sv.sv_verify_host(t, t, torch.zeros((2, 1), dtype=torch.int32), torch.zeros((2, 2), dtype=torch.float64),
                          torch.ones(2, dtype=torch.float32))
