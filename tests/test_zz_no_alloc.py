"""sv_verify_static: verification without a caller workspace and without any allocation.

Some callers cannot allocate device memory when they verify: a serving engine whose KV-cache
pool took all free HBM at start-up, or a host program that loads the library as a plug-in
and owns every allocation.  sv_verify_static serves them from a fixed 32 MiB scratch array
inside the library.  These tests call it through the C ABI (the ctypes binding) twice in a
row and check each result against sv_verify with its own workspace on the same inputs.

The file name puts it last in collection order, after every other test.
"""

import numpy as np
import pytest
import torch

import speculative_decoding_verification_gb300 as sv
from speculative_decoding_verification_gb300 import _abi
from synth import workloads as W
from tests.helpers import gpu_args, make_inputs

def test_oversize_call_is_refused_before_device_work():
    """B=4096, K=5, V=128256 bf16 needs more scratch than the library's fixed array holds: refused
    with SV_ERR_WORKSPACE, on any machine, before the library touches a device (the pointers
    below are never dereferenced)."""
    from speculative_decoding_verification_gb300 import build
    build.build()
    lib = sv.load()
    fake = 1 << 20
    B, K, V = 4096, 5, 128256
    assert lib.sv_verify_workspace_size(B, K, V) > _abi.SV_STATIC_SCRATCH_BYTES
    code = lib.sv_verify_static(fake, V, fake, V, K, _abi.SV_BF16, fake, fake, B, K, V, fake, None, None, 0, 1.0,
                                fake, fake, None, None, None)
    assert code == _abi.SV_ERR_WORKSPACE
    assert lib.sv_verify_static(fake, V, fake, V, K, 7, fake, fake, 4, K, V, fake, None, None, 0, 1.0, fake, fake,
                                None, None, None) == _abi.SV_ERR_INVALID_ARG


def _outputs(B, K, dev):
    return (torch.empty(B, dtype=torch.int32, device=dev), torch.empty((B, K + 1), dtype=torch.int32, device=dev),
            torch.empty((B, K + 1, _abi.SV_DEBUG_FIELDS), dtype=torch.float64, device=dev), sv.new_stats(dev))


def _call(fn, inp, w, top_p, outs=None):
    a = gpu_args(inp)
    tp = torch.as_tensor(inp["top_p"], dtype=torch.float32, device="cuda") if top_p else None
    kw = dict(top_p=tp, saguaro_F=w.saguaro_F, saguaro_C=w.saguaro_C)
    if outs is None:
        return fn(inp["target"], inp["draft"], a["draft_tokens"], a["uniforms"], a["temperature"], debug=True, **kw)
    al, ot, dbg, st = outs
    return fn(inp["target"], inp["draft"], a["draft_tokens"], a["uniforms"], a["temperature"], accept_len=al,
              out_tokens=ot, debug=dbg, stats=st, **kw)


def _check_same(ref, got, w):
    """Outputs, counters and debug fields equal sv_verify's bit for bit.  The two calls run the
    same kernels on the same inputs, and every value they compute has a fixed place and a fixed
    order of summation, so leftovers of an earlier call in the shared scratch would show up as a
    difference here.  One field may differ in its last bits: the float-float tier's R (residual
    mass) adds the few tokens whose sign it had to settle exactly in the order they were queued by
    atomics, so there R is held to 1e-12 relative (its float-float sums carry about 2^-44)."""
    ral, rot, rdbg, rst = ref
    gal, got_, gdbg, gst = got
    torch.cuda.synchronize()
    rs, gs = sv.read_stats(rst), sv.read_stats(gst)
    assert rs["status"] == 0 and gs["status"] == 0, (rs, gs)
    np.testing.assert_array_equal(gal.cpu().numpy(), ral.cpu().numpy())
    np.testing.assert_array_equal(got_.cpu().numpy(), rot.cpu().numpy())
    rd, gd = rdbg.cpu().numpy(), gdbg.cpu().numpy()
    r_field = _abi.DBG["R"]
    others = [f for f in range(rd.shape[-1]) if f != r_field]
    np.testing.assert_array_equal(gd[..., others], rd[..., others])
    np.testing.assert_allclose(gd[..., r_field], rd[..., r_field], rtol=1e-12, atol=0)
    for k in ("rows", "accept_tests", "draws", "reresolved", "near_boundary", "unresolved"):
        assert gs[k] == rs[k], k


@pytest.mark.gpu
def test_two_calls_in_a_row_match_sv_verify():
    """Call 1: Saguaro draft transform (F=8, C=0.3) with top-p on B=16, V=128256.  Call 2: the
    full B=512, K=5, V=128256 half-greedy batch, which finds call 1's leftovers in the shared
    scratch.  Each must equal sv_verify on the same inputs; the second call allocates nothing."""
    w1 = W.SAGUARO
    inp1 = make_inputs(w1, 0)
    w2 = W.LARGE_BATCH
    inp2 = make_inputs(w2, 1, chunk=64)

    ref1 = _call(sv.sv_verify, inp1, w1, top_p=True)
    ref2 = _call(sv.sv_verify, inp2, w2, top_p=False)
    torch.cuda.synchronize()

    outs1 = _outputs(w1.B, w1.K, "cuda")
    outs2 = _outputs(w2.B, w2.K, "cuda")
    got1 = _call(sv.sv_verify_static, inp1, w1, top_p=True, outs=outs1)
    torch.cuda.synchronize()
    # The device address of the scratch is known now; the second call must not allocate.
    a2 = gpu_args(inp2)
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    torch_before = torch.cuda.memory_allocated()
    got2 = sv.sv_verify_static(inp2["target"], inp2["draft"], a2["draft_tokens"], a2["uniforms"], a2["temperature"],
                               saguaro_F=w2.saguaro_F, saguaro_C=w2.saguaro_C, accept_len=outs2[0],
                               out_tokens=outs2[1], debug=outs2[2], stats=outs2[3])
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == torch_before
    assert torch.cuda.mem_get_info()[0] == free_before

    _check_same(ref1, got1, w1)
    _check_same(ref2, got2, w2)


@pytest.mark.gpu
def test_repeat_on_same_inputs_is_identical():
    """Two calls in a row on the sampled top-p batch (B=8, K=5, V=128256, T=0.8, top-p=0.9):
    both equal sv_verify, so nothing the first call left in the scratch leaks into the second."""
    w = W.SAMPLED_TOPP
    inp = make_inputs(w, 2)
    ref = _call(sv.sv_verify, inp, w, top_p=True)
    for _ in range(2):
        got = _call(sv.sv_verify_static, inp, w, top_p=True, outs=_outputs(w.B, w.K, "cuda"))
        _check_same(ref, got, w)


@pytest.mark.gpu
def test_fp32_rounds_match_sv_verify():
    """The float32 recipe (B=1, K=4, V=32000, T=1): two rounds in a row, whose scratch layout
    differs from the bf16 calls' above; each equals sv_verify on the same inputs."""
    w = W.PLAIN
    for r in range(2):
        inp = make_inputs(w, r)
        ref = _call(sv.sv_verify, inp, w, top_p=False)
        got = _call(sv.sv_verify_static, inp, w, top_p=False, outs=_outputs(w.B, w.K, "cuda"))
        _check_same(ref, got, w)
