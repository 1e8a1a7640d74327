"""libspecverify Python binding: argument marshalling for the C ABI, nothing else.

Every function here forwards to the entry point of the same name in libspecverify.so (built
for sm_103a by ``build.build()``).  Tensors are torch CUDA tensors; torch supplies device
memory and the current stream, the computation runs in the library's kernels.  If the shared
library is absent, importing the binding still works but every call raises ImportError; no
other implementation stands in.
"""
from __future__ import annotations

import ctypes

import torch

from . import _abi
from ._abi import (DBG, SV_BF16, SV_F32, SV_MAX_K, STATS_BYTES, STATS_FIELDS, SvError,  # noqa: F401
                   load, status_string)

__all__ = ["sv_verify", "sv_saguaro_sample", "sv_fanout", "sv_cache_keys", "sv_cache_lookup", "sv_topk_rows",
           "sv_mirror_reuse", "sv_selftest_timeout", "sv_selftest_exp2", "read_stats", "load", "status_string",
           "SvError", "Workspace"]


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(stream, dev):
    """The stream a call runs on: the caller's, which must belong to `dev`, or dev's current one.
    The library launches on this stream and plans for the current device, so the two agree."""
    if stream is None:
        s = torch.cuda.current_stream(dev)
    else:
        s = stream
        if s.device != dev:
            raise ValueError(f"the stream is on {s.device}, the call's arrays on {dev}")
    return ctypes.c_void_p(s.cuda_stream)


def _on(dev, fn, *args):
    """Call the library with `dev` current: it takes the device of its workspace plan, static
    scratch and SM count from the current device."""
    with torch.cuda.device(dev):
        return fn(*args)


def _dtype_code(t):
    if t.dtype == torch.float32:
        return SV_F32
    if t.dtype == torch.bfloat16:
        return SV_BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


def _rows(t, name):
    """(row pitch in elements, rows per sequence) of a [B, R, V] or [N, V] logit tensor."""
    if t.stride(-1) != 1:
        raise ValueError(f"{name}: the vocabulary axis must be contiguous")
    if t.dim() == 3:
        if t.shape[1] > 1 and t.stride(0) != t.shape[1] * t.stride(1):
            raise ValueError(f"{name}: rows of a sequence must be consecutive rows of one pitch")
        pitch = t.stride(1) if t.shape[1] > 1 else t.stride(0)
        return pitch, t.shape[1]
    if t.dim() == 2:
        return t.stride(0), 1
    raise ValueError(f"{name}: expected [B, R, V] or [N, V]")


class Workspace:
    """A caller-owned device workspace (torch memory) reused across calls on one stream."""

    def __init__(self):
        self._buf = {}

    def get(self, nbytes: int, device) -> torch.Tensor:
        key = torch.device(device)
        buf = self._buf.get(key)
        if buf is None or buf.numel() < nbytes:
            buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
            self._buf[key] = buf
        return buf


_default_ws = Workspace()


def new_stats(device) -> torch.Tensor:
    return torch.zeros(STATS_BYTES, dtype=torch.uint8, device=device)


def read_stats(t: torch.Tensor) -> dict:
    """Decode an sv_stats block (synchronises with the device)."""
    raw = t.detach().cpu()
    i32 = raw.view(torch.int32)
    i64 = raw.view(torch.int64)
    out = {"status": int(i32[0]), "error_index": int(i32[1])}
    for k, name in enumerate(STATS_FIELDS[2:]):
        out[name] = int(i64[1 + k])
    return out


def _cuda(t, name):
    """The CUDA device of a logit tensor: the device entry points read device memory only."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor (host buffers go through sv_verify_host)")
    return t.device


def _arr(t, name, dtype, n, dev):
    """t as the library reads or writes it: a contiguous `dtype` tensor on `dev` holding at least
    n elements.  Anything else would be read with the wrong layout or past its end, so it is
    refused here, before any work is queued."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device != dev:
        raise ValueError(f"{name} must be on {dev}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.numel() < n:
        raise ValueError(f"{name} holds {t.numel()} elements, needs {n}")
    return t


def _opt(t, name, dtype, n, dev):
    return None if t is None else _arr(t, name, dtype, n, dev)


def _out(t, name, dtype, shape, dev):
    """An output array: allocated when the caller passes none, else checked like an input."""
    if t is None:
        return torch.empty(shape, dtype=dtype, device=dev)
    n = 1
    for d in shape:
        n *= d
    return _arr(t, name, dtype, n, dev)


def _pair(first, second, names, K, dev):
    """Row pitch and rows of the first logit tensor and, when K > 0, of the second (same dtype and
    device); with K = 0 the second is not read and its pointer is null."""
    f_pitch, _ = _rows(first, names[0])
    if K == 0:
        return f_pitch, f_pitch, 1, ctypes.c_void_p(0)
    if _cuda(second, names[1]) != dev:
        raise ValueError(f"{names[0]} and {names[1]} must be on one device")
    if second.dtype != first.dtype:
        raise TypeError(f"{names[0]} and {names[1]} logits must share a dtype")
    s_pitch, s_rows = _rows(second, names[1])
    return f_pitch, s_pitch, s_rows, _ptr(second)


def _seq_inputs(draft_tokens, uniforms, temperature, top_p, top_k, B, K, dev):
    """The per-sequence inputs of the verify entry points, checked (draft tokens only when K > 0)."""
    if K > 0:
        _arr(draft_tokens, "draft_tokens", torch.int32, B * K, dev)
    _arr(uniforms, "uniforms", torch.float64, B * (K + 1), dev)
    _arr(temperature, "temperature", torch.float32, B, dev)
    _opt(top_p, "top_p", torch.float32, B, dev)
    _opt(top_k, "top_k", torch.int32, B, dev)


def _stats(stats, dev):
    return new_stats(dev) if stats is None else _arr(stats, "stats", torch.uint8, STATS_BYTES, dev)


def sv_verify(target, draft, draft_tokens, uniforms, temperature, top_p=None, saguaro_F=0, saguaro_C=1.0,
              accept_len=None, out_tokens=None, debug=False, stats=None, workspace=None, stream=None, lazy=False,
              top_k=None):
    """sv_verify (or, with lazy=True, sv_verify_lazy: same outputs, rows after each sequence's
    first rejection left unread) on torch CUDA tensors.

    target [B, K+1, V] and draft [B, R>=K, V] (float32 or bfloat16, same dtype); draft_tokens
    int32 [B, K]; uniforms float64 [B, K+1]; temperature float32 [B]; top_p float32 [B] or None;
    top_k int32 [B] or None (top-k acts before top-p).
    Returns (accept_len int32 [B], out_tokens int32 [B, K+1], debug float64 [B, K+1, 8] or None,
    stats uint8 block).
    """
    lib = load()
    B, K1, V = target.shape
    K = K1 - 1
    dev = _cuda(target, "target")
    t_pitch, d_pitch, d_rows, d_ptr = _pair(target, draft, ("target", "draft"), K, dev)
    _seq_inputs(draft_tokens, uniforms, temperature, top_p, top_k, B, K, dev)
    accept_len = _out(accept_len, "accept_len", torch.int32, (B,), dev)
    out_tokens = _out(out_tokens, "out_tokens", torch.int32, (B, K + 1), dev)
    dbg = torch.empty((B, K + 1, _abi.SV_DEBUG_FIELDS), dtype=torch.float64, device=dev) if debug else None
    stats = _stats(stats, dev)
    ws_bytes = lib.sv_verify_workspace_size(B, K, V)
    ws = (workspace or _default_ws).get(ws_bytes, dev)
    fn = lib.sv_verify_lazy if lazy else lib.sv_verify
    code = _on(dev, fn, _ptr(target), t_pitch, d_ptr, d_pitch, d_rows, _dtype_code(target),
              _ptr(draft_tokens if K > 0 else None), _ptr(uniforms), B, K, V, _ptr(temperature),
              _ptr(top_p), _ptr(top_k), int(saguaro_F), float(saguaro_C), _ptr(accept_len),
              _ptr(out_tokens), _ptr(dbg), _ptr(stats), _ptr(ws), ws.numel(), _stream(stream, dev))
    _abi.check("sv_verify_lazy" if lazy else "sv_verify", code)
    return accept_len, out_tokens, dbg, stats


def sv_verify_host(target, draft, draft_tokens, uniforms, temperature, top_p=None, saguaro_F=0, saguaro_C=1.0,
                   accept_len=None, out_tokens=None, stats=None, workspace=None, stream=None, top_k=None,
                   device=None):
    """sv_verify_host on host (CPU) tensors: the library copies the rows the verification reads
    (every target row; the draft rows of sequences with a nonzero temperature) and the small
    inputs to the device, verifies there, and copies the outputs back, all on `stream`.

    Pinned tensors (tensor.pin_memory()) make the copies asynchronous and full-speed.  target
    [B, K+1, V] and draft [B, R>=K, V] (float32 or bfloat16); draft_tokens int32 [B, K]; uniforms
    float64 [B, K+1]; temperature float32 [B]; top_p float32 [B] or None; top_k int32 [B] or
    None.  Returns (accept_len int32 [B], out_tokens int32 [B, K+1]) as CPU tensors, valid once
    the stream has synchronised, the stats block (device) and the bytes copied to the device."""
    lib = load()
    for name, t in (("target", target), ("draft", draft), ("draft_tokens", draft_tokens), ("uniforms", uniforms),
                    ("temperature", temperature), ("top_p", top_p), ("top_k", top_k)):
        if t is not None and t.is_cuda:
            raise TypeError(f"sv_verify_host: {name} must be a host tensor")
    dev = torch.device(device if device is not None else "cuda")
    if dev.index is None:
        dev = torch.device(dev.type, torch.cuda.current_device())
    B, K1, V = target.shape
    K = K1 - 1
    t_pitch, _ = _rows(target, "target")
    if K > 0:
        if draft.dtype != target.dtype:
            raise TypeError("target and draft logits must share a dtype")
        d_pitch, d_rows = _rows(draft, "draft")
        d_ptr = _ptr(draft)
    else:
        d_pitch, d_rows, d_ptr = t_pitch, 1, ctypes.c_void_p(0)
    pin = target.is_pinned()
    if accept_len is None:
        accept_len = torch.empty(B, dtype=torch.int32, pin_memory=pin)
    if out_tokens is None:
        out_tokens = torch.empty((B, K + 1), dtype=torch.int32, pin_memory=pin)
    host = torch.device("cpu")
    for name, t, dt, n in (("draft_tokens", draft_tokens if K > 0 else None, torch.int32, B * K),
                           ("uniforms", uniforms, torch.float64, B * (K + 1)),
                           ("temperature", temperature, torch.float32, B), ("top_p", top_p, torch.float32, B),
                           ("top_k", top_k, torch.int32, B), ("accept_len", accept_len, torch.int32, B),
                           ("out_tokens", out_tokens, torch.int32, B * (K + 1))):
        _opt(t, name, dt, n, host)
    stats = _stats(stats, dev)
    ws_bytes = lib.sv_verify_host_workspace_size(B, K, V, _dtype_code(target))
    ws = (workspace or _default_ws).get(ws_bytes, dev)
    moved = ctypes.c_size_t(0)
    code = _on(dev, lib.sv_verify_host, _ptr(target), t_pitch, d_ptr, d_pitch, d_rows, _dtype_code(target),
                              _ptr(draft_tokens if K > 0 else None), _ptr(uniforms), B, K, V, _ptr(temperature),
                              _ptr(top_p), _ptr(top_k), int(saguaro_F), float(saguaro_C), _ptr(accept_len),
                              _ptr(out_tokens), _ptr(stats), _ptr(ws), ws.numel(), ctypes.c_void_p(ctypes.addressof(moved)),
                              _stream(stream, dev))
    _abi.check("sv_verify_host", code)
    return accept_len, out_tokens, stats, moved.value


def sv_verify_static(target, draft, draft_tokens, uniforms, temperature, top_p=None, saguaro_F=0, saguaro_C=1.0,
                     accept_len=None, out_tokens=None, debug=None, stats=None, stream=None, top_k=None):
    """sv_verify without a workspace, for callers that cannot allocate device memory (a server
    whose KV-cache pool holds all free HBM, a host program that owns every allocation).

    The library's own scratch array (SV_STATIC_SCRATCH_BYTES, 32 MiB per device) stands in for
    the workspace, so the C call allocates nothing.  Pass accept_len int32 [B], out_tokens int32
    [B, K+1], stats (new_stats) and, optionally, debug float64 [B, K+1, 8] to keep this wrapper
    from allocating them.  Calls that overlap on the GPU share the scratch and race; the first
    call on a device looks up the array's address and belongs before any stream capture.
    Returns (accept_len, out_tokens, debug, stats) like sv_verify.
    """
    lib = load()
    B, K1, V = target.shape
    K = K1 - 1
    dev = _cuda(target, "target")
    t_pitch, d_pitch, d_rows, d_ptr = _pair(target, draft, ("target", "draft"), K, dev)
    _seq_inputs(draft_tokens, uniforms, temperature, top_p, top_k, B, K, dev)
    accept_len = _out(accept_len, "accept_len", torch.int32, (B,), dev)
    out_tokens = _out(out_tokens, "out_tokens", torch.int32, (B, K + 1), dev)
    if debug is True:
        debug = torch.empty((B, K + 1, _abi.SV_DEBUG_FIELDS), dtype=torch.float64, device=dev)
    elif debug is False:
        debug = None
    _opt(debug, "debug", torch.float64, B * (K + 1) * _abi.SV_DEBUG_FIELDS, dev)
    stats = _stats(stats, dev)
    code = _on(dev, lib.sv_verify_static, _ptr(target), t_pitch, d_ptr, d_pitch, d_rows, _dtype_code(target),
                                _ptr(draft_tokens if K > 0 else None), _ptr(uniforms), B, K, V, _ptr(temperature),
                                _ptr(top_p), _ptr(top_k), int(saguaro_F), float(saguaro_C), _ptr(accept_len),
                                _ptr(out_tokens), _ptr(debug), _ptr(stats), _stream(stream, dev))
    if code == _abi.SV_ERR_WORKSPACE:
        raise ValueError(f"sv_verify_static: B={B}, K={K}, V={V} needs more scratch than the "
                         f"{_abi.SV_STATIC_SCRATCH_BYTES >> 20} MiB static array; use sv_verify with a workspace")
    _abi.check("sv_verify_static", code)
    return accept_len, out_tokens, debug, stats


def sv_fuzzy_verify(verifier, drafter, draft_tokens, uniforms, temperature, tau=0.5, mode="divergence",
                    divergence=False, accept_len=None, out_tokens=None, stats=None, workspace=None, stream=None):
    """sv_fuzzy_verify: one stage of three-model speculative decoding on torch CUDA tensors.

    verifier [B, K+1, V] and drafter [B, R>=K, V] logits (same dtype); draft_tokens int32 [B, K];
    uniforms float64 [B, K+1]; temperature float32 [B]; mode "divergence" (accept while the
    Jensen-Shannon divergence <= tau) or "assisted".  Returns (accept_len, out_tokens,
    divergence float64 [B, K] or None, stats).
    """
    lib = load()
    B, K1, V = verifier.shape
    K = K1 - 1
    dev = _cuda(verifier, "verifier")
    v_pitch, d_pitch, d_rows, d_ptr = _pair(verifier, drafter, ("verifier", "drafter"), K, dev)
    _seq_inputs(draft_tokens, uniforms, temperature, None, None, B, K, dev)
    code_mode = {"divergence": _abi.SV_ACCEPT_DIVERGENCE, "assisted": _abi.SV_ACCEPT_ASSISTED}[mode]
    accept_len = _out(accept_len, "accept_len", torch.int32, (B,), dev)
    out_tokens = _out(out_tokens, "out_tokens", torch.int32, (B, K + 1), dev)
    div = torch.full((B, max(K, 1)), float("nan"), dtype=torch.float64, device=dev) if divergence else None
    stats = _stats(stats, dev)
    ws_bytes = lib.sv_fuzzy_verify_workspace_size(B, K, V)
    ws = (workspace or _default_ws).get(ws_bytes, dev)
    code = _on(dev, lib.sv_fuzzy_verify, _ptr(verifier), v_pitch, d_ptr, d_pitch, d_rows, _dtype_code(verifier),
                               _ptr(draft_tokens if K > 0 else None), _ptr(uniforms), B, K, V, _ptr(temperature),
                               float(tau), code_mode, _ptr(accept_len), _ptr(out_tokens), _ptr(div), _ptr(stats),
                               _ptr(ws), ws.numel(), _stream(stream, dev))
    _abi.check("sv_fuzzy_verify", code)
    return accept_len, out_tokens, (div[:, :K] if div is not None else None), stats


def sv_tree_verify(target, draft, parents, tokens, uniforms, temperature, accept_len=None, out_tokens=None, path=True,
                   stats=None, workspace=None, stream=None):
    """sv_tree_verify on torch CUDA tensors: target and draft [B, N+1, V] (same dtype; row i follows
    node i), parents and tokens int32 [B, N], uniforms float64 [B, N+1], temperature float32 [B].
    Returns (accept_len int32 [B], out_tokens int32 [B, N+1], path int32 [B, N] or None, stats)."""
    lib = load()
    B, N1, V = target.shape
    N = N1 - 1
    dev = _cuda(target, "target")
    if _cuda(draft, "draft") != dev:
        raise ValueError("target and draft must be on one device")
    if draft.dtype != target.dtype or draft.shape[1] < N1:
        raise TypeError("draft must share the target's dtype and hold N+1 rows per sequence")
    t_pitch, _ = _rows(target, "target")
    d_pitch, _ = _rows(draft, "draft")
    if N > 0:
        _arr(parents, "parents", torch.int32, B * N, dev)
        _arr(tokens, "tokens", torch.int32, B * N, dev)
    _arr(uniforms, "uniforms", torch.float64, B * (N + 1), dev)
    _arr(temperature, "temperature", torch.float32, B, dev)
    accept_len = _out(accept_len, "accept_len", torch.int32, (B,), dev)
    out_tokens = _out(out_tokens, "out_tokens", torch.int32, (B, N + 1), dev)
    if path is True:
        path = torch.empty((B, max(N, 1)), dtype=torch.int32, device=dev)
    elif path is False:
        path = None
    _opt(path, "path", torch.int32, B * N, dev)
    stats = _stats(stats, dev)
    ws = (workspace or _default_ws).get(lib.sv_tree_verify_workspace_size(B, N, V), dev)
    code = _on(dev, lib.sv_tree_verify, _ptr(target), t_pitch, _ptr(draft), d_pitch, _dtype_code(target),
                              _ptr(parents if N > 0 else None), _ptr(tokens if N > 0 else None), _ptr(uniforms), B, N,
                              V, _ptr(temperature), _ptr(accept_len), _ptr(out_tokens), _ptr(path), _ptr(stats),
                              _ptr(ws), ws.numel(), _stream(stream, dev))
    _abi.check("sv_tree_verify", code)
    return accept_len, out_tokens, (path[:, :N] if path is not None else None), stats


def sv_tree_reuse(parents, tokens, accept_len, out_tokens, reuse_node=None, stream=None):
    """sv_tree_reuse: per sequence the node where the committed prefix ends as a path of the
    drafted tree (parents / tokens int32 [B, N]), or -1."""
    lib = load()
    B, N = parents.shape
    K = out_tokens.shape[1] - 1
    dev = _cuda(parents, "parents")
    _arr(parents, "parents", torch.int32, B * N, dev)
    _arr(tokens, "tokens", torch.int32, B * N, dev)
    _arr(accept_len, "accept_len", torch.int32, B, dev)
    _arr(out_tokens, "out_tokens", torch.int32, B * (K + 1), dev)
    reuse_node = _out(reuse_node, "reuse_node", torch.int32, (B,), dev)
    code = _on(dev, lib.sv_tree_reuse, _ptr(parents), _ptr(tokens), N, _ptr(accept_len), _ptr(out_tokens), K, B,
                             _ptr(reuse_node), _stream(stream, dev))
    _abi.check("sv_tree_reuse", code)
    return reuse_node


def sv_saguaro_sample(draft, uniforms, temperature, top_p=None, F=0, C=1.0, n_rows=None, tokens=None, debug=False,
                      stats=None, workspace=None, stream=None, top_k=None):
    """sv_saguaro_sample: one token per row j < n_rows of each sequence of draft [B, R, V].
    uniforms float64 [B, n_rows]; temperature float32 [B]; top_p float32 [B] or None; top_k
    int32 [B] or None; returns (tokens int32 [B, n_rows],
    debug float64 [B, n_rows, 4] or None, stats)."""
    lib = load()
    B, R, V = draft.shape
    n_rows = R if n_rows is None else n_rows
    dev = _cuda(draft, "draft")
    pitch, rows = _rows(draft, "draft")
    _arr(uniforms, "uniforms", torch.float64, B * n_rows, dev)
    _arr(temperature, "temperature", torch.float32, B, dev)
    _opt(top_p, "top_p", torch.float32, B, dev)
    _opt(top_k, "top_k", torch.int32, B, dev)
    tokens = _out(tokens, "tokens", torch.int32, (B, n_rows), dev)
    dbg = torch.empty((B, n_rows, 4), dtype=torch.float64, device=dev) if debug else None
    stats = _stats(stats, dev)
    ws_bytes = lib.sv_saguaro_sample_workspace_size(B, n_rows, V)
    ws = (workspace or _default_ws).get(ws_bytes, dev)
    code = _on(dev, lib.sv_saguaro_sample, _ptr(draft), pitch, rows, _dtype_code(draft), B, n_rows, V, _ptr(temperature),
                                 _ptr(top_p), _ptr(top_k), int(F), float(C), _ptr(uniforms), _ptr(tokens),
                                 _ptr(dbg), _ptr(stats),
                                 _ptr(ws), ws.numel(), _stream(stream, dev))
    _abi.check("sv_saguaro_sample", code)
    return tokens, dbg, stats


def sv_fanout(budget: float, a: float, r: float, K: int):
    """Host-only Theorem 12 fan-out: returns (F_real list[float], F_int list[int])."""
    lib = load()
    fr = (ctypes.c_double * (K + 1))()
    fi = (ctypes.c_int32 * (K + 1))()
    code = lib.sv_fanout(float(budget), float(a), float(r), int(K), ctypes.cast(fr, ctypes.c_void_p),
                         ctypes.cast(fi, ctypes.c_void_p))
    _abi.check("sv_fanout", code)
    return list(fr), list(fi)


def _host_i32(values):
    arr = (ctypes.c_int32 * len(values))(*[int(v) for v in values])
    return arr, ctypes.cast(arr, ctypes.c_void_p)


def sv_cache_keys(draft, draft_tokens, F_int, keys=None, stats=None, workspace=None, stream=None):
    """sv_cache_keys: draft [B, R>=K+1, V]; draft_tokens int32 [B, K]; F_int host list of K+1 ints.
    Returns keys int32 [B, sum F_int]."""
    lib = load()
    B, R, V = draft.shape
    K = len(F_int) - 1
    dev = _cuda(draft, "draft")
    pitch, rows = _rows(draft, "draft")
    if K > 0:
        _arr(draft_tokens, "draft_tokens", torch.int32, B * K, dev)
    keys = _out(keys, "keys", torch.int32, (B, int(sum(F_int))), dev)
    stats = _stats(stats, dev)
    f_arr, f_ptr = _host_i32(F_int)
    ws_bytes = lib.sv_cache_keys_workspace_size(B, K, V)
    ws = (workspace or _default_ws).get(ws_bytes, dev)
    code = _on(dev, lib.sv_cache_keys, _ptr(draft), pitch, rows, _dtype_code(draft), _ptr(draft_tokens), f_ptr, B, K, V,
                             _ptr(keys), _ptr(stats), _ptr(ws), ws.numel(), _stream(stream, dev))
    _abi.check("sv_cache_keys", code)
    return keys, stats


def sv_cache_lookup(accept_len, out_tokens, keys, F_int, hit=None, stream=None):
    lib = load()
    B = accept_len.shape[0]
    K = len(F_int) - 1
    dev = _cuda(accept_len, "accept_len")
    _arr(accept_len, "accept_len", torch.int32, B, dev)
    _arr(out_tokens, "out_tokens", torch.int32, B * (K + 1), dev)
    _arr(keys, "keys", torch.int32, B * int(sum(F_int)), dev)
    hit = _out(hit, "hit", torch.uint8, (B,), dev)
    f_arr, f_ptr = _host_i32(F_int)
    code = _on(dev, lib.sv_cache_lookup, _ptr(accept_len), _ptr(out_tokens), _ptr(keys), f_ptr, B, K, _ptr(hit),
                               _stream(stream, dev))
    _abi.check("sv_cache_lookup", code)
    return hit


def sv_topk_rows(logits, kappa, temperature=None, ids=None, logprobs=None, stats=None, workspace=None, stream=None):
    """sv_topk_rows: logits [N, V]; returns (ids int32 [N, kappa], logprobs float64 [N, kappa], stats)."""
    lib = load()
    N, V = logits.shape
    dev = _cuda(logits, "logits")
    pitch, _ = _rows(logits, "logits")
    _opt(temperature, "temperature", torch.float32, N, dev)
    ids = _out(ids, "ids", torch.int32, (N, kappa), dev)
    logprobs = _out(logprobs, "logprobs", torch.float64, (N, kappa), dev)
    stats = _stats(stats, dev)
    ws_bytes = lib.sv_topk_rows_workspace_size(N, V)
    ws = (workspace or _default_ws).get(ws_bytes, dev)
    code = _on(dev, lib.sv_topk_rows, _ptr(logits), pitch, _dtype_code(logits), N, V, int(kappa), _ptr(temperature), _ptr(ids),
                            _ptr(logprobs), _ptr(stats), _ptr(ws), ws.numel(), _stream(stream, dev))
    _abi.check("sv_topk_rows", code)
    return ids, logprobs, stats


def sv_mirror_reuse(branches, accept_len, out_tokens, reuse=None, stream=None):
    lib = load()
    B, kappa, gamma = branches.shape
    dev = _cuda(branches, "branches")
    _arr(branches, "branches", torch.int32, B * kappa * gamma, dev)
    _arr(accept_len, "accept_len", torch.int32, B, dev)
    _arr(out_tokens, "out_tokens", torch.int32, B * (gamma + 1), dev)
    reuse = _out(reuse, "reuse", torch.uint8, (B,), dev)
    code = _on(dev, lib.sv_mirror_reuse, _ptr(branches), _ptr(accept_len), _ptr(out_tokens), B, kappa, gamma, _ptr(reuse),
                               _stream(stream, dev))
    _abi.check("sv_mirror_reuse", code)
    return reuse


def sv_selftest_timeout(limit_cycles: int, stats=None, stream=None):
    lib = load()
    dev = torch.device("cuda", torch.cuda.current_device())
    if stats is None:
        stats = new_stats(dev)
    _abi.check("sv_selftest_timeout", lib.sv_selftest_timeout(int(limit_cycles), _ptr(stats), _stream(stream, dev)))
    return stats


def sv_selftest_exp2(lo: float, hi: float, n: int, stream=None):
    lib = load()
    dev = torch.device("cuda", torch.cuda.current_device())
    out = torch.zeros(2, dtype=torch.float64, device=dev)
    _abi.check("sv_selftest_exp2", lib.sv_selftest_exp2(float(lo), float(hi), int(n), _ptr(out), _stream(stream, dev)))
    return out


def sv_selftest_exp2_all(lo: float, hi: float, stream=None):
    """Largest relative errors (fast, float-float) of the library's exponentials over every
    float32 input in [lo, hi], and the number of inputs evaluated."""
    lib = load()
    dev = torch.device("cuda", torch.cuda.current_device())
    out = torch.zeros(3, dtype=torch.float64, device=dev)
    _abi.check("sv_selftest_exp2_all", lib.sv_selftest_exp2_all(float(lo), float(hi), _ptr(out), _stream(stream, dev)))
    torch.cuda.synchronize()
    r = out.cpu().tolist()
    return r[0], r[1], int(r[2])
