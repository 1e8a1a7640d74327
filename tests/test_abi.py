"""CPU checks of the C ABI: the library builds, loads and exports every declared entry point;
host-only calls work; argument errors are returned before any device work."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verification_gb300 import build
    build.build()
    import speculative_decoding_verification_gb300 as sv
    return sv.load()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "specverify.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = set(re.findall(r"\b(sv_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert "sv_verify" in names and "sv_fanout" in names and len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n


def test_binding_declares_every_symbol():
    from speculative_decoding_verification_gb300 import _abi
    assert sorted(_abi.SIGNATURES) == declared_symbols()


def test_status_strings(lib):
    import speculative_decoding_verification_gb300 as sv
    assert sv.status_string(0) == "ok"
    assert "timed out" in sv.status_string(4)


@pytest.mark.parametrize("budget,a,r,K", [(64, 0.7, 1.0, 5), (23, 0.8, 1.0, 5), (100, 0.5, 2.0, 3), (7.5, 0.3, 0.0, 0),
                                          (1000, 0.95, 0.25, 12), (3, 0.5, 0.0, 1), (6, 0.5, 0.0, 2)])
def test_fanout_matches_oracle(lib, budget, a, r, K):
    import speculative_decoding_verification_gb300 as sv
    fr, fi = sv.sv_fanout(budget, a, r, K)
    ofr, ofi = oracle.fanout(budget, a, r, K)
    np.testing.assert_allclose(fr, ofr, rtol=1e-13)
    assert list(fi) == list(ofi)


def test_fanout_rejects_bad_arguments(lib):
    fr = (ctypes.c_double * 8)()
    fi = (ctypes.c_int32 * 8)()
    p1, p2 = ctypes.cast(fr, ctypes.c_void_p), ctypes.cast(fi, ctypes.c_void_p)
    assert lib.sv_fanout(64.0, 1.0, 1.0, 5, p1, p2) == 1
    assert lib.sv_fanout(64.0, 0.5, -1.0, 5, p1, p2) == 1
    assert lib.sv_fanout(-1.0, 0.5, 1.0, 5, p1, p2) == 1
    assert lib.sv_fanout(64.0, 0.5, 1.0, 99, p1, p2) == 1
    assert lib.sv_fanout(64.0, 0.5, 1.0, 5, None, p2) == 1


def test_verify_rejects_bad_arguments_before_launch(lib):
    """Argument errors come back synchronously; no device is touched (none exists here)."""
    fake = 1 << 20   # a 16-byte aligned non-null address, never dereferenced
    ws = lib.sv_verify_workspace_size(4, 3, 1000)
    assert ws > 0 and lib.sv_verify_workspace_size(0, 3, 1000) == 0

    def call(**kw):
        args = dict(t=fake, tp=1024, d=fake, dp=1024, dr=3, dtype=1, tok=fake, u=fake, B=4, K=3, V=1000, T=fake,
                    top_p=None, F=0, C=1.0, al=fake, ot=fake, dbg=None, st=None, ws=fake, wsb=ws)
        kw = {**args, **kw}
        return lib.sv_verify(kw["t"], kw["tp"], kw["d"], kw["dp"], kw["dr"], kw["dtype"], kw["tok"], kw["u"], kw["B"],
                             kw["K"], kw["V"], kw["T"], kw["top_p"], None, kw["F"], kw["C"], kw["al"], kw["ot"], kw["dbg"],
                             kw["st"], kw["ws"], kw["wsb"], None)
    assert call(B=0) == 1
    assert call(K=33) == 1
    assert call(V=0) == 1
    assert call(tp=999) == 1                     # pitch < V
    assert call(tp=1001) == 1                    # row start not 16-byte aligned for bf16
    assert call(t=fake + 2) == 1                 # misaligned base
    assert call(t=None) == 1
    assert call(tok=None) == 1
    assert call(dr=2) == 1                       # fewer draft rows than K
    assert call(dtype=7) == 1
    assert call(C=1.5) == 1
    assert call(F=-1) == 1
    assert call(ws=None) == 5
    assert call(wsb=255) == 5
    assert call(ws=fake + 8) == 5                # workspace not 256-byte aligned


def test_verify_host_rejects_bad_arguments_before_any_copy(lib):
    """sv_verify_host: argument and workspace errors come back before any copy is enqueued."""
    fake = 1 << 20
    ws = lib.sv_verify_host_workspace_size(4, 3, 1000, 1)
    assert ws > lib.sv_verify_workspace_size(4, 3, 1000)          # staging on top of the verify workspace
    assert lib.sv_verify_host_workspace_size(0, 3, 1000, 1) == 0
    assert lib.sv_verify_host_workspace_size(4, 3, 1000, 7) == 0

    def call(**kw):
        args = dict(t=fake, tp=1000, d=fake, dp=1000, dr=3, dtype=1, tok=fake, u=fake, B=4, K=3, V=1000, T=fake,
                    al=fake, ot=fake, ws=fake, wsb=ws)
        kw = {**args, **kw}
        return lib.sv_verify_host(kw["t"], kw["tp"], kw["d"], kw["dp"], kw["dr"], kw["dtype"], kw["tok"], kw["u"],
                                  kw["B"], kw["K"], kw["V"], kw["T"], None, None, 0, 1.0, kw["al"], kw["ot"], None,
                                  kw["ws"], kw["wsb"], None, None)
    assert call(B=0) == 1
    assert call(K=33) == 1
    assert call(V=0) == 1
    assert call(dtype=7) == 1
    assert call(t=None) == 1
    assert call(tp=999) == 1                     # pitch < V (host rows need no alignment)
    assert call(tok=None) == 1
    assert call(d=None) == 1
    assert call(dr=2) == 1
    assert call(u=None) == 1
    assert call(T=None) == 1
    assert call(al=None) == 1
    assert call(ot=None) == 1
    assert call(ws=None) == 5
    assert call(wsb=ws - 1) == 5
    assert call(ws=fake + 8) == 5


def test_lookup_and_reuse_reject_bad_arguments(lib):
    f = (ctypes.c_int32 * 3)(1, 2, 3)
    fp = ctypes.cast(f, ctypes.c_void_p)
    fake = 1 << 20
    assert lib.sv_cache_lookup(fake, fake, fake, fp, 0, 2, fake, None) == 1
    assert lib.sv_cache_lookup(fake, fake, fake, None, 4, 2, fake, None) == 1
    assert lib.sv_mirror_reuse(fake, fake, fake, 4, 0, 7, fake, None) == 1
    assert lib.sv_mirror_reuse(None, fake, fake, 4, 8, 7, fake, None) == 1


def test_exp2_table_header_values():
    """The float-float table of 2^(j/256) used by the library's float-float exponential: hi is the
    float32 nearest to 2^(j/256), lo the float32 nearest to the remainder (checked in float64
    and against a 50-digit decimal evaluation for a sample)."""
    import decimal
    import struct
    path = os.path.join(ROOT, "speculative_decoding_verification_gb300", "csrc", "sv_exp2_table.h")
    pairs = re.findall(r"\{(-?0x[0-9a-f.p+-]+)f, (-?0x[0-9a-f.p+-]+)f\}", open(path).read())
    assert len(pairs) == 256
    f32 = lambda x: struct.unpack("<f", struct.pack("<f", x))[0]
    decimal.getcontext().prec = 50
    ln2 = decimal.Decimal(2).ln()
    for j, (h, l) in enumerate(pairs):
        hi, lo = float.fromhex(h), float.fromhex(l)
        assert f32(hi) == hi and f32(lo) == lo
        assert abs((hi + lo) / np.exp2(j / 256.0) - 1.0) < 2.0 ** -47
        if j % 17 == 0:
            t = (ln2 * j / 256).exp()
            assert abs(decimal.Decimal(hi) + decimal.Decimal(lo) - t) / t < decimal.Decimal(2) ** -47
            assert abs(decimal.Decimal(hi) - t) <= decimal.Decimal(2) ** -24 * t


def _js_table():
    path = os.path.join(ROOT, "speculative_decoding_verification_gb300", "csrc", "sv_js_table.h")
    text = open(path).read()
    num = r"(-?0x[0-9a-f.p+-]+)f"
    rows = re.findall(r"\{" + ", ".join([num] * 4) + r"\}", text)
    consts = {k: float(v) for k, v in re.findall(r"constexpr (?:int|double) (kJs\w+) = ([0-9.e+-]+);", text)}
    return np.array([[float.fromhex(x) for x in r] for r in rows]), consts


def test_js_table_header_values():
    """The cubic table of g(l) behind the divergence kernel: its interpolant stays within
    kJsTableErr of g (evaluated here with 50-digit arithmetic at points the generator did not
    sample), kJsSlopeMax bounds g', and M g(l) summed over tokens is the Jensen-Shannon divergence
    of the oracle."""
    import mpmath
    import oracle
    mpmath.mp.dps = 30
    tab, c = _js_table()
    N, L = int(c["kJsTableN"]), int(c["kJsTableL"])
    assert tab.shape == (N * L, 4) and c["kJsTableErr"] < 1e-7

    def g_exact(l):
        z = mpmath.power(2, -mpmath.mpf(l))
        return float(((1 + z) * (1 - mpmath.log(1 + z, 2)) - l * z) / 2)

    def g_tab(l):
        x = l * N
        if x >= N * L:
            return 0.5
        i = int(x)
        t = x - i
        g0, d, a, b = tab[i]
        return g0 + t * (d + t * (a + t * b))

    rng = np.random.default_rng(3)
    ls = np.concatenate([rng.uniform(0, 4, 300), rng.uniform(4, L + 4, 200), [0.0, 1e-3, L - 1e-6, L + 1e-6]])
    for l in ls:
        assert abs(g_tab(l) - g_exact(l)) <= c["kJsTableErr"], l
    for l in rng.uniform(0, 10, 200):
        h = 1e-6
        assert abs(g_exact(l + h) - g_exact(l)) / h <= c["kJsSlopeMax"]
    for _ in range(20):
        q = rng.random(50) ** 4
        p = rng.random(50) ** 4
        q /= q.sum()
        p /= p.sum()
        terms = [max(a, b) * g_exact(abs(np.log2(a / b))) for a, b in zip(q, p)]
        assert sum(terms) == pytest.approx(oracle.jensen_shannon(q, p), rel=1e-12, abs=1e-15)


def test_binding_refuses_bad_tensors_before_any_call(lib):
    """The Python binding checks each array's dtype, device, contiguity and size before the library
    sees its pointer: a float32 uniforms block, for one, would be read past its end as float64."""
    import torch
    import speculative_decoding_verification_gb300 as sv
    B, K, V = 4, 3, 64
    cpu = torch.device("cpu")
    t = torch.zeros((B, K + 1, V))
    tok = torch.zeros((B, K), dtype=torch.int32)
    u = torch.zeros((B, K + 1), dtype=torch.float64)
    T = torch.ones(B)
    # the device entry points take CUDA tensors only: host memory goes through sv_verify_host
    host_calls = [
        lambda: sv.sv_verify(t, t[:, :K], tok, u, T),
        lambda: sv.sv_verify(t, t[:, :K], tok, u, T, lazy=True),
        lambda: sv.sv_verify_static(t, t[:, :K], tok, u, T),
        lambda: sv.sv_fuzzy_verify(t, t[:, :K], tok, u, T),
        lambda: sv.sv_tree_verify(t, t, tok, tok, u, T),
        lambda: sv.sv_tree_reuse(tok, tok, T.int(), tok),
        lambda: sv.sv_saguaro_sample(t, u, T),
        lambda: sv.sv_cache_keys(t, tok, [1, 1, 1, 1]),
        lambda: sv.sv_cache_lookup(T.int(), u.int(), tok, [1, 1, 1, 1]),
        lambda: sv.sv_topk_rows(t[:, 0], 2),
        lambda: sv.sv_mirror_reuse(tok[:, None, :], T.int(), u.int()),
    ]
    for call in host_calls:
        with pytest.raises(TypeError, match="CUDA tensor"):
            call()
    # each refusal of the array check
    sv._arr(u, "uniforms", torch.float64, B * (K + 1), cpu)
    with pytest.raises(TypeError, match="float64"):
        sv._arr(u.float(), "uniforms", torch.float64, B * (K + 1), cpu)
    with pytest.raises(ValueError, match="contiguous"):
        sv._arr(torch.zeros((K + 1, B), dtype=torch.float64).t(), "uniforms", torch.float64, B * (K + 1), cpu)
    with pytest.raises(ValueError, match="elements"):
        sv._arr(u[:2], "uniforms", torch.float64, B * (K + 1), cpu)
    with pytest.raises(ValueError, match="must be on"):
        sv._arr(torch.empty(B * (K + 1), dtype=torch.float64, device="meta"), "uniforms", torch.float64,
                B * (K + 1), cpu)
    with pytest.raises(TypeError, match="torch tensor"):
        sv._arr(np.zeros(B * (K + 1)), "uniforms", torch.float64, B * (K + 1), cpu)
    # the host entry: input sizes and the host buffers its copies write into
    d = t[:, :K].contiguous()
    with pytest.raises(ValueError, match="uniforms"):
        sv.sv_verify_host(t, d, tok, u[:, :K].contiguous(), T, device="cuda:0")
    with pytest.raises(TypeError, match="accept_len"):
        sv.sv_verify_host(t, d, tok, u, T, accept_len=torch.zeros(B, dtype=torch.int64), device="cuda:0")
    with pytest.raises(ValueError, match="out_tokens"):
        sv.sv_verify_host(t, d, tok, u, T, out_tokens=torch.zeros((B, K), dtype=torch.int32), device="cuda:0")


def test_every_entry_point_cites_its_passage():
    """Each declaration in the header follows a comment (the nearest one above it) that cites
    the passage defining the operation (a bracketed page and section) or says that the pages
    have no counterpart."""
    text = open(os.path.join(ROOT, "include", "specverify.h")).read()
    seen = set()
    for m in re.finditer(r"^(?:[A-Za-z_0-9]+\s+)+\**\s*(sv_[a-z0-9_]+)\s*\(", text, re.M):
        name = m.group(1)
        before = text[: m.start()]
        com = before[before.rindex("/*"): before.rindex("*/")]
        seen.add(name)
        assert "[" in com or "no counterpart" in com, name
    assert {"sv_verify", "sv_saguaro_sample", "sv_fanout", "sv_cache_lookup", "sv_tree_verify"} <= seen
    assert seen == set(declared_symbols())


def test_binding_refuses_a_stream_of_another_device():
    """The library plans for the current device and launches on the stream it is given, so the
    binding runs each call with the arrays' device current and refuses a stream that belongs to
    another device before the library is called (a fake stream object stands in: no GPU)."""
    import types

    import torch

    import speculative_decoding_verification_gb300 as sv
    other = types.SimpleNamespace(device=torch.device("cuda", 1), cuda_stream=0)
    with pytest.raises(ValueError, match="stream is on cuda:1"):
        sv._stream(other, torch.device("cuda", 0))
    same = types.SimpleNamespace(device=torch.device("cuda", 0), cuda_stream=1234)
    assert sv._stream(same, torch.device("cuda", 0)).value == 1234
