"""CPU checks that the product and the oracle stay apart: the binding and the CUDA sources never
reach the oracle, the oracle never reaches the product, and the binding raises instead of
falling back when the shared library is missing."""
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "speculative_decoding_verification_gb300")


def _sources(top, exts):
    for d, _, files in os.walk(top):
        if "__pycache__" in d or "_build" in d:
            continue
        for f in files:
            if f.endswith(exts):
                yield os.path.join(d, f)


def test_product_sources_never_import_the_oracle():
    pat = re.compile(r"^\s*(import\s+oracle|from\s+oracle\b)|#include\s+[<\"][^>\"]*oracle", re.M)
    for p in _sources(PKG, (".py", ".cu", ".cuh", ".h", ".cpp")):
        assert not pat.search(open(p).read()), p


def test_oracle_never_imports_or_reads_the_product():
    pat = re.compile(r"^\s*(import|from)\s+speculative_decoding_verification_gb300\b|#include\s+[<\"][^>\"]*"
                     r"(csrc|specverify|sv_)|open\([^)]*csrc", re.M)
    for p in _sources(os.path.join(ROOT, "oracle"), (".py", ".c", ".h")):
        assert not pat.search(open(p).read()), p


def test_importing_the_product_loads_no_oracle():
    code = ("import sys; import speculative_decoding_verification_gb300 as sv; "
            "print(any(m == 'oracle' or m.startswith('oracle.') for m in sys.modules))")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip() == "False"


def test_missing_library_raises():
    from speculative_decoding_verification_gb300 import _abi
    saved = _abi._lib
    _abi._lib = None
    try:
        with pytest.raises(ImportError, match="not built"):
            _abi.load(os.path.join(ROOT, "_no_such_dir", "libspecverify.so"))
    finally:
        _abi._lib = saved
