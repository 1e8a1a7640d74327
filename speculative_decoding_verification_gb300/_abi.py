"""ctypes declarations of the libspecverify C ABI (include/specverify.h).

Loading fails loudly when the shared library is missing: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspecverify.so")

c_int, c_i32p, c_i64, c_f32, c_f64 = ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_double
c_vp, c_size = ctypes.c_void_p, ctypes.c_size_t

SV_OK, SV_ERR_INVALID_ARG, SV_ERR_CUDA, SV_ERR_NONFINITE, SV_ERR_TIMEOUT, SV_ERR_WORKSPACE, SV_ERR_BAD_TOKEN = range(7)
SV_F32, SV_BF16 = 0, 1
SV_DEBUG_FIELDS = 8
SV_MAX_K = 32
SV_STATIC_SCRATCH_BYTES = 32 << 20
SV_ACCEPT_DIVERGENCE, SV_ACCEPT_ASSISTED = 0, 1   # sv_accept_mode   # scratch array behind sv_verify_static
DBG = dict(lse_q=0, lse_p=1, q_s=2, p_s=3, ratio=4, mass_q=5, mass_p=6, R=7)


class SvStats(ctypes.Structure):
    _fields_ = [("status", ctypes.c_int32), ("error_index", ctypes.c_int32), ("rows", ctypes.c_int64),
                ("accept_tests", ctypes.c_int64), ("draws", ctypes.c_int64), ("reresolved", ctypes.c_int64),
                ("near_boundary", ctypes.c_int64), ("unresolved", ctypes.c_int64)]


STATS_FIELDS = [f for f, _ in SvStats._fields_]
STATS_BYTES = ctypes.sizeof(SvStats)

# name -> (restype, argtypes); the order follows the header.
SIGNATURES = {
    "sv_status_string": (ctypes.c_char_p, [c_int]),
    "sv_version": (c_int, []),
    "sv_verify_workspace_size": (c_size, [c_int, c_int, c_int]),
    "sv_verify": (c_int, [c_vp, c_i64, c_vp, c_i64, c_int, c_int, c_vp, c_vp, c_int, c_int, c_int, c_vp, c_vp,
                          c_vp, c_int, c_f32, c_vp, c_vp, c_vp, c_vp, c_vp, c_size, c_vp]),
    "sv_verify_host_workspace_size": (c_size, [c_int, c_int, c_int, c_int]),
    "sv_verify_host": (c_int, [c_vp, c_i64, c_vp, c_i64, c_int, c_int, c_vp, c_vp, c_int, c_int, c_int, c_vp, c_vp,
                               c_vp, c_int, c_f32, c_vp, c_vp, c_vp, c_vp, c_size, c_vp, c_vp]),
    "sv_verify_lazy": (c_int, [c_vp, c_i64, c_vp, c_i64, c_int, c_int, c_vp, c_vp, c_int, c_int, c_int, c_vp, c_vp,
                               c_vp, c_int, c_f32, c_vp, c_vp, c_vp, c_vp, c_vp, c_size, c_vp]),
    "sv_verify_static": (c_int, [c_vp, c_i64, c_vp, c_i64, c_int, c_int, c_vp, c_vp, c_int, c_int, c_int, c_vp,
                                 c_vp, c_vp, c_int, c_f32, c_vp, c_vp, c_vp, c_vp, c_vp]),
    "sv_tree_verify_workspace_size": (c_size, [c_int, c_int, c_int]),
    "sv_tree_verify": (c_int, [c_vp, c_i64, c_vp, c_i64, c_int, c_vp, c_vp, c_vp, c_int, c_int, c_int, c_vp, c_vp, c_vp,
                               c_vp, c_vp, c_vp, c_size, c_vp]),
    "sv_tree_reuse": (c_int, [c_vp, c_vp, c_int, c_vp, c_vp, c_int, c_int, c_vp, c_vp]),
    "sv_fuzzy_verify_workspace_size": (c_size, [c_int, c_int, c_int]),
    "sv_fuzzy_verify": (c_int, [c_vp, c_i64, c_vp, c_i64, c_int, c_int, c_vp, c_vp, c_int, c_int, c_int, c_vp, c_f32,
                                c_int, c_vp, c_vp, c_vp, c_vp, c_vp, c_size, c_vp]),
    "sv_saguaro_sample_workspace_size": (c_size, [c_int, c_int, c_int]),
    "sv_saguaro_sample": (c_int, [c_vp, c_i64, c_int, c_int, c_int, c_int, c_int, c_vp, c_vp, c_vp, c_int, c_f32,
                                  c_vp, c_vp, c_vp, c_vp, c_vp, c_size, c_vp]),
    "sv_fanout": (c_int, [c_f64, c_f64, c_f64, c_int, c_vp, c_vp]),
    "sv_cache_keys_workspace_size": (c_size, [c_int, c_int, c_int]),
    "sv_cache_keys": (c_int, [c_vp, c_i64, c_int, c_int, c_vp, c_vp, c_int, c_int, c_int, c_vp, c_vp, c_vp, c_size,
                              c_vp]),
    "sv_cache_lookup": (c_int, [c_vp, c_vp, c_vp, c_vp, c_int, c_int, c_vp, c_vp]),
    "sv_topk_rows_workspace_size": (c_size, [c_int, c_int]),
    "sv_topk_rows": (c_int, [c_vp, c_i64, c_int, c_int, c_int, c_int, c_vp, c_vp, c_vp, c_vp, c_vp, c_size, c_vp]),
    "sv_mirror_reuse": (c_int, [c_vp, c_vp, c_vp, c_int, c_int, c_int, c_vp, c_vp]),
    "sv_set_profile_events": (None, [c_vp, c_vp]),
    "sv_selftest_timeout": (c_int, [c_i64, c_vp, c_vp]),
    "sv_selftest_exp2": (c_int, [c_f64, c_f64, c_i64, c_vp, c_vp]),
    "sv_selftest_exp2_all": (c_int, [c_f32, c_f32, c_vp, c_vp]),
}

_lib = None


def load(path: str = LIB_PATH):
    """Load libspecverify and declare every entry point; raise if it is not built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libspecverify is not built ({path} missing); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load().sv_status_string(code).decode()


class SvError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {status_string(code)} ({code})")
        self.code = code


def check(fn: str, code: int):
    if code != SV_OK:
        raise SvError(fn, code)
