"""The float-float tier's bf16 weight tables rest on an exact split of every bf16 logit.

A bf16 value x = s 2^(E-127) (1 + m/128) with m = 8 m_h + m_l (m_h the top three, m_l the low
four mantissa bits) equals v1 + v2 with v1 = s 2^(E-127) (1 + m_h/8) and v2 = s 2^(E-127)
m_l/128, both exact float32 values; so 2^(x c - r) = 2^(v1 c - r) 2^(v2 c) for any c and r.
Checked here for every bit pattern of the tables' exponent range (read from the kernel source),
together with the index layout: (sign, exponent) groups of 8 first-factor and 16
second-factor entries, each pattern reaching exactly one pair of entries.
"""
import re
from pathlib import Path

import numpy as np

SRC = Path(__file__).resolve().parents[1] / "speculative_decoding_verification_gb300" / "csrc" / "sv_exact.cuh"


def _const(name):
    return int(re.search(rf"constexpr int {name} = (\d+);", SRC.read_text()).group(1))


def test_bf16_split_is_exact_and_indices_cover_each_pattern_once():
    e0, ne = _const("kTabE0"), _const("kTabNE")
    b = np.arange(1 << 16, dtype=np.uint32)
    xf = (b << 16).view(np.float32)
    x = np.where(np.isfinite(xf), xf, 0.0).astype(np.float64)   # inf / NaN patterns lie outside the tables
    s = np.where(b >> 15, -1.0, 1.0)
    E = ((b >> 7) & 0xFF).astype(np.int64)
    mh, ml = ((b >> 4) & 7).astype(np.int64), (b & 15).astype(np.int64)
    inr = (E >= e0) & (E < e0 + ne)
    assert inr.sum() == 2 * ne * 128
    scale = s * np.ldexp(1.0, E - 127)
    v1 = scale * (1.0 + mh / 8.0)
    v2 = scale * (ml / 128.0)
    # exact in float64, and both parts exact float32 values
    np.testing.assert_array_equal((v1 + v2)[inr], x[inr])
    np.testing.assert_array_equal(v1[inr].astype(np.float32).astype(np.float64), v1[inr])
    np.testing.assert_array_equal(v2[inr].astype(np.float32).astype(np.float64), v2[inr])
    # first-factor argument: |v1| in [2^-9, 2^7) for the range the tables hold
    assert np.abs(v1[inr]).min() == 2.0 ** (e0 - 127) and np.abs(v1[inr]).max() < 2.0 ** (e0 + ne - 127)
    # index layout of the kernel: group g = (E - e0) + sign * ne; t1[g*8 + m_h], t2[g*16 + m_l]
    g = (E - e0) + (b >> 15).astype(np.int64) * ne
    i1, i2 = g * 8 + mh, g * 16 + ml
    assert i1[inr].min() == 0 and i1[inr].max() == 2 * ne * 8 - 1
    assert i2[inr].min() == 0 and i2[inr].max() == 2 * ne * 16 - 1
    pair = i1[inr] * (2 * ne * 16) + i2[inr]
    assert len(np.unique(pair)) == inr.sum()
    # each table entry is the factor of its own argument: v1 depends on (g, m_h) only, v2 on (g, m_l) only
    for idx, v in ((i1, v1), (i2, v2)):
        order = np.argsort(idx[inr], kind="stable")
        ii, vv = idx[inr][order], v[inr][order]
        first = np.r_[True, ii[1:] != ii[:-1]]
        np.testing.assert_array_equal(vv, np.repeat(vv[first], np.diff(np.r_[np.nonzero(first)[0], len(ii)])))
    # the product of the two factors is the weight, for a spread of c and r, wherever the kernel
    # takes both factors from the tables (first exponent in [-100, 64], second within 32)
    for c, r in ((1.4426950408889634, 9), (0.48089834696298783, 3), (9.617966939259756, 40)):
        y1, y2 = v1[inr] * c - r, v2[inr] * c
        use = (y1 >= -100) & (y1 <= 64) & (np.abs(y2) <= 32)
        assert use.sum() > 1000
        w = np.exp2(x[inr][use] * c - r)
        f = np.exp2(y1[use]) * np.exp2(y2[use])
        np.testing.assert_allclose(f, w, rtol=1e-12, atol=0)
