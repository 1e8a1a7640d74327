#!/usr/bin/env python
"""Writes sv_js_table.h: the per-token Jensen-Shannon term as a function of the log-ratio.

For one token with weights q and p, M = max(q, p) and l = |log2(q/p)|, the term of the divergence
(in bits) is (q log2(2q/(q+p)) + p log2(2p/(q+p))) / 2 = M g(l) with, for z = 2^-l,

    g(l) = ( (1 + z)(1 - log2(1 + z)) - l z ) / 2,     g(0) = 0,  g(l) -> 1/2,
    g'(l) = z ln2 (l + log2(1 + z) - 1) / 2.

The table holds, on l in [0, L] with step 1/N, one float4 per interval: the cubic Hermite
interpolant of g through the interval's ends in Horner form, g(l_i + t/N) = g_i + t (d_i + t (a_i +
t b_i)) for t in [0, 1), with d_i = g'(l_i)/N, a_i = 3(g_i+1 - g_i) - 2 d_i - d_i+1, b_i = 2(g_i -
g_i+1) + d_i + d_i+1; beyond L the term is M / 2 (g differs from 1/2 by less than l 2^-l / 2).
Values come from a 50-digit evaluation, rounded to nearest float32.  The script also measures
the worst absolute error of the float32 table's interpolation (on 64 points per interval, in
float64) and of g past L, and writes their sum, rounded up, as kJsTableErr, and the largest
slope of g as kJsSlopeMax.  The header is committed; run this script only to regenerate it.
"""
import os
import struct

import mpmath

mpmath.mp.dps = 50
N = 32          # intervals per unit of l
L = 48          # table range
NT = N * L      # intervals


def f32(x: float) -> float:
    return struct.unpack("<f", struct.pack("<f", x))[0]


def g_exact(l):
    l = mpmath.mpf(l)
    z = mpmath.power(2, -l)
    return ((1 + z) * (1 - mpmath.log(1 + z, 2)) - l * z) / 2


def dg_exact(l):
    l = mpmath.mpf(l)
    z = mpmath.power(2, -l)
    return z * mpmath.log(2) * (l + mpmath.log(1 + z, 2) - 1) / 2


def horner(e, t):
    g0, d0, a, b = e
    return g0 + t * (d0 + t * (a + t * b))


def main():
    gv = [g_exact(mpmath.mpf(i) / N) for i in range(NT + 1)]
    dv = [dg_exact(mpmath.mpf(i) / N) / N for i in range(NT + 1)]
    entries = []
    for i in range(NT):
        a = 3 * (gv[i + 1] - gv[i]) - 2 * dv[i] - dv[i + 1]
        b = 2 * (gv[i] - gv[i + 1]) + dv[i] + dv[i + 1]
        entries.append(tuple(f32(float(v)) for v in (gv[i], dv[i], a, b)))
    worst = 0.0
    for i in range(NT):
        for k in range(65):
            t = k / 64.0
            l = (i + t) / N
            err = abs(horner(entries[i], t) - float(g_exact(l)))
            worst = max(worst, err)
    slope = max(float(dg_exact(mpmath.mpf(k) / 256)) for k in range(256 * 8))   # g' peaks near l = 1.5
    tail = float(L * mpmath.power(2, -L) / 2)   # |g - 1/2| past L is below l 2^-l / 2, largest at L
    bound = float(mpmath.mpf(worst + tail) * mpmath.mpf("1.25"))
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "sv_js_table.h")
    with open(out, "w") as f:
        f.write("// sv_js_table.h — the per-token Jensen-Shannon term M g(l) (M = max(q, p), l = |log2(q/p)|)\n"
                "// as a cubic Hermite table of g on [0, %d] with step 1/%d, written by gen_js_table.py\n"
                "// (50-digit evaluation, rounded to nearest float32); kernels copy it to shared memory.\n"
                "#pragma once\n\n#include <cuda_runtime.h>\n\nnamespace sv {\n\n" % (L, N))
        f.write("constexpr int kJsTableN = %d;      // intervals per unit of l\n" % N)
        f.write("constexpr int kJsTableL = %d;      // past this l the term is M / 2\n" % L)
        f.write("constexpr int kJsTableSize = %d;  // intervals\n" % NT)
        f.write("// Worst absolute error of g from the float32 table (interpolation, in float64) and from\n"
                "// g = 1/2 past kJsTableL, times 1.25: %.3e measured.\n" % (worst + tail))
        f.write("constexpr double kJsTableErr = %.3e;\n" % bound)
        f.write("// Largest slope of g (the term moves by at most this times M per unit error in l), x 1.01.\n")
        f.write("constexpr double kJsSlopeMax = %.4f;\n\n" % (slope * 1.01))
        f.write("static __device__ const float4 kJsTable[%d] = {\n" % NT)
        for i, e in enumerate(entries):
            f.write("    {%s, %s, %s, %s},\n" % tuple(f"{v.hex()}f" if v != 0.0 else "0x0p+0f" for v in e))
        f.write("};\n\n}  // namespace sv\n")
    print("worst", worst, "tail", tail, "bound", bound, "slope", slope)


if __name__ == "__main__":
    main()
