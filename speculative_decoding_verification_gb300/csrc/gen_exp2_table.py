#!/usr/bin/env python
"""Writes sv_exp2_table.h: 2^(j/256), j = 0..255, as float-float pairs (hi, lo).

hi is the float32 nearest to 2^(j/256) and lo the float32 nearest to the remainder, both from
a 60-digit decimal evaluation, so hi + lo carries about 48 significant bits.  The header is
committed; run this script only to regenerate it.
"""
import decimal
import os
import struct

decimal.getcontext().prec = 60


def f32(x: float) -> float:
    return struct.unpack("<f", struct.pack("<f", x))[0]


def main():
    ln2 = decimal.Decimal(2).ln()
    rows = []
    for j in range(256):
        t = (ln2 * decimal.Decimal(j) / decimal.Decimal(256)).exp()
        hi = f32(float(t))
        lo = f32(float(t - decimal.Decimal(hi)))
        rows.append(f"    {{{hi.hex()}f, {lo.hex()}f}},   // 2^({j}/256)")
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "sv_exp2_table.h")
    with open(out, "w") as f:
        f.write("// sv_exp2_table.h — 2^(j/256) for j = 0..255 as float-float pairs {hi, lo}, written by\n"
                "// gen_exp2_table.py (60-digit decimal evaluation, each part rounded to nearest float32).\n"
                "// Used by the float-float exponential (Tang's table method); kernels copy it to shared memory.\n"
                "#pragma once\n\n#include <cuda_runtime.h>\n\nnamespace sv {\n\n"
                "static __device__ const float2 kExp2Table[256] = {\n")
        f.write("\n".join(rows))
        f.write("\n};\n\n}  // namespace sv\n")


if __name__ == "__main__":
    main()
