"""Philox4x32-10 counter-based random numbers, written from the published definition.

Reference: J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel random numbers:
as easy as 1, 2, 3", SC'11.  A Philox4x32 round multiplies counter words 0 and 2 by two
fixed 32-bit constants, splits each 64-bit product into its high and low halves, and forms
the new counter as (hi(c2*M1) ^ c1 ^ k0, lo(c2*M1), hi(c0*M0) ^ c3 ^ k1, lo(c0*M0)).
Between rounds each key word is advanced by a Weyl constant.  Ten rounds make Philox4x32-10.

This module draws the uniforms that the verification method consumes (accept tests,
residual draws, draft sampling, branch construction).  It holds none of the method's
arithmetic: it only turns (seed, stream, round, row, slot) into doubles in [0, 1).
"""
from __future__ import annotations

import numpy as np

PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85
_MASK32 = np.uint64(0xFFFFFFFF)

# Stream ids: one key word per purpose so that no two purposes share a counter.
STREAM_DRAFT = 0      # draft-token sampling, one uniform per (sequence, draft position)
STREAM_ACCEPT = 1     # accept tests, one per (sequence, draft position)
STREAM_RESIDUAL = 2   # residual / bonus draw, one per sequence
STREAM_BRANCH = 3     # Mirror-style branch construction, one per (sequence, branch, depth)


def philox4x32_10(counter, key):
    """Apply Philox4x32-10.

    counter: uint32-valued array [..., 4]; key: uint32-valued array [..., 2] (broadcastable).
    Returns uint32 array [..., 4].
    """
    ctr = np.asarray(counter, dtype=np.uint64) & _MASK32
    k = np.asarray(key, dtype=np.uint64) & _MASK32
    c0, c1, c2, c3 = ctr[..., 0], ctr[..., 1], ctr[..., 2], ctr[..., 3]
    k0 = np.broadcast_to(k[..., 0], c0.shape).copy()
    k1 = np.broadcast_to(k[..., 1], c0.shape).copy()
    m0 = np.uint64(PHILOX_M0)
    m1 = np.uint64(PHILOX_M1)
    for rnd in range(10):
        if rnd > 0:
            k0 = (k0 + np.uint64(PHILOX_W0)) & _MASK32
            k1 = (k1 + np.uint64(PHILOX_W1)) & _MASK32
        p0 = c0 * m0  # < 2^64: both factors < 2^32
        p1 = c2 * m1
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK32
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return np.stack([c0, c1, c2, c3], axis=-1).astype(np.uint32)


def uniforms(seed: int, stream: int, round_idx: int, rows: int, slots: int) -> np.ndarray:
    """Doubles in [0, 1) of shape [rows, slots].

    Key = (seed, stream); counter = (slot, row, round, 0).  The first two output words
    form a 64-bit integer (word 1 high, word 0 low) whose top 53 bits, scaled by 2^-53,
    give the uniform.
    """
    slot = np.arange(slots, dtype=np.uint64)[None, :]
    row = np.arange(rows, dtype=np.uint64)[:, None]
    ctr = np.zeros((rows, slots, 4), dtype=np.uint64)
    ctr[..., 0] = slot
    ctr[..., 1] = row
    ctr[..., 2] = np.uint64(round_idx) & _MASK32
    key = np.array([seed & 0xFFFFFFFF, stream & 0xFFFFFFFF], dtype=np.uint64)
    out = philox4x32_10(ctr, key).astype(np.uint64)
    bits = ((out[..., 1] << np.uint64(32)) | out[..., 0]) >> np.uint64(11)
    return bits.astype(np.float64) * (2.0 ** -53)


def seed_words(seed: int, stream: int, round_idx: int, tag: int) -> int:
    """A 63-bit integer seed for bulk (logit) generators, derived through Philox."""
    ctr = np.array([[tag & 0xFFFFFFFF, 0, round_idx & 0xFFFFFFFF, 0x5EED]], dtype=np.uint64)
    key = np.array([seed & 0xFFFFFFFF, stream & 0xFFFFFFFF], dtype=np.uint64)
    w = philox4x32_10(ctr, key)[0].astype(np.uint64)
    return int(((w[1] << np.uint64(32)) | w[0]) & np.uint64(0x7FFFFFFFFFFFFFFF))
