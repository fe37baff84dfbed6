"""Philox4x32-10 counter-based generator (oracle; test infrastructure only).

Published definition: J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel
Random Numbers: As Easy as 1, 2, 3", SC'11 -- the Philox-4x32 bijection with 10 rounds.
One round maps counter (c0, c1, c2, c3) under key (k0, k1) to

    (hi(M1*c2) ^ c1 ^ k0,  lo(M1*c2),  hi(M0*c0) ^ c3 ^ k1,  lo(M0*c0))

with M0 = 0xD2511F53, M1 = 0xCD9E8D57; between rounds the key is bumped by the Weyl
constants W0 = 0x9E3779B9, W1 = 0xBB67AE85 (mod 2^32).

Use in stochastic rounding (reading; the pages give no generator): element with
row-major linear index i of the quantised tensor draws 16 bits from block
j = rng_offset + i // 8 with counter (lo32(j), hi32(j), 0, 0) and key
(lo32(seed), hi32(seed)); word (i % 8) // 2 of the output, low half for even i and high
half for odd i.
"""
from __future__ import annotations

import numpy as np

M0 = np.uint64(0xD2511F53)
M1 = np.uint64(0xCD9E8D57)
W0 = np.uint64(0x9E3779B9)
W1 = np.uint64(0xBB67AE85)
MASK32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(ctr, key):
    """ctr: uint32-valued array [..., 4]; key: [..., 2].  Returns uint32 [..., 4]."""
    c = [np.asarray(ctr, dtype=np.uint64)[..., i] & MASK32 for i in range(4)]
    k0 = np.asarray(key, dtype=np.uint64)[..., 0] & MASK32
    k1 = np.asarray(key, dtype=np.uint64)[..., 1] & MASK32
    for rnd in range(10):
        if rnd > 0:
            k0 = (k0 + W0) & MASK32
            k1 = (k1 + W1) & MASK32
        p0 = M0 * c[0]                     # < 2^64, exact in uint64
        p1 = M1 * c[2]
        hi0, lo0 = p0 >> np.uint64(32), p0 & MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & MASK32
        c = [hi1 ^ c[1] ^ k0, lo1, hi0 ^ c[3] ^ k1, lo0]
    return np.stack([x.astype(np.uint32) for x in c], axis=-1)


def sr_bits16(linear_index, seed: int, rng_offset: int) -> np.ndarray:
    """The 16 random bits that stochastic rounding uses for each element index."""
    i = np.asarray(linear_index, dtype=np.uint64)
    j = np.uint64(rng_offset) + i // np.uint64(8)
    ctr = np.stack([j & MASK32, j >> np.uint64(32), np.zeros_like(j), np.zeros_like(j)], axis=-1)
    seed = int(seed)
    key = np.broadcast_to(np.array([seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF],
                                   dtype=np.uint64), ctr.shape[:-1] + (2,))
    out = philox4x32_10(ctr, key)
    word = ((i % np.uint64(8)) // np.uint64(2)).astype(np.int64)
    w = np.take_along_axis(out, word[..., None], axis=-1)[..., 0].astype(np.uint32)
    half = (i % np.uint64(2)).astype(np.uint32)
    return ((w >> (half * np.uint32(16))) & np.uint32(0xFFFF)).astype(np.uint32)
