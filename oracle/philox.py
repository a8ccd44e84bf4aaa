"""Philox4x32-10 counter-based generator, written from its published definition
(Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3",
SC'11, section 4.2 and table 2: the Philox-4x32 S-box, multipliers and Weyl
key schedule).

One round maps counter (x0, x1, x2, x3) under round key (k0, k1) to
    (hi(M1*x2) ^ x1 ^ k0,  lo(M1*x2),  hi(M0*x0) ^ x3 ^ k1,  lo(M0*x0));
the key is bumped by the Weyl constants (W0, W1) between rounds; ten rounds.

The step's stream layout (a reading: the pages fix no layout for the random
numbers): key = (seed lo32, seed hi32); counter = (offset lo32, offset hi32,
slot, purpose), purpose 0 = selector walk, 1 = accept test, 2 = residual or
bonus draw; the uniform is u = (x0 >> 8) * 2^-24 in [0, 1).

Test infrastructure only (see oracle/__init__.py).
"""
from __future__ import annotations

M0 = 0xD2511F53
M1 = 0xCD9E8D57
W0 = 0x9E3779B9
W1 = 0xBB67AE85
_MASK = 0xFFFFFFFF

PURPOSE_WALK = 0
PURPOSE_ACCEPT = 1
PURPOSE_RESAMPLE = 2


def _round(x, k):
    p0 = M0 * x[0]
    p1 = M1 * x[2]
    return ((((p1 >> 32) ^ x[1] ^ k[0]) & _MASK), p1 & _MASK,
            (((p0 >> 32) ^ x[3] ^ k[1]) & _MASK), p0 & _MASK)


def philox4x32_10(counter, key):
    """counter: 4 uint32, key: 2 uint32 -> 4 uint32."""
    x = tuple(int(c) & _MASK for c in counter)
    k = (int(key[0]) & _MASK, int(key[1]) & _MASK)
    for _ in range(10):
        x = _round(x, k)
        k = ((k[0] + W0) & _MASK, (k[1] + W1) & _MASK)
    return x


def uniform(seed: int, offset: int, slot: int, purpose: int) -> float:
    """The step's uniform draw for (seed, offset, slot, purpose)."""
    key = (seed & _MASK, (seed >> 32) & _MASK)
    ctr = (offset & _MASK, (offset >> 32) & _MASK, slot & _MASK, purpose & _MASK)
    x0 = philox4x32_10(ctr, key)[0]
    return (x0 >> 8) * (1.0 / 16777216.0)
