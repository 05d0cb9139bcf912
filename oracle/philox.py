"""Philox4x32-10, written from its published definition (oracle side).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this package; the CUDA library never does.

Source of the definition: J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel Random
Numbers: As Easy as 1, 2, 3", SC'11, section 3 (the Philox S-box: two 32x32->64 multiplies whose
high halves are xored with the other counter words and the round key; the Weyl key schedule;
ten rounds for the 4x32 variant).  The multipliers and Weyl increments below are the ones the
paper publishes for Philox4x32.

How the sampler keys and counts it (a definition of this project, because the pages name
"Philox(seed, position)" and a counter that persists across verify windows but give no layout):
key = (seed low 32 bits, seed high 32 bits); counter = (position low, position high,
draw-counter low, draw-counter high); the row's uniform is the top 24 bits of the first output
word scaled by 2^-24, so u is an exact float in [0, 1).
"""
from __future__ import annotations

MASK32 = 0xFFFFFFFF
PHILOX_M4x32_0 = 0xD2511F53
PHILOX_M4x32_1 = 0xCD9E8D57
PHILOX_W32_0 = 0x9E3779B9
PHILOX_W32_1 = 0xBB67AE85


def philox4x32_10(ctr, key):
    """Ten Philox4x32 rounds of the 128-bit counter `ctr` (4 ints) under the 64-bit key `key` (2 ints)."""
    c0, c1, c2, c3 = (int(v) & MASK32 for v in ctr)
    k0, k1 = (int(v) & MASK32 for v in key)
    for _ in range(10):
        prod0 = PHILOX_M4x32_0 * c0
        prod1 = PHILOX_M4x32_1 * c2
        hi0, lo0 = prod0 >> 32, prod0 & MASK32
        hi1, lo1 = prod1 >> 32, prod1 & MASK32
        c0, c1, c2, c3 = (hi1 ^ c1 ^ k0) & MASK32, lo1, (hi0 ^ c3 ^ k1) & MASK32, lo0
        k0 = (k0 + PHILOX_W32_0) & MASK32
        k1 = (k1 + PHILOX_W32_1) & MASK32
    return (c0, c1, c2, c3)


def row_uniform(seed: int, position: int, counter: int) -> float:
    """The row's uniform u in [0, 1) for Philox(seed, position) at the slot's draw counter."""
    seed &= (1 << 64) - 1
    position &= (1 << 64) - 1
    counter &= (1 << 64) - 1
    out = philox4x32_10((position & MASK32, position >> 32, counter & MASK32, counter >> 32),
                        (seed & MASK32, seed >> 32))
    return (out[0] >> 8) * (2.0 ** -24)
