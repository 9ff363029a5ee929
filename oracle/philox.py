"""Counter-based standard-normal draws for the oracle (test infrastructure only).

Philox4x32 with 10 rounds, from its published definition (Salmon, Moraes,
Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011): a
round multiplies counter words 0 and 2 by 0xD2511F53 and 0xCD9E8D57, and the
new counter is (hi(c2*M1) ^ c1 ^ k0, lo(c2*M1), hi(c0*M0) ^ c3 ^ k1,
lo(c0*M0)); the key is bumped by the Weyl constants 0x9E3779B9 and
0xBB67AE85 between rounds.  A standard normal is formed from the first two
output words by Box-Muller: u1 = (x0 + 1) / 2^32, u2 = x1 / 2^32,
z = sqrt(-2 ln u1) cos(2 pi u2), evaluated here in float64.

The library draws Q this way when no draw is injected; element (j, k) of
compressed tensor number t (in bucket order among compressed tensors), drawn
at call number `counter`, uses counter words (e mod 2^32, (e >> 32) xor
(t << 8), counter mod 2^32, counter >> 32) with e = j * RP + k (RP the rank
rounded up to a power of two) and key (seed mod 2^32, seed >> 32).  This file
restates that layout and shares no code with the library.
"""

from __future__ import annotations

import numpy as np

M0 = np.uint64(0xD2511F53)
M1 = np.uint64(0xCD9E8D57)
W0 = np.uint32(0x9E3779B9)
W1 = np.uint32(0xBB67AE85)
MASK = np.uint64(0xFFFFFFFF)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Vectorised Philox4x32-10 over numpy uint32 arrays; returns 4 arrays."""
    c0, c1, c2, c3 = (np.asarray(x, dtype=np.uint32) for x in (c0, c1, c2, c3))
    k0 = np.asarray(k0, dtype=np.uint32).copy()
    k1 = np.asarray(k1, dtype=np.uint32).copy()
    with np.errstate(over="ignore"):
        for _ in range(10):
            p0 = c0.astype(np.uint64) * M0
            p1 = c2.astype(np.uint64) * M1
            hi0 = (p0 >> np.uint64(32)).astype(np.uint32)
            lo0 = (p0 & MASK).astype(np.uint32)
            hi1 = (p1 >> np.uint64(32)).astype(np.uint32)
            lo1 = (p1 & MASK).astype(np.uint32)
            c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
            k0 = k0 + W0
            k1 = k1 + W1
    return c0, c1, c2, c3


def library_draw(cols, rank, rp, tensor, counter, seed):
    """The (cols x rank) standard-normal draw the library makes for
    compressed tensor number `tensor` at call `counter` (float64)."""
    j = np.arange(cols, dtype=np.uint64)[:, None]
    k = np.arange(rank, dtype=np.uint64)[None, :]
    e = j * np.uint64(rp) + k
    c0 = (e & MASK).astype(np.uint32)
    c1 = ((e >> np.uint64(32)) & MASK).astype(np.uint32) ^ np.uint32((tensor << 8) & 0xFFFFFFFF)
    c2 = np.full(e.shape, counter & 0xFFFFFFFF, dtype=np.uint32)
    c3 = np.full(e.shape, (counter >> 32) & 0xFFFFFFFF, dtype=np.uint32)
    x0, x1, _, _ = philox4x32_10(c0, c1, c2, c3, seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF)
    u1 = (x0.astype(np.float64) + 1.0) / 4294967296.0
    u2 = x1.astype(np.float64) / 4294967296.0
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
