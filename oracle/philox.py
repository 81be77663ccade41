"""Philox4x32-10 counter-based random number generator — oracle side.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Definition (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
1, 2, 3", SC'11, section on the Philox family): the state is four 32-bit
counter words and two 32-bit key words.  One round maps

    (c0, c1, c2, c3) -> (hi(M1*c2) ^ c1 ^ k0,  lo(M1*c2),
                         hi(M0*c0) ^ c3 ^ k1,  lo(M0*c0))

with the multipliers M0 = 0xD2511F53, M1 = 0xCD9E8D57, where hi/lo are the
upper/lower 32 bits of the 64-bit product.  Between rounds the key is bumped
by the Weyl constants (0x9E3779B9, 0xBB67AE85) modulo 2^32.  Philox4x32-10
applies ten rounds (nine key bumps).

Two implementations live here: `philox4x32_10` (vectorised numpy, uint64
arithmetic masked to 32 bits) and `philox4x32_10_scalar` (Python integers).
Tests require them to agree, and pin both to cuRAND's host-side Philox4x32-10
generator (an independent implementation of the same published generator,
run on the CPU): its first output blocks are the counters (0, 0, i, 0) under
the key (seed low word, seed high word).
"""

import numpy as np

PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85
MASK32 = 0xFFFFFFFF


def philox4x32_10_scalar(counter, key):
    """Ten Philox rounds on one counter, with Python integers.

    counter: 4 ints in [0, 2^32); key: 2 ints in [0, 2^32).
    Returns a tuple of 4 ints in [0, 2^32).
    """
    c0, c1, c2, c3 = (int(x) & MASK32 for x in counter)
    k0, k1 = (int(x) & MASK32 for x in key)
    for r in range(10):
        if r > 0:
            k0 = (k0 + PHILOX_W0) & MASK32
            k1 = (k1 + PHILOX_W1) & MASK32
        p0 = PHILOX_M0 * c0
        p1 = PHILOX_M1 * c2
        c0, c1, c2, c3 = (
            ((p1 >> 32) ^ c1 ^ k0) & MASK32,
            p1 & MASK32,
            ((p0 >> 32) ^ c3 ^ k1) & MASK32,
            p0 & MASK32,
        )
    return c0, c1, c2, c3


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Vectorised Philox4x32-10.

    c0..c3: integer arrays (broadcastable) holding 32-bit counter words;
    k0, k1: 32-bit key words (Python ints).  Returns four uint32 arrays.
    Products of two 32-bit numbers fit in uint64 exactly.
    """
    m = np.uint64(MASK32)
    c0 = np.asarray(c0, dtype=np.uint64) & m
    c1 = np.asarray(c1, dtype=np.uint64) & m
    c2 = np.asarray(c2, dtype=np.uint64) & m
    c3 = np.asarray(c3, dtype=np.uint64) & m
    c0, c1, c2, c3 = np.broadcast_arrays(c0, c1, c2, c3)
    k0 = int(k0) & MASK32
    k1 = int(k1) & MASK32
    for r in range(10):
        if r > 0:
            k0 = (k0 + PHILOX_W0) & MASK32
            k1 = (k1 + PHILOX_W1) & MASK32
        p0 = np.uint64(PHILOX_M0) * c0
        p1 = np.uint64(PHILOX_M1) * c2
        n0 = ((p1 >> np.uint64(32)) ^ c1 ^ np.uint64(k0)) & m
        n1 = p1 & m
        n2 = ((p0 >> np.uint64(32)) ^ c3 ^ np.uint64(k1)) & m
        n3 = p0 & m
        c0, c1, c2, c3 = n0, n1, n2, n3
    return (c0.astype(np.uint32), c1.astype(np.uint32),
            c2.astype(np.uint32), c3.astype(np.uint32))
