"""Philox4x32-10 counter-based generator for the oracle (test infrastructure).

TEST INFRASTRUCTURE ONLY: imported by tests/, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py``; never by the CUDA path.

Written from the generator's published definition (Salmon, Moraes, Dror,
Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11, the Philox-4x32
S-box with 10 rounds).  One round maps the counter (c0, c1, c2, c3) under key
(k0, k1) to

    (hi(B*c2) ^ c1 ^ k0,  lo(B*c2),  hi(A*c0) ^ c3 ^ k1,  lo(A*c0))

with A = 0xD2511F53, B = 0xCD9E8D57 (hi/lo = upper/lower 32 bits of the
64-bit product); between rounds the key is bumped by the Weyl constants
(0x9E3779B9, 0xBB67AE85).  The pages ask only for "seeded Philox uniforms
per position"; the stream layout below is this library's own:

    counter = (b, t, purpose, cycle mod 2**32),  key = (seed lo, seed hi)
    purpose 0 = walk draw at position t, 1 = accept draw at position t,
            2 = residual / bonus draw (t = K)
    u = (x0 >> 8) * 2**-24  in [0, 1)   (x0 = first output word)
"""
from __future__ import annotations

import numpy as np

PHILOX_A = 0xD2511F53
PHILOX_B = 0xCD9E8D57
WEYL_0 = 0x9E3779B9
WEYL_1 = 0xBB67AE85
MASK32 = 0xFFFFFFFF

PURPOSE_WALK = 0
PURPOSE_ACCEPT = 1
PURPOSE_RESAMPLE = 2


def philox4x32_10(ctr, key):
    """Philox4x32-10 on an array of counters.

    ctr: uint32-compatible array [..., 4]; key: uint32-compatible [..., 2]
    (broadcast against ctr).  Returns uint32 [..., 4].
    """
    c = np.asarray(ctr, dtype=np.uint64) & MASK32
    k = np.asarray(key, dtype=np.uint64) & MASK32
    c0, c1, c2, c3 = (c[..., i].copy() for i in range(4))
    k0 = np.broadcast_to(k[..., 0], c0.shape).copy()
    k1 = np.broadcast_to(k[..., 1], c0.shape).copy()
    A = np.uint64(PHILOX_A)
    B = np.uint64(PHILOX_B)
    for rnd in range(10):
        if rnd:
            k0 = (k0 + np.uint64(WEYL_0)) & np.uint64(MASK32)
            k1 = (k1 + np.uint64(WEYL_1)) & np.uint64(MASK32)
        p0 = A * c0          # < 2**64: both factors < 2**32
        p1 = B * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & np.uint64(MASK32)
        hi1, lo1 = p1 >> np.uint64(32), p1 & np.uint64(MASK32)
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return np.stack([c0, c1, c2, c3], axis=-1).astype(np.uint32)


def philox_scalar(ctr, key):
    """The same generator in plain Python integers (one counter)."""
    c0, c1, c2, c3 = (int(x) & MASK32 for x in ctr)
    k0, k1 = (int(x) & MASK32 for x in key)
    for rnd in range(10):
        if rnd:
            k0 = (k0 + WEYL_0) & MASK32
            k1 = (k1 + WEYL_1) & MASK32
        p0 = PHILOX_A * c0
        p1 = PHILOX_B * c2
        c0, c1, c2, c3 = ((p1 >> 32) ^ c1 ^ k0, p1 & MASK32,
                          (p0 >> 32) ^ c3 ^ k1, p0 & MASK32)
    return (c0, c1, c2, c3)


def seed_key(seed: int):
    s = int(seed) & 0xFFFFFFFFFFFFFFFF
    return (s & MASK32, s >> 32)


def uniforms(seed: int, cycle: int, b, t, purpose: int) -> np.ndarray:
    """u in [0,1) (float64, exactly a multiple of 2**-24) for the streams
    (b, t, purpose, cycle) under ``seed``; b and t broadcast."""
    b = np.asarray(b, dtype=np.uint64)
    t = np.asarray(t, dtype=np.uint64)
    b, t = np.broadcast_arrays(b, t)
    ctr = np.stack([b, t, np.full(b.shape, purpose, np.uint64),
                    np.full(b.shape, int(cycle) & MASK32, np.uint64)], -1)
    x0 = philox4x32_10(ctr, seed_key(seed))[..., 0].astype(np.uint64)
    return (x0 >> np.uint64(8)).astype(np.float64) * 2.0 ** -24


def walk_uniforms(seed, cycle, B, K):
    b, t = np.meshgrid(np.arange(B), np.arange(K), indexing="ij")
    return uniforms(seed, cycle, b, t, PURPOSE_WALK)


def accept_uniforms(seed, cycle, B, K):
    b, t = np.meshgrid(np.arange(B), np.arange(K), indexing="ij")
    return uniforms(seed, cycle, b, t, PURPOSE_ACCEPT)


def resample_uniforms(seed, cycle, B, K):
    return uniforms(seed, cycle, np.arange(B), np.full(B, K), PURPOSE_RESAMPLE)
