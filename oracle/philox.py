"""Philox4x32-10 counter-based generator, written from its published definition
(Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC'11).

Test infrastructure (see the package docstring). The GPU path carries its own,
independent implementation of the same published function; the two are tied
together only by the published known-answer vectors in ``tests/golden``.

Uniforms drawn by the stochastic verify (EAGLE-2 page, §"先把投机解码的账本摆清楚":
accept with probability a, else resample from the residual):

* acceptance test of the child at tree position j of request b in round r:
  counter (r_lo, r_hi, 512*b + j, 0x80000000), word 0, top 24 bits,
  u = k * 2^-24 in [0, 1).
* Gumbel noise for token v when the residual of position i is sampled:
  counter (r_lo, r_hi, 512*b + i, v >> 2), word v & 3, top 23 bits,
  u = (k + 0.5) * 2^-23 in (0, 1).

Key = (seed_lo, seed_hi).
"""

import numpy as np

M0 = np.uint64(0xD2511F53)
M1 = np.uint64(0xCD9E8D57)
W0 = np.uint32(0x9E3779B9)
W1 = np.uint32(0xBB67AE85)
MASK32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(ctr, key):
    """Ten Philox rounds. ``ctr`` is a (4, n) uint32 array (or 4-tuple), ``key`` a 2-tuple.

    One round: multiply words 0 and 2 by the two round constants (64-bit
    products split into hi/lo halves), then permute and xor the high halves
    with the other two words and the key; the key is bumped by the Weyl
    constants between rounds.
    """
    c = [np.asarray(x, dtype=np.uint64) & MASK32 for x in ctr]
    k0 = np.uint64(int(key[0]) & 0xFFFFFFFF)
    k1 = np.uint64(int(key[1]) & 0xFFFFFFFF)
    for rnd in range(10):
        if rnd > 0:
            k0 = (k0 + np.uint64(W0)) & MASK32
            k1 = (k1 + np.uint64(W1)) & MASK32
        p0 = M0 * c[0]
        p1 = M1 * c[2]
        hi0, lo0 = p0 >> np.uint64(32), p0 & MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & MASK32
        c = [hi1 ^ c[1] ^ k0, lo1, hi0 ^ c[3] ^ k1, lo0]
    return [x.astype(np.uint32) for x in c]


def _key(seed):
    return (seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF)


def accept_uniform(seed, rnd, b, pos):
    """24-bit uniform in [0, 1) for the acceptance test of tree position ``pos``."""
    w = philox4x32_10((rnd & 0xFFFFFFFF, (rnd >> 32) & 0xFFFFFFFF, 512 * b + pos, 0x80000000),
                      _key(seed))
    k = int(w[0]) >> 8
    return k * 2.0 ** -24


def gumbel_uniforms(seed, rnd, b, pos, V):
    """23-bit uniforms in (0, 1) for every token 0..V-1 (Gumbel noise of the residual sample)."""
    v = np.arange(V, dtype=np.uint64)
    n = v.size
    ctr = (np.full(n, rnd & 0xFFFFFFFF, np.uint64), np.full(n, (rnd >> 32) & 0xFFFFFFFF, np.uint64),
           np.full(n, 512 * b + pos, np.uint64), v >> np.uint64(2))
    w = philox4x32_10(ctr, _key(seed))
    words = np.stack(w, axis=0)  # (4, n)
    sel = words[(v & np.uint64(3)).astype(np.int64), np.arange(n)]
    k = (sel >> np.uint32(9)).astype(np.float64)
    return (k + 0.5) * 2.0 ** -23
