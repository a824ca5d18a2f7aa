"""Attention dropout regenerated from a counter-based generator.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Passage followed
----------------
P3 section 05 (production kernels, fourth difference): dropout keeps no
B x H x N x N mask for the backward pass; the kernel stores only the seed
and offset of a Philox counter-based generator and the backward pass draws
the very same mask again from them.

The generator is Philox4x32-10 as published by Salmon, Moraes, Dror and
Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3" (SC 2011): a 128-bit
counter (four 32-bit words) and a 64-bit key (two words) go through ten
rounds; each round multiplies counter words 0 and 2 by two fixed 32-bit
multipliers, keeps the high and low halves of the 64-bit products, XORs the
high halves with the other two counter words and the key words, and permutes
the words; between rounds each key word is incremented by its Weyl constant
(the golden ratio and sqrt(3) - 1 in 32-bit fixed point).

The pages fix neither how counters map to attention entries nor how random
bits become keep decisions.  The reading taken here:

* entry (head bh, query row i, key column j) uses the counter
  (j // 16, i, bh, offset) under the key (seed mod 2^32, seed div 2^32);
  bh = b * H + h;
* the four 32-bit output words give sixteen 8-bit integers: word (j // 4) % 4
  and its byte j % 4, counted from the least significant byte;
* the entry is kept iff that integer is >= t, with t = round(p * 256) (so
  the drop probability is t / 256, p quantised to 2^-8); kept probabilities
  are multiplied by 256 / (256 - t), the inverse of the keep probability, so
  that the expected output equals the plain output.

One generator call thus serves sixteen entries of a row; the coarser
quantisation of p (the realised drop probability of p = 0.1 is 26/256) is
the price of half the generator work per entry.

Dropout acts on the normalised probabilities P (after the softmax); LSE is
the softmax normaliser and is not affected.
"""
from __future__ import annotations

import numpy as np

# Philox4x32 constants of the published definition.
PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9  # golden ratio, 32-bit fixed point
PHILOX_W1 = 0xBB67AE85  # sqrt(3) - 1, 32-bit fixed point
_LO = np.uint64(0xFFFFFFFF)


def philox4x32_10(counters, key):
    """Philox4x32 with ten rounds.

    ``counters``: integer array [..., 4] (32-bit words); ``key``: two 32-bit
    words.  Returns uint32 [..., 4].  Products are formed in uint64, where a
    32 x 32 bit product is exact.
    """
    c = np.asarray(counters, dtype=np.uint64) & _LO
    x0, x1, x2, x3 = (c[..., n] for n in range(4))
    k0 = np.uint64(int(key[0]) & 0xFFFFFFFF)
    k1 = np.uint64(int(key[1]) & 0xFFFFFFFF)
    for _ in range(10):
        p0 = np.uint64(PHILOX_M0) * x0
        p1 = np.uint64(PHILOX_M1) * x2
        hi0, lo0 = p0 >> np.uint64(32), p0 & _LO
        hi1, lo1 = p1 >> np.uint64(32), p1 & _LO
        x0, x1, x2, x3 = hi1 ^ x1 ^ k0, lo1, hi0 ^ x3 ^ k1, lo0
        k0 = (k0 + np.uint64(PHILOX_W0)) & _LO
        k1 = (k1 + np.uint64(PHILOX_W1)) & _LO
    return np.stack([x0, x1, x2, x3], axis=-1).astype(np.uint32)


def threshold(p: float) -> int:
    """t = round(p * 256); entries whose 8-bit draw is below t are dropped."""
    if not (0.0 <= p < 1.0):
        raise ValueError("dropout probability must be in [0, 1)")
    t = int(np.floor(p * 256.0 + 0.5))
    if t >= 256:
        raise ValueError("dropout probability rounds to 1")
    return t


def keep_scale(p: float) -> float:
    """1 / keep probability = 256 / (256 - t)."""
    return 256.0 / (256.0 - threshold(p))


def draws8(seed: int, offset: int, bh: int, rows, n_keys: int):
    """The 8-bit draws of head ``bh`` for query rows ``rows`` and keys
    0 .. n_keys-1: uint32 array [len(rows), n_keys] with values < 256."""
    rows = np.asarray(rows, dtype=np.int64)
    n_groups = (n_keys + 15) // 16
    ctr = np.empty((len(rows), n_groups, 4), dtype=np.uint64)
    ctr[..., 0] = np.arange(n_groups, dtype=np.uint64)[None, :]
    ctr[..., 1] = rows.astype(np.uint64)[:, None]
    ctr[..., 2] = np.uint64(bh)
    ctr[..., 3] = np.uint64(offset & 0xFFFFFFFF)
    words = philox4x32_10(ctr, (seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF))  # [rows, groups, 4]
    octets = np.stack([(words >> (8 * b)) & 0xFF for b in range(4)], axis=-1)  # [rows, groups, 4, 4]
    return octets.reshape(len(rows), n_groups * 16)[:, :n_keys]


def keep_mask(seed: int, offset: int, p: float, bh: int, n_queries: int, n_keys: int, rows=None):
    """Boolean keep mask [rows, n_keys] of head ``bh`` (all rows if None)."""
    if rows is None:
        rows = np.arange(n_queries)
    return draws8(seed, offset, bh, rows, n_keys) >= threshold(p)
