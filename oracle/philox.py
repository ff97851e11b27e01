"""Philox4x32-10 and the per-element random draw of stochastic rounding.
Test infrastructure only (see ``oracle/__init__.py``).

Philox4x32 is the counter-based generator of Salmon, Moraes, Dror and Shaw,
"Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11), section 3: a 128-bit
counter (four 32-bit words) and a 64-bit key (two words); each of the ten
rounds multiplies words 0 and 2 by the constants 0xD2511F53 and 0xCD9E8D57
into 64-bit products and permutes/XORs the halves with the other two words
and the round key; the key is bumped by the Weyl constants 0x9E3779B9 and
0xBB67AE85 between rounds.

The pages ask that the re-quantization use stochastic rounding ("Re-quantization
with stochastic rounding", which also notes that Blackwell accelerates SR in
hardware) and that the kernels be fully deterministic ("Kernels for
low-precision training"); the generator makes SR a pure function of
(seed, counter offset, position).  Draw layout (a convention, shared by the GPU
library by contract):
  * draws are 16-bit values U, one per PAIR of output elements (two
    consecutive elements along the output row, i.e. along the MXFP8 block);
    the pair's first element uses U, its second bitrev16(U);
  * U(K) is the 16-bit half (K & 1) -- the low half when K is even -- of
    output word (K >> 1) & 3 of Philox4x32-10 with
      key     = (seed & 0xFFFFFFFF, seed >> 32)
      counter = (q & 0xFFFFFFFF, q >> 32, off & 0xFFFFFFFF, off >> 32), q = K >> 3
  * the pair key K comes from the source coordinates of the pair's first
    element (see ``requant``).
Pairing two elements on one draw is how Blackwell's stochastic-rounding
conversion consumes its random operand (two elements per 16 bits, the second
bit-reversed), so the GPU can use it and stay bit-exact with this rule.
"""
from __future__ import annotations

import numpy as np

M0 = 0xD2511F53
M1 = 0xCD9E8D57
W0 = 0x9E3779B9
W1 = 0xBB67AE85
ROUNDS = 10
_MASK = np.uint64(0xFFFFFFFF)


def philox4x32(counter, key, rounds: int = ROUNDS):
    """Apply Philox4x32-``rounds`` to counters.

    counter: uint array [..., 4] (32-bit words); key: (k0, k1) scalars or
    arrays broadcastable to counter[..., 0].  Returns uint32 [..., 4]."""
    c = np.asarray(counter, dtype=np.uint64) & _MASK
    c0, c1, c2, c3 = c[..., 0], c[..., 1], c[..., 2], c[..., 3]
    k0 = np.asarray(key[0], dtype=np.uint64) & _MASK
    k1 = np.asarray(key[1], dtype=np.uint64) & _MASK
    for rnd in range(rounds):
        if rnd > 0:
            k0 = (k0 + np.uint64(W0)) & _MASK
            k1 = (k1 + np.uint64(W1)) & _MASK
        p0 = np.uint64(M0) * c0            # exact: both factors < 2^32
        p1 = np.uint64(M1) * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK
        c0, c1, c2, c3 = (hi1 ^ c1 ^ k0), lo1, (hi0 ^ c3 ^ k1), lo0
    return np.stack([c0, c1, c2, c3], axis=-1).astype(np.uint32)


def pair_draws16(seed: int, offset: int, K) -> np.ndarray:
    """The 16-bit draw U(K) of each pair key K (int64 array) under
    (seed, counter offset).  One Philox call serves 8 consecutive keys."""
    K = np.asarray(K, dtype=np.uint64)
    q = K >> np.uint64(3)
    off = np.uint64(offset)
    ctr = np.stack([q & _MASK, q >> np.uint64(32),
                    np.broadcast_to(off & _MASK, q.shape),
                    np.broadcast_to(off >> np.uint64(32), q.shape)], axis=-1)
    key = (np.uint64(seed) & _MASK, np.uint64(seed) >> np.uint64(32))
    words = philox4x32(ctr, key)
    w = np.take_along_axis(words, ((K >> np.uint64(1)) & np.uint64(3)).astype(np.int64)[..., None],
                           axis=-1)[..., 0].astype(np.uint32)
    odd = (K & np.uint64(1)).astype(bool)
    return np.where(odd, w >> np.uint32(16), w & np.uint32(0xFFFF)).astype(np.uint32)


def bitrev16(u) -> np.ndarray:
    """Reverse the order of the low 16 bits."""
    u = np.asarray(u, dtype=np.uint32)
    r = np.zeros_like(u)
    for b in range(16):
        r |= ((u >> np.uint32(b)) & np.uint32(1)) << np.uint32(15 - b)
    return r
