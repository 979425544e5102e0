"""Philox-4x32-10, written from its published definition.

Source: J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel Random
Numbers: As Easy as 1, 2, 3", SC'11 -- section 4 (the Philox S-box) and its
table of round multipliers / Weyl key increments for the 4x32 variant.

The FlashSampling pages only say that each tile draws its Gumbel noise "from
the tile's RNG state" (FlashSampling: Fast and Memory-Efficient Exact Sampling,
summary page, Method); the generator itself is this build's reading: a
counter-based generator, so every (row, step, vocabulary id) owns its own
stream position and the noise does not depend on how the vocabulary is tiled.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Pinned by ``tests/test_oracle_philox.py`` against (a) the Random123
known-answer vectors and (b) Triton's ``tl.philox`` run in its CPU interpreter.
"""

import numpy as np

# Round multipliers of the 4x32 variant (SC'11, Philox parameter table).
PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
# Weyl-sequence key increments: golden ratio and sqrt(3) - 1, as 32-bit fractions.
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85
PHILOX_ROUNDS = 10

_MASK32 = 0xFFFFFFFF


def _mulhilo32(m, x):
    """Full 64-bit product of the 32-bit constant ``m`` and uint32 array ``x``,
    returned as its (high, low) 32-bit halves."""
    p = np.uint64(m) * x.astype(np.uint64)
    return (p >> np.uint64(32)).astype(np.uint32), (p & np.uint64(_MASK32)).astype(np.uint32)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Apply the 10-round Philox-4x32 bijection to counter (c0, c1, c2, c3)
    under key (k0, k1).

    ``c*`` are uint32 arrays of one shape (broadcastable); ``k0``/``k1`` are
    Python ints (the key is the same for every element).  Returns the four
    uint32 output words.

    One round (SC'11 section 4): two 32x32->64 multiplies of words 0 and 2 by
    the round multipliers; the high halves are xored with the other two words
    and the round key, the low halves pass through, and the words are permuted:
        out0 = hi(M1*c2) ^ c1 ^ k0      out1 = lo(M1*c2)
        out2 = hi(M0*c0) ^ c3 ^ k1      out3 = lo(M0*c0)
    Between rounds the key advances by the Weyl increments (W0, W1) mod 2^32.
    """
    c0 = np.asarray(c0, dtype=np.uint32)
    c1 = np.asarray(c1, dtype=np.uint32)
    c2 = np.asarray(c2, dtype=np.uint32)
    c3 = np.asarray(c3, dtype=np.uint32)
    c0, c1, c2, c3 = np.broadcast_arrays(c0, c1, c2, c3)
    k0 = int(k0) & _MASK32
    k1 = int(k1) & _MASK32
    for r in range(PHILOX_ROUNDS):
        if r > 0:
            k0 = (k0 + PHILOX_W0) & _MASK32
            k1 = (k1 + PHILOX_W1) & _MASK32
        hi0, lo0 = _mulhilo32(PHILOX_M0, c0)
        hi1, lo1 = _mulhilo32(PHILOX_M1, c2)
        c0, c1, c2, c3 = (hi1 ^ c1 ^ np.uint32(k0), lo1,
                          hi0 ^ c3 ^ np.uint32(k1), lo0)
    return c0, c1, c2, c3
