"""Philox4x64-10 counter-based generator for the oracle (test infrastructure).

Written from the published definition: J. K. Salmon, M. A. Moraes, R. O. Dror,
D. E. Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11), the
Philox-4x64 bijection with 10 rounds.  One round maps the counter words
(c0, c1, c2, c3) with key (k0, k1) to

    (hi(M1*c2) ^ c1 ^ k0,  lo(M1*c2),  hi(M0*c0) ^ c3 ^ k1,  lo(M0*c0))

and the key is bumped by the Weyl constants between rounds.

The pages on speculative sampling only say that a seeded 32-bit generator makes
draws reproducible ("Choosing the next word", section "Where the randomness
comes from, and where it stops"); the counter layout below is this project's
reading: key = (seed, 0), counter = (offset, row, draw, 0) and the uniform is
the top 53 bits of the first output word, u = (w0 >> 11) * 2**-53 in [0, 1).

Plain Python integers are used on purpose: slow, but every operation is exact
and visible.  The CUDA side carries its own, separately written copy.
"""

MASK64 = (1 << 64) - 1

# Round multipliers and key-schedule (Weyl) constants of Philox-4x64.
PHILOX_M0 = 0xD2E7470EE14C6C93
PHILOX_M1 = 0xCA5A826395121157
PHILOX_W0 = 0x9E3779B97F4A7C15  # golden ratio
PHILOX_W1 = 0xBB67AE8584CAA73B  # sqrt(3) - 1

ROUNDS = 10


def _mulhilo(a, b):
    """Full 128-bit product of two 64-bit words, as (high word, low word)."""
    prod = a * b
    return prod >> 64, prod & MASK64


def philox4x64_10(counter, key):
    """Apply the 10-round Philox-4x64 bijection.

    counter: 4 unsigned 64-bit words; key: 2 unsigned 64-bit words.
    Returns the 4 output words.
    """
    c0, c1, c2, c3 = (int(w) & MASK64 for w in counter)
    k0, k1 = (int(w) & MASK64 for w in key)
    for rnd in range(ROUNDS):
        if rnd:
            k0 = (k0 + PHILOX_W0) & MASK64
            k1 = (k1 + PHILOX_W1) & MASK64
        hi0, lo0 = _mulhilo(PHILOX_M0, c0)
        hi1, lo1 = _mulhilo(PHILOX_M1, c2)
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return c0, c1, c2, c3


def first_word(seed, offset, row, draw):
    """First 64-bit output word of the block at counter (offset, row, draw, 0)."""
    return philox4x64_10((offset, row, draw, 0), (seed, 0))[0]


def uniform(seed, offset, row, draw):
    """The uniform in [0, 1) used for draw number `draw` of batch row `row`."""
    return (first_word(seed, offset, row, draw) >> 11) * 2.0 ** -53
