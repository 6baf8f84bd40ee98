"""Philox4x32-10 counter-based generator and the uniform stream of the cycle.

Test infrastructure only (see the package docstring).

Philox4x32-10 is taken from its published definition (Salmon et al., "Parallel
random numbers: as easy as 1, 2, 3", SC'11): ten rounds of two 32x32->64-bit
multiplies with a Weyl-sequence key schedule. The pages on the method do not
name a generator; the cycle keys one uniform per (request, position, stage):

    key = (seed & 0xffffffff, seed >> 32)
    ctr = (request, position, stage, 0)        position is 1-based
    u   = (word0 + 0.5) * 2**-32                strictly inside (0, 1)

Stage ids: 0 = draft sample, 1 = accept test, 2 = residual / bonus sample.
"""

MASK32 = 0xFFFFFFFF
PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85

STAGE_DRAFT = 0
STAGE_ACCEPT = 1
STAGE_RESAMPLE = 2


def philox4x32_10(ctr, key):
    """Return the four 32-bit output words of Philox4x32 with 10 rounds.

    ``ctr`` is four 32-bit ints, ``key`` two. Each round multiplies counter
    words 0 and 2 by the two round constants, splits the 64-bit products into
    high and low halves, and recombines them with words 1 and 3 and the key;
    the key is bumped by the Weyl constants between rounds.
    """
    c0, c1, c2, c3 = (int(v) & MASK32 for v in ctr)
    k0, k1 = (int(v) & MASK32 for v in key)
    for rnd in range(10):
        if rnd > 0:
            k0 = (k0 + PHILOX_W0) & MASK32
            k1 = (k1 + PHILOX_W1) & MASK32
        prod0 = PHILOX_M0 * c0
        prod1 = PHILOX_M1 * c2
        hi0, lo0 = prod0 >> 32, prod0 & MASK32
        hi1, lo1 = prod1 >> 32, prod1 & MASK32
        c0, c1, c2, c3 = (hi1 ^ c1 ^ k0) & MASK32, lo1, (hi0 ^ c3 ^ k1) & MASK32, lo0
    return (c0, c1, c2, c3)


def uniform(seed, request, position, stage):
    """One uniform in (0, 1) for (seed, request, position, stage), exact in float64."""
    seed = int(seed)
    words = philox4x32_10((request, position, stage, 0), (seed & MASK32, (seed >> 32) & MASK32))
    return (words[0] + 0.5) * 2.0 ** -32
