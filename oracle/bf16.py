"""bfloat16 storage format: bit patterns to float64 (test infrastructure only).

A bfloat16 value is the upper 16 bits of an IEEE binary32; widening it is exact.
"""

import numpy as np


def bf16_bits_to_f64(bits):
    """Widen an array of bfloat16 bit patterns (uint16) to float64, exactly."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def as_f64(x):
    """float64 view of an input that is either bfloat16 bits (uint16) or a float array."""
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return bf16_bits_to_f64(x)
    return x.astype(np.float64)


def round_bf16(x):
    """Round float64 values to the nearest bfloat16 (ties to even), returned as float64.

    Rounds from float64 directly (no intermediate float32, so no double
    rounding): x = m * 2^e with 0.5 <= |m| < 1 has 8 significant bits kept.
    Values are assumed inside the normal bfloat16 range (|x| >= 2^-126 or 0).
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.rint(m * 256.0), e - 8)


def bf16_tie_distance(x):
    """Distance of x to the nearest bfloat16 rounding boundary, relative to |x|.

    A value this close to a boundary may round the other way in any other
    working precision; comparisons with another implementation excuse it.
    """
    x = np.asarray(x, dtype=np.float64)
    m, _ = np.frexp(x)
    s = np.abs(m) * 256.0                      # in [128, 256): rounding boundaries at k + 0.5
    d = np.abs(s - (np.floor(s) + 0.5))
    with np.errstate(divide="ignore", invalid="ignore"):
        return np.where(x == 0, np.inf, d / s)
