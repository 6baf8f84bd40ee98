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
