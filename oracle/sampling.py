"""Inverse-CDF sampling and greedy selection, float64 (test infrastructure only).

The pages fix the sampling law (softmax of the logits, sampled left to right,
DSpark summary page, 방법论 › 반자기회귀 생성) but not the sampler. The reading
used throughout: one uniform u per draw, tokens in index order,

    x = min{ i : u * S < C_i },   C_i = w_0 + ... + w_i,   S = C_{V-1}.

A zero-weight token is never drawn: C_i = C_{i-1} there, so the first index
with C_i > u*S always has w_i > 0.
"""

import numpy as np


def softmax_weights(logits, temperature):
    """Unnormalised weights exp(l/T - max(l/T)) in float64, and their sum."""
    scaled = np.asarray(logits, dtype=np.float64) / np.float64(temperature)
    w = np.exp(scaled - scaled.max())
    return w, float(w.sum())


def inverse_cdf(weights, u):
    """Draw min{i : u*S < C_i} and report the draw's margin.

    Returns (index, margin). The margin is the distance, in probability units,
    from u*S to the nearer end of the chosen token's CDF interval,
    min(u*S - C_{x-1}, C_x - u*S) / S; a draw whose margin is tiny is a near-tie
    that any other rounding of the same arithmetic may resolve differently.
    """
    w = np.asarray(weights, dtype=np.float64)
    if w.ndim != 1 or w.size == 0:
        raise ValueError("weights must be a non-empty vector")
    if np.any(w < 0) or not np.all(np.isfinite(w)):
        raise ValueError("weights must be finite and non-negative")
    c = np.cumsum(w)
    s = c[-1]
    if not s > 0:
        raise ValueError("weights sum to zero")
    t = u * s
    above = np.flatnonzero(c > t)
    x = int(above[0]) if above.size else int(np.flatnonzero(w > 0)[-1])
    lower = c[x - 1] if x > 0 else 0.0
    margin = min(t - lower, c[x] - t) / s
    return x, float(margin)


def argmax_first(values):
    """Greedy choice: the largest value, lowest index on ties. Returns (index, gap).

    ``gap`` is the difference between the largest and the second-largest value
    (0 on an exact tie), the near-tie measure for greedy decisions.
    """
    v = np.asarray(values, dtype=np.float64)
    x = int(np.argmax(v))  # numpy returns the first occurrence of the maximum
    if v.size == 1:
        return x, float("inf")
    rest = np.delete(v, x)
    return x, float(v[x] - rest.max())
