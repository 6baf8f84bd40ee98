"""Confidence head, STS temperatures and survival, float64 (test infrastructure only).

DSpark summary page, 방법론 › 신뢰도 기반 검증 (confidence-scheduled verification):
the confidence head is a light linear projection plus a sigmoid over the
backbone hidden state h_k and the Markov embedding of the previous draft token.
Its output models the probability that position k passes verification given
that every earlier position passed. Sequential Temperature Scaling (STS) divides
each position's confidence logit by its own temperature T_k (order-preserving),
and the survival of a prefix is the cumulative product of the confidences:

    c_k = sigmoid((w_h . h_k + w_e . E[x_{k-1}] + b) / T_k),   x_0 = anchor
    s_k = c_1 * c_2 * ... * c_k
"""

import numpy as np

from .bf16 import as_f64


def confidence(h, E, anchor, tokens, w_h, w_e, bias, sts_temp):
    """Per-position confidences c [B, K] in float64.

    h: [B, K, d]; E: [V, r]; anchor: [B]; tokens: [B, K] draft tokens;
    w_h: [d]; w_e: [r]; bias: scalar b; sts_temp: [K] per-position temperatures.
    """
    hf = as_f64(h)
    B, K, _ = hf.shape
    tokens = np.asarray(tokens, dtype=np.int64)
    prev = np.concatenate([np.asarray(anchor, dtype=np.int64)[:, None], tokens[:, :K - 1]], axis=1)
    head = hf @ as_f64(w_h)                                 # [B, K]
    markov = as_f64(E)[prev] @ as_f64(w_e)                  # [B, K]
    logit = (head + markov + np.float64(bias)) / np.asarray(sts_temp, dtype=np.float64)[None, :]
    return 1.0 / (1.0 + np.exp(-logit))


def survival(c):
    """Prefix survival s_k = prod_{j <= k} c_j along each request's block."""
    return np.cumprod(np.asarray(c, dtype=np.float64), axis=1)
