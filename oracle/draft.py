"""Markov-head draft block, float64 (test infrastructure only).

DSpark summary page, 방법론 › 반자기회귀 생성 (semi-autoregressive generation):
a parallel backbone gives base logits z_k for every block position in one pass;
a sequential head then adds a prefix-dependent transition bias so that each
position is conditioned on the token sampled just before it. The Markov head
restricts that bias to a first-order transition, a V x V matrix in principle,
factored at low rank r into an embedding lookup E (V x r) and a projection
P (r x V):

    l_k = z_k + E[x_{k-1}] . P,      x_0 = the anchor (the last verified token),
    x_k ~ softmax(l_k / T)           (T = 0: greedy, lowest index on ties)

The loop is sequential over k. The anchor is the first prediction position
(same section), so x_0 is an input. Temperature divides the full logit (base
plus bias): the same T is used for draft and target, since verification must
preserve the target's own sampling law (background section, 배경).
"""

import numpy as np

from .bf16 import as_f64
from .philox import uniform, STAGE_DRAFT
from .sampling import inverse_cdf, argmax_first, softmax_weights


def markov_logits(z_rows, E, P, prev_tokens):
    """Rows of l = z + E[x_prev] . P in float64 (the matmul is a library step)."""
    z = as_f64(z_rows)
    e_rows = as_f64(E)[np.asarray(prev_tokens, dtype=np.int64)]
    return z + e_rows @ as_f64(P)


def draft_distribution(z_row, E, P, prev_token, temperature):
    """Draft probabilities q(. | x_prev) of one position, float64 (T > 0)."""
    ell = markov_logits(np.asarray(z_row)[None, :], E, P, [prev_token])[0]
    w, s = softmax_weights(ell, temperature)
    return w / s


def draft_step(ell_row, temperature, u):
    """One draw from one position's logits.

    Returns (token, q(token), margin). For T > 0 the draw is the inverse CDF of
    softmax(l/T) at u and the margin is in probability units; for T = 0 the
    token is the argmax, q = 1, and the margin is the top-1 / top-2 logit gap.
    """
    if temperature == 0:
        x, gap = argmax_first(ell_row)
        return x, 1.0, gap
    w, s = softmax_weights(ell_row, temperature)
    x, margin = inverse_cdf(w, u)
    return x, float(w[x] / s), margin


def draft_block(base_logits, E, P, anchor, temperature, seed, prev_tokens=None, request_ids=None):
    """Sample a whole draft block, position by position.

    base_logits: [B, K, V] (bfloat16 bits or floats); E: [V, r]; P: [r, V];
    anchor: [B]; temperature: [B]; seed: the Philox key.

    ``prev_tokens`` (optional [B, K]) teacher-forces the conditioning token of
    every position: position k then uses prev_tokens[:, k-2] (the anchor for
    k = 1) instead of the oracle's own previous draw, so each draw can be
    compared on its own against another implementation's prefix.

    ``request_ids`` (optional [B]) gives each row's request index in the Philox
    counter when the rows are a subset of a larger batch (default: 0..B-1).

    Returns a dict with tokens [B, K] (int64), q_token [B, K] (float64),
    margin [B, K] and greedy [B] (bool).
    """
    B, K, _ = base_logits.shape
    anchor = np.asarray(anchor, dtype=np.int64)
    temperature = np.asarray(temperature, dtype=np.float32)
    tokens = np.zeros((B, K), dtype=np.int64)
    q_token = np.zeros((B, K), dtype=np.float64)
    margin = np.zeros((B, K), dtype=np.float64)
    rid = np.arange(B) if request_ids is None else np.asarray(request_ids, dtype=np.int64)
    prev = anchor.copy()
    for k in range(K):
        if prev_tokens is not None and k > 0:
            prev = np.asarray(prev_tokens, dtype=np.int64)[:, k - 1]
        ell = markov_logits(base_logits[:, k, :], E, P, prev)
        for b in range(B):
            u = uniform(seed, int(rid[b]), k + 1, STAGE_DRAFT)
            x, q, m = draft_step(ell[b], float(temperature[b]), u)
            tokens[b, k] = x
            q_token[b, k] = q
            margin[b, k] = m
        prev = tokens[:, k].copy()
    return {"tokens": tokens, "q_token": q_token, "margin": margin,
            "greedy": temperature == 0}
