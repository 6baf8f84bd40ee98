"""Analytic per-position acceptance rate, float64 (test infrastructure only).

DSpark summary page, 방법론 › 신뢰도 기반 검증 (the STS paragraph): the STS
temperatures are fitted against the analytic probability that a drafted
position passes verification, 1 - TV(p_k, q_k). Under the accept rule of the
배경 section (accept x ~ q_k with probability min(1, p_k(x) / q_k(x))) that
probability is

    alpha_k = sum_x q_k(x) min(1, p_k(x) / q_k(x)) = sum_x min(p_k(x), q_k(x)),

one minus the total-variation distance between the target distribution p_k =
softmax(target_k / T) and the draft distribution q_k = softmax(draft_k / T).

Reading where the pages leave it open: the temperature is the request's
sampling temperature, applied to both rows as the verifier applies it; at
T = 0 both laws are point masses on their argmax (lowest index on ties), so
alpha is 1 when the argmaxes agree and 0 otherwise (the greedy exact-match
rule).
"""

import numpy as np

from .bf16 import as_f64
from .sampling import softmax_weights, argmax_first


def acceptance_rate(target_logits, draft_logits, temperature):
    """alpha[n] = sum_i min(p_n(i), q_n(i)) for rows n of [n, V] logits (float64)."""
    t = as_f64(target_logits)
    d = as_f64(draft_logits)
    temperature = np.asarray(temperature, dtype=np.float64)
    n = t.shape[0]
    out = np.empty(n)
    for i in range(n):
        T = float(temperature[i])
        if T == 0.0:
            out[i] = 1.0 if argmax_first(t[i])[0] == argmax_first(d[i])[0] else 0.0
            continue
        wp, sp = softmax_weights(t[i], T)
        wq, sq = softmax_weights(d[i], T)
        out[i] = float(np.minimum(wp / sp, wq / sq).sum())
    return out
