"""Lossless rejection-sampling verification, float64 (test infrastructure only).

DSpark summary page, 배경 (background): verification runs left to right over the
drafted tokens and accepts the longest prefix that agrees with the target; after
the first rejection every later token is discarded, and the rejection rule
preserves the target distribution exactly. The rule itself (standard
speculative sampling):

    accept x_k with probability min(1, p_k(x_k) / q_k(x_k))       (u*q < p)
    on the first rejection at k: y ~ normalize(max(0, p_k - q_k))
    if all L scheduled tokens pass: y ~ p_{L+1}   (the bonus token)

One uniform per decision: u = U(seed, request, k, 1) for the accept test at
position k, U(seed, request, k, 2) for the residual or bonus draw at position k.
The target has K+1 rows per request, one per drafted position plus the bonus
position (vLLM MTP/DFlash page, DFlashProposer 초기화: one bonus token plus K
drafted tokens per request). T = 0 reduces to exact-match greedy: accept iff
x_k = argmax p_k, emit argmax on the first mismatch or at the bonus position.
"""

import numpy as np

from .bf16 import as_f64
from .draft import markov_logits
from .philox import uniform, STAGE_ACCEPT, STAGE_RESAMPLE
from .sampling import inverse_cdf, argmax_first, softmax_weights


def _probs(logits, temperature):
    w, s = softmax_weights(logits, temperature)
    return w / s


def verify_request(tokens, L, p_row, q_row, u_accept, u_resample, greedy=False):
    """Verify one request's first L drafted tokens.

    tokens: drafted tokens x_1..x_K (index j holds position j+1).
    p_row(j): target probabilities at position j+1 (target logits if greedy).
    q_row(j): draft probabilities at position j+1 (unused if greedy).
    u_accept(j), u_resample(j): the uniforms of position j+1.

    Returns (accepted, emitted_tokens, decisions) where decisions lists, per
    decision taken, (kind, margin): kind is "accept", "argmax", "residual" or
    "bonus"; the margin is |u - p/q| for accept tests, the top-1/top-2 logit
    gap for greedy choices and the inverse-CDF margin for draws.
    """
    decisions = []
    accepted = 0
    for j in range(L):
        x = int(tokens[j])
        if greedy:
            y, gap = argmax_first(p_row(j))
            decisions.append(("argmax", gap))
            ok = x == y
        else:
            p, q = p_row(j)[x], q_row(j)[x]
            u = u_accept(j)
            ok = u * q < p
            decisions.append(("accept", abs(u - p / q) if q > 0 else np.inf))
        if not ok:
            break
        accepted += 1
    j = accepted
    if greedy:
        y, gap = argmax_first(p_row(j))
        decisions.append(("argmax", gap))
    elif accepted < L:
        residual = np.maximum(0.0, p_row(j) - q_row(j))
        y, m = inverse_cdf(residual, u_resample(j))
        decisions.append(("residual", m))
    else:
        y, m = inverse_cdf(p_row(j), u_resample(j))
        decisions.append(("bonus", m))
    return accepted, [int(t) for t in tokens[:accepted]] + [int(y)], decisions


def verify(target_logits, base_logits, E, P, anchor, tokens, sched_len, temperature, seed,
           request_ids=None, states=None, with_p=False):
    """Verify a batch. target_logits: [B, K+1, V]; base_logits: [B, K, V].

    The draft distribution q_k is recomputed from the base logits and the Markov
    bias of the drafted prefix (x_0 = anchor), exactly as the draft defined it.

    ``request_ids`` (optional [B]) gives each row's request index in the Philox
    counter when the rows are a subset of a larger batch.

    ``states`` (optional [B, K, r]) selects the RNN head: q_k is then rebuilt
    from the base logits and the bias s_k . P of the state the draft used at
    that position, exactly as the RNN draft defined it.

    ``with_p`` adds ``p_token`` [B, K]: the target probability p_k(x_k) of
    every scheduled drafted token (k <= L_b, whether or not an earlier position
    rejected; NaN beyond L_b). For a greedy request (T = 0) the target law is
    the point mass on its argmax, so p_k(x_k) is 1 if x_k is the argmax and 0
    otherwise. The accept rule reads exactly this p_k(x_k).

    Returns a dict with accept_count [B], num_emitted [B], out_tokens [B, K+1]
    (-1 padded) and decisions (per request, see verify_request).
    """
    B, K1, V = target_logits.shape
    K = K1 - 1
    tokens = np.asarray(tokens, dtype=np.int64)
    anchor = np.asarray(anchor, dtype=np.int64)
    temperature = np.asarray(temperature, dtype=np.float32)
    out = -np.ones((B, K + 1), dtype=np.int64)
    acc = np.zeros(B, dtype=np.int64)
    p_token = np.full((B, K), np.nan)
    decisions = []
    rid = np.arange(B) if request_ids is None else np.asarray(request_ids, dtype=np.int64)
    for b in range(B):
        T = float(temperature[b])
        greedy = T == 0
        L = int(sched_len[b])
        if not 0 <= L <= K:
            raise ValueError("scheduled length out of range")

        def p_row(j, b=b, T=T, greedy=greedy):
            row = as_f64(target_logits[b, j])
            return row if greedy else _probs(row, T)

        def q_row(j, b=b, T=T):
            if states is not None:
                ell = as_f64(base_logits[b, j]) + as_f64(states[b, j]) @ as_f64(P)
                return _probs(ell, T)
            prev = anchor[b] if j == 0 else tokens[b, j - 1]
            ell = markov_logits(np.asarray(base_logits[b, j])[None, :], E, P, [prev])[0]
            return _probs(ell, T)

        a, emitted, dec = verify_request(
            tokens[b], L, p_row, q_row,
            lambda j, b=b: uniform(seed, int(rid[b]), j + 1, STAGE_ACCEPT),
            lambda j, b=b: uniform(seed, int(rid[b]), j + 1, STAGE_RESAMPLE),
            greedy=greedy)
        acc[b] = a
        out[b, :len(emitted)] = emitted
        decisions.append(dec)
        if with_p:
            for j in range(L):
                x = int(tokens[b, j])
                if greedy:
                    p_token[b, j] = 1.0 if argmax_first(p_row(j))[0] == x else 0.0
                else:
                    p_token[b, j] = p_row(j)[x]
    res = {"accept_count": acc, "num_emitted": acc + 1, "out_tokens": out,
           "decisions": decisions}
    if with_p:
        res["p_token"] = p_token
    return res
