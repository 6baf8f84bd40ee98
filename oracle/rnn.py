"""RNN-head draft block, float64 (test infrastructure only).

DSpark summary page, 방법론 › 반자기회귀 생성: the second sequential head keeps
a recurrent state that accumulates the whole prefix drafted so far inside the
block, where the Markov head sees only the previous token. At every step it
combines the current state, the previous token's embedding and the backbone
hidden state through a gated update. 주요 결과 (proposal-length experiment):
it adds only a small gain over the Markov head at long proposals, and the
Markov head is the default.

Readings where the pages leave the head open:
  * the gated update is a GRU cell in the form cuDNN and PyTorch use (the
    reset gate scales the recurrent product), with gate rows in the order
    reset, update, new:
        g_i = W_ih [e ; h] + b_ih,      g_h = W_hh s + b_hh
        r = sigmoid(g_i^r + g_h^r),     u = sigmoid(g_i^u + g_h^u)
        n = tanh(g_i^n + r * g_h^n),    s' = (1 - u) * n + u * s
  * the state has the Markov rank r as its size and goes through the same
    logit projection P:  l_k = z_k + s_k . P;
  * s_0 = 0; step k reads e = E[x_{k-1}] (x_0 = the anchor) and h = h_k;
  * the state is kept in the model's storage type: with bfloat16 weights it is
    rounded to bfloat16 (nearest even) after every step.
The draw itself is the Markov head's: softmax(l_k / T) by inverse CDF with the
same Philox stream, greedy argmax at T = 0.
"""

import numpy as np

from .bf16 import as_f64, round_bf16
from .draft import draft_step
from .philox import uniform, STAGE_DRAFT


def _sigmoid(x):
    x = np.asarray(x, dtype=np.float64)
    out = np.empty_like(x)
    pos = x >= 0
    out[pos] = 1.0 / (1.0 + np.exp(-x[pos]))
    e = np.exp(x[~pos])
    out[~pos] = e / (1.0 + e)
    return out


def gru_cell(x, s, W_ih, W_hh, b_ih, b_hh):
    """One gated update, float64. x: [..., n_in]; s: [..., r]; W_ih: [3r, n_in];
    W_hh: [3r, r]; b_ih, b_hh: [3r]. Returns s' [..., r]."""
    x = as_f64(x)
    s = as_f64(s)
    W_ih = as_f64(W_ih)
    W_hh = as_f64(W_hh)
    r = s.shape[-1]
    gi = x @ W_ih.T + as_f64(b_ih)
    gh = s @ W_hh.T + as_f64(b_hh)
    reset = _sigmoid(gi[..., :r] + gh[..., :r])
    update = _sigmoid(gi[..., r:2 * r] + gh[..., r:2 * r])
    new = np.tanh(gi[..., 2 * r:] + reset * gh[..., 2 * r:])
    return (1.0 - update) * new + update * s


def rnn_draft_block(base_logits, E, P, anchor, temperature, seed, h, W_ih, W_hh, b_ih, b_hh,
                    bf16_state, prev_tokens=None, prev_states=None, request_ids=None):
    """Sample a whole draft block with the RNN head, position by position.

    base_logits: [B, K, V]; E: [V, r]; P: [r, V]; anchor, temperature: [B];
    h: [B, K, d]; W_ih: [3r, r + d]; W_hh: [3r, r]; b_ih, b_hh: [3r].

    Teacher forcing, for comparison with another implementation:
      ``prev_tokens`` [B, K]: step k conditions on prev_tokens[:, k-2] (the
      anchor for k = 1) instead of the oracle's own draw;
      ``prev_states`` [B, K, r]: step k updates from prev_states[:, k-2]
      (zero for k = 1) and draws with prev_states[:, k-1], so that each state
      and each draw can be checked on its own.

    Returns a dict: tokens [B, K], q_token [B, K], margin [B, K], states
    [B, K, r] (the oracle's own stored state of every position, after the
    storage rounding), states_pre [B, K, r] (before it) and greedy [B].
    """
    base = base_logits
    B, K, V = base.shape
    Ef = as_f64(E)
    Pf = as_f64(P)
    hf = as_f64(h)
    r = Ef.shape[1]
    anchor = np.asarray(anchor, dtype=np.int64)
    temperature = np.asarray(temperature, dtype=np.float32)
    rid = np.arange(B) if request_ids is None else np.asarray(request_ids, dtype=np.int64)
    tokens = np.zeros((B, K), dtype=np.int64)
    q_token = np.zeros((B, K))
    margin = np.zeros((B, K))
    states = np.zeros((B, K, r))
    states_pre = np.zeros((B, K, r))
    s = np.zeros((B, r))
    prev = anchor.copy()
    for k in range(K):
        if k > 0:
            if prev_tokens is not None:
                prev = np.asarray(prev_tokens, dtype=np.int64)[:, k - 1]
            if prev_states is not None:
                s = as_f64(prev_states[:, k - 1])
        x_in = np.concatenate([Ef[prev], hf[:, k, :]], axis=1)
        pre = gru_cell(x_in, s, W_ih, W_hh, b_ih, b_hh)
        stored = round_bf16(pre) if bf16_state else pre
        states_pre[:, k] = pre
        states[:, k] = stored
        s_draw = as_f64(prev_states[:, k]) if prev_states is not None else stored
        ell = as_f64(base[:, k, :]) + s_draw @ Pf
        for b in range(B):
            u = uniform(seed, int(rid[b]), k + 1, STAGE_DRAFT)
            x, q, m = draft_step(ell[b], float(temperature[b]), u)
            tokens[b, k] = x
            q_token[b, k] = q
            margin[b, k] = m
        s = stored
        prev = tokens[:, k].copy()
    return {"tokens": tokens, "q_token": q_token, "margin": margin, "states": states,
            "states_pre": states_pre, "greedy": temperature == 0}
