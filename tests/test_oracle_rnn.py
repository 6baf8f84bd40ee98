"""Pins of the RNN-head oracle against facts the pages, the mathematics and an
independent library fix.

DSpark summary page, 방법론 › 반자기회귀 생성: the RNN head keeps a recurrent
state over the whole drafted prefix and applies a gated update to the state,
the previous token's embedding and the backbone hidden state.
"""
import numpy as np
import pytest

from oracle.bf16 import bf16_tie_distance, round_bf16
from oracle.rnn import gru_cell, rnn_draft_block
from oracle.sampling import inverse_cdf, softmax_weights
from oracle.philox import uniform, STAGE_DRAFT


def _weights(rng, r, n_in, scale=0.3):
    return (rng.normal(0, scale, (3 * r, n_in)), rng.normal(0, scale, (3 * r, r)),
            rng.normal(0, 0.2, 3 * r), rng.normal(0, 0.2, 3 * r))


def test_gru_cell_matches_torch_float64():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    r, n_in, n = 12, 20, 7
    W_ih, W_hh, b_ih, b_hh = _weights(rng, r, n_in)
    x = rng.normal(size=(n, n_in))
    s = np.tanh(rng.normal(size=(n, r)))
    cell = torch.nn.GRUCell(n_in, r).double()
    with torch.no_grad():
        cell.weight_ih.copy_(torch.from_numpy(W_ih))
        cell.weight_hh.copy_(torch.from_numpy(W_hh))
        cell.bias_ih.copy_(torch.from_numpy(b_ih))
        cell.bias_hh.copy_(torch.from_numpy(b_hh))
        want = cell(torch.from_numpy(x), torch.from_numpy(s)).numpy()
    assert np.allclose(gru_cell(x, s, W_ih, W_hh, b_ih, b_hh), want, rtol=0, atol=1e-14)


def test_gru_cell_closed_forms():
    rng = np.random.default_rng(1)
    r, n_in = 5, 9
    s = np.tanh(rng.normal(size=(3, r)))
    x = rng.normal(size=(3, n_in))
    Z = np.zeros
    # all weights and biases zero: reset = update = 1/2, new = tanh(0) = 0
    assert np.array_equal(gru_cell(x, s, Z((3 * r, n_in)), Z((3 * r, r)), Z(3 * r), Z(3 * r)), 0.5 * s)
    # update gate saturated open: the state is carried unchanged
    W_ih, W_hh, b_ih, b_hh = _weights(rng, r, n_in)
    b_hh = b_hh.copy()
    b_hh[r:2 * r] = 60.0
    assert np.array_equal(gru_cell(x, s, W_ih, W_hh, b_ih, b_hh), s)
    # update gate saturated shut, recurrent weights zero: s' = tanh(W_in x + b_in + r * b_hn)
    W_ih, W_hh, b_ih, b_hh = _weights(rng, r, n_in)
    b_hh = b_hh.copy()
    b_hh[r:2 * r] = -60.0
    W_hh = np.zeros_like(W_hh)
    reset = 1 / (1 + np.exp(-(x @ W_ih[:r].T + b_ih[:r] + b_hh[:r])))
    want = np.tanh(x @ W_ih[2 * r:].T + b_ih[2 * r:] + reset * b_hh[2 * r:])
    assert np.allclose(gru_cell(x, s, W_ih, W_hh, b_ih, b_hh), want, rtol=0, atol=1e-15)


def _case(rng, B=3, K=4, V=11, r=6, d=5):
    return dict(base_logits=rng.normal(0, 1.5, (B, K, V)), E=rng.normal(0, 0.6, (V, r)),
                P=rng.normal(0, 0.6, (r, V)), anchor=rng.integers(0, V, B),
                temperature=np.array([1.0, 0.7, 0.0][:B], dtype=np.float32),
                h=rng.normal(size=(B, K, d)))


def test_frozen_zero_state_draws_from_base_logits_alone():
    rng = np.random.default_rng(2)
    c = _case(rng)
    r, d = c["E"].shape[1], c["h"].shape[2]
    W_ih, W_hh, b_ih, b_hh = _weights(rng, r, r + d)
    b_hh[r:2 * r] = 60.0                    # the state never leaves s_0 = 0
    seed = 0xABCDEF
    out = rnn_draft_block(**c, seed=seed, W_ih=W_ih, W_hh=W_hh, b_ih=b_ih, b_hh=b_hh, bf16_state=False)
    assert np.all(out["states"] == 0.0)
    for b in range(3):
        for k in range(4):
            T = float(c["temperature"][b])
            z = c["base_logits"][b, k]
            if T == 0:
                assert out["tokens"][b, k] == int(np.argmax(z))
            else:
                w, _ = softmax_weights(z, T)
                x, _ = inverse_cdf(w, uniform(seed, b, k + 1, STAGE_DRAFT))
                assert out["tokens"][b, k] == x


def test_state_remembers_more_than_the_previous_token():
    rng = np.random.default_rng(3)
    c = _case(rng, B=1, K=3)
    r, d = c["E"].shape[1], c["h"].shape[2]
    W = _weights(rng, r, r + d)
    a = np.array([[2, 5, 0]])
    b = np.array([[7, 5, 0]])               # differs only two steps before position 3
    oa = rnn_draft_block(**c, seed=1, W_ih=W[0], W_hh=W[1], b_ih=W[2], b_hh=W[3], bf16_state=False,
                         prev_tokens=a)
    ob = rnn_draft_block(**c, seed=1, W_ih=W[0], W_hh=W[1], b_ih=W[2], b_hh=W[3], bf16_state=False,
                         prev_tokens=b)
    assert not np.allclose(oa["states_pre"][0, 1], ob["states_pre"][0, 1])   # s_2 reads x_1
    assert not np.allclose(oa["states_pre"][0, 2], ob["states_pre"][0, 2])   # x_1 still matters
    assert np.array_equal(oa["states_pre"][0, 0], ob["states_pre"][0, 0])    # s_1 sees only x_0


def test_states_bounded_and_teacher_forcing_is_identity():
    rng = np.random.default_rng(4)
    c = _case(rng)
    r, d = c["E"].shape[1], c["h"].shape[2]
    W = _weights(rng, r, r + d, scale=1.5)
    kw = dict(W_ih=W[0], W_hh=W[1], b_ih=W[2], b_hh=W[3], bf16_state=True)
    own = rnn_draft_block(**c, seed=9, **kw)
    assert np.all(np.abs(own["states"]) <= 1.0)
    forced = rnn_draft_block(**c, seed=9, prev_tokens=own["tokens"], prev_states=own["states"], **kw)
    for key in ("tokens", "q_token", "states", "states_pre"):
        assert np.array_equal(own[key], forced[key]), key
    assert np.array_equal(own["states"], round_bf16(own["states_pre"]))


def test_round_bf16_against_generator_rounding():
    from speculative_decoding_draft_block_gb300.workloads import to_bf16_bits
    from oracle.bf16 import bf16_bits_to_f64
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.normal(0, 1, 20000), rng.normal(0, 1e-3, 2000),
                        rng.normal(0, 100, 2000)]).astype(np.float32)
    assert np.array_equal(round_bf16(x.astype(np.float64)), bf16_bits_to_f64(to_bf16_bits(x)))
    # ties go to the even neighbour
    assert round_bf16(1 + 2.0 ** -8) == 1.0
    assert round_bf16(1 + 3 * 2.0 ** -8) == 1 + 2.0 ** -6
    assert round_bf16(-(1 + 3 * 2.0 ** -8)) == -(1 + 2.0 ** -6)
    assert round_bf16(0.0) == 0.0
    assert bf16_tie_distance(1 + 2.0 ** -8) == 0.0
    assert bf16_tie_distance(1.0) == pytest.approx(0.5 / 128)


def test_verify_with_states_reduces_to_markov_when_states_are_embeddings():
    import oracle
    rng = np.random.default_rng(6)
    B, K, V, r = 4, 3, 9, 5
    base = rng.normal(0, 1.2, (B, K, V))
    target = rng.normal(0, 1.2, (B, K + 1, V))
    E = rng.normal(0, 0.5, (V, r))
    P = rng.normal(0, 0.5, (r, V))
    anchor = rng.integers(0, V, B)
    tokens = rng.integers(0, V, (B, K))
    T = np.array([1.0, 0.8, 1.3, 1.0], dtype=np.float32)
    L = np.array([3, 2, 1, 3])
    prev = np.concatenate([anchor[:, None], tokens[:, :-1]], axis=1)
    states = E[prev]                          # the Markov head's A rows as "states"
    a = oracle.verify(target, base, E, P, anchor, tokens, L, T, 77)
    b = oracle.verify(target, base, E, P, anchor, tokens, L, T, 77, states=states)
    assert np.array_equal(a["out_tokens"], b["out_tokens"])
    assert np.array_equal(a["accept_count"], b["accept_count"])
