"""Pins for the oracle's Markov head and draft block (CPU only)."""
import math

import numpy as np

from oracle import markov_logits, draft_block, uniform
from oracle.draft import draft_step
from oracle.philox import STAGE_DRAFT
from tests._exact import outcome_measures


def test_full_rank_head_is_an_explicit_transition_matrix():
    """r = V, E = I, P = M: the factored bias must reproduce row M[x_prev] exactly."""
    rng = np.random.default_rng(0)
    V = 12
    M = rng.normal(size=(V, V))
    z = rng.normal(size=(V, V))
    prev = rng.integers(0, V, size=V)
    ell = markov_logits(z, np.eye(V), M, prev)
    for i in range(V):
        assert np.array_equal(ell[i], z[i] + M[prev[i]])


def test_toy_of_course_no_problem():
    """Two plausible continuations; independent positions would mix them.

    Vocabulary: 0 "of", 1 "course", 2 "no", 3 "problem". Position 1 favours
    "of" and "no" equally, position 2 favours "course" and "problem" equally.
    A full-rank Markov head that lifts "course" after "of" and "problem" after
    "no" (and suppresses the crossed pairs) must make "of problem" rare.
    """
    V = 4
    z = np.array([[2.0, -8.0, 2.0, -8.0],       # position 1
                  [-8.0, 2.0, -8.0, 2.0]])      # position 2
    M = np.zeros((V, V))
    M[0, 1], M[0, 3] = 4.0, -4.0                # after "of"
    M[2, 3], M[2, 1] = 4.0, -4.0                # after "no"
    anchor = 3                                  # a row of M that is all zero
    # exact per-position laws measured over u
    law1 = outcome_measures(lambda u: draft_step(markov_logits(z[:1], np.eye(V), M, [anchor])[0], 1.0, u)[0])
    law2_of = outcome_measures(lambda u: draft_step(markov_logits(z[1:], np.eye(V), M, [0])[0], 1.0, u)[0])
    law2_no = outcome_measures(lambda u: draft_step(markov_logits(z[1:], np.eye(V), M, [2])[0], 1.0, u)[0])
    e = math.exp
    den1 = 2 * e(2.0) + 2 * e(-8.0)
    assert abs(law1[0] - e(2.0) / den1) < 1e-14
    den_of = e(6.0) + e(-2.0) + 2 * e(-8.0)
    assert abs(law2_of[1] - e(6.0) / den_of) < 1e-14         # P(course | of)
    assert abs(law2_of.get(3, 0.0) - e(-2.0) / den_of) < 1e-14  # P(problem | of)
    p_of_problem = law1[0] * law2_of.get(3, 0.0)
    assert p_of_problem < 2e-4                   # independent positions would give ~0.25
    assert law2_no[3] > 0.999


def test_draft_block_teacher_forcing_and_rng_keys():
    rng = np.random.default_rng(1)
    B, K, V, r = 3, 4, 16, 4
    base = rng.normal(size=(B, K, V))
    E = rng.normal(size=(V, r))
    P = rng.normal(size=(r, V))
    anchor = np.array([1, 2, 3])
    T = np.array([1.0, 0.5, 0.0], dtype=np.float32)
    out = draft_block(base, E, P, anchor, T, 99)
    # re-derive every draw from its own uniform (b, k, stage 0) and conditioning token
    for b in range(B):
        prev = anchor[b]
        for k in range(K):
            ell = base[b, k] + E[prev] @ P
            x, q, _ = draft_step(ell, float(T[b]), uniform(99, b, k + 1, STAGE_DRAFT))
            assert x == out["tokens"][b, k]
            prev = x
    # teacher forcing with the oracle's own tokens changes nothing
    tf = draft_block(base, E, P, anchor, T, 99, prev_tokens=out["tokens"])
    assert np.array_equal(tf["tokens"], out["tokens"])
    assert np.array_equal(tf["q_token"], out["q_token"])
    assert np.all(out["q_token"][2] == 1.0)      # greedy request


def test_block_law_is_the_markov_chain():
    """Exact law of a 2-position block = product of the chain's conditionals."""
    rng = np.random.default_rng(2)
    V, r = 5, 3
    z = rng.normal(size=(2, V))
    E = rng.normal(size=(V, r))
    P = rng.normal(size=(r, V))
    a = 4
    law1 = outcome_measures(lambda u: draft_step(markov_logits(z[:1], E, P, [a])[0], 1.0, u)[0])
    for x1 in range(V):
        q1 = np.exp(z[0] + E[a] @ P); q1 /= q1.sum()
        assert abs(law1.get(x1, 0.0) - q1[x1]) < 1e-14
        law2 = outcome_measures(lambda u: draft_step(markov_logits(z[1:], E, P, [x1])[0], 1.0, u)[0])
        q2 = np.exp(z[1] + E[x1] @ P); q2 /= q2.sum()
        for x2 in range(V):
            assert abs(law2.get(x2, 0.0) - q2[x2]) < 1e-14
