"""Pins for the oracle's analytic acceptance rate (CPU only).

The rate is pinned against the verify oracle's own accept rule: for every
drafted token x the measure of {u : verify accepts x} is computed exactly
(tests/_exact.py integrates over u piecewise), weighted by q(x) and summed.
That path never forms min(p, q), so a wrong temperature, a swapped operand or
a missing normalisation in acceptance_rate shows up as a mismatch."""
import numpy as np

from oracle import acceptance_rate, verify_request
from oracle.sampling import softmax_weights
from tests._exact import outcome_measures


def _accept_measure(p, q, x):
    meas = outcome_measures(lambda u: verify_request([x], 1, lambda j: p, lambda j: q,
                                                     lambda j: u, lambda j: 0.5)[0])
    return meas.get(1, 0.0)


def test_equals_the_verify_rule_integrated_over_u():
    rng = np.random.default_rng(3)
    for T in (1.0, 0.6, 1.7):
        V = 10
        t = rng.normal(0, 1.5, size=(1, V))
        d = t + rng.normal(0, 0.8, size=(1, V))
        wp, sp = softmax_weights(t[0], T)
        wq, sq = softmax_weights(d[0], T)
        p, q = wp / sp, wq / sq
        want = sum(q[x] * _accept_measure(p, q, x) for x in range(V))
        got = acceptance_rate(t, d, [T])[0]
        assert abs(got - want) < 1e-13, (T, got, want)


def test_special_cases():
    rng = np.random.default_rng(4)
    t = rng.normal(size=(3, 16))
    # identical rows: always accepted
    assert np.allclose(acceptance_rate(t, t, [1.0, 0.5, 2.0]), 1.0, atol=1e-14)
    # disjoint supports (the rest at -inf): never accepted
    a = np.full((1, 8), -np.inf)
    b = np.full((1, 8), -np.inf)
    a[0, :4] = 0.0
    b[0, 4:] = 0.0
    assert acceptance_rate(a, b, [1.0])[0] == 0.0
    # two-token closed form: p = (0.75, 0.25), q = (0.5, 0.5) -> 0.75
    t2 = np.array([[np.log(3.0), 0.0]])
    d2 = np.zeros((1, 2))
    assert abs(acceptance_rate(t2, d2, [1.0])[0] - 0.75) < 1e-15
    # temperature applies to both rows: T = 2 on logits 2 ln 3, 0 is the same law
    assert abs(acceptance_rate(2 * t2, d2, [2.0])[0] - 0.75) < 1e-15


def test_greedy_rows_compare_argmaxes():
    t = np.array([[0.0, 2.0, 2.0, 1.0], [5.0, 0.0, 0.0, 0.0]])
    d = np.array([[0.0, 3.0, 1.0, 3.0], [0.0, 5.0, 0.0, 0.0]])
    # row 0: both first argmax is index 1 (ties go to the lowest index); row 1 differs
    assert acceptance_rate(t, d, [0.0, 0.0]).tolist() == [1.0, 0.0]
