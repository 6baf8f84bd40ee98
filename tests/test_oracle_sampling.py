"""Pins for the oracle's inverse-CDF sampler and greedy choice (CPU only)."""
import numpy as np

from oracle import inverse_cdf, argmax_first, softmax_weights
from oracle.draft import draft_step
from tests._exact import outcome_measures


def test_hand_built_cdf_boundaries():
    w = [1.0, 1.0, 2.0, 4.0]          # C = 1, 2, 4, 8; S = 8 (all exact)
    assert inverse_cdf(w, 0.125 - 2.0 ** -40)[0] == 0
    assert inverse_cdf(w, 0.125)[0] == 1          # u*S == C_0 is not < C_0
    assert inverse_cdf(w, 0.25 - 2.0 ** -40)[0] == 1
    assert inverse_cdf(w, 0.25)[0] == 2
    assert inverse_cdf(w, 0.5)[0] == 3
    assert inverse_cdf(w, 1.0 - 2.0 ** -40)[0] == 3
    x, m = inverse_cdf(w, 0.375)                  # u*S = 3, inside [2, 4)
    assert x == 2 and abs(m - 1.0 / 8.0) < 1e-15


def test_zero_weight_never_drawn():
    w = [0.0, 1.0, 0.0, 0.0, 1.0, 0.0]
    meas = outcome_measures(lambda u: inverse_cdf(w, u)[0])
    assert set(meas) == {1, 4}
    assert abs(meas[1] - 0.5) < 1e-15 and abs(meas[4] - 0.5) < 1e-15


def test_draw_law_equals_normalised_weights():
    rng = np.random.default_rng(3)
    for _ in range(5):
        w = rng.exponential(size=13) * (rng.random(13) > 0.2)
        meas = outcome_measures(lambda u: inverse_cdf(w, u)[0])
        for i in range(13):
            assert abs(meas.get(i, 0.0) - w[i] / w.sum()) < 1e-14


def test_softmax_weights_scale_free():
    rng = np.random.default_rng(4)
    ell = rng.normal(0, 3, size=50)
    w1, s1 = softmax_weights(ell, 0.7)
    w2, s2 = softmax_weights(ell + 123.0, 0.7)
    np.testing.assert_allclose(w1 / s1, w2 / s2, rtol=1e-12)
    p = np.exp(ell / 0.7) / np.exp(ell / 0.7).sum()   # textbook softmax, small logits
    np.testing.assert_allclose(w1 / s1, p, rtol=1e-12)


def test_argmax_first_ties_and_gap():
    assert argmax_first([1.0, 3.0, 3.0, 2.0]) == (1, 0.0)
    x, g = argmax_first([0.5, -1.0, 2.5, 2.0])
    assert x == 2 and abs(g - 0.5) < 1e-15


def test_zero_temperature_limit_is_argmax():
    rng = np.random.default_rng(5)
    ell = rng.normal(0, 1, size=40)
    top = int(np.argmax(ell))
    meas = outcome_measures(lambda u: draft_step(ell, 1e-4, u)[0])
    assert meas.get(top, 0.0) > 1 - 1e-12
    assert draft_step(ell, 0.0, 0.3)[0] == top
