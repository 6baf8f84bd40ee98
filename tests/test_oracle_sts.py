"""Pins of the STS fit oracle against facts the pages and the mathematics fix.

DSpark summary page, 방법론 › 신뢰도 기반 검증 (STS paragraph): left-to-right
temperature fits by 1-D grid search on ECE, order-preserving; 주요 결과: the raw
head is over-confident and STS lowers ECE.
"""
import numpy as np
import pytest

from oracle.sts import ece, sigmoid, sts_curves, sts_fit


def test_ece_hand_values():
    # bins of width 0.1: 0.05 -> bin 0, 0.15 -> bin 1, 0.95 -> bin 9
    assert ece([0.05, 0.15, 0.95], [0.0, 1.0, 1.0], 10) == pytest.approx((0.05 + 0.85 + 0.05) / 3,
                                                                          abs=1e-15)
    # two samples in one bin average before the absolute value:
    # bin 0 holds 0.1 and 0.4 (mean 0.25, labels mean 0.5), bin 1 holds 0.9 (exact)
    assert ece([0.1, 0.4, 0.9], [0.0, 1.0, 0.9], 2) == pytest.approx(2 / 3 * 0.25, abs=1e-15)
    # an exact bin edge goes up (floor), and 1.0 is clamped to the last bin
    assert ece([0.1, 1.0], [0.1, 0.0], 10) == pytest.approx(0.5, abs=1e-15)


def test_ece_single_bin_is_mean_gap():
    rng = np.random.default_rng(3)
    p, y = rng.uniform(size=500), rng.uniform(size=500)
    assert ece(p, y, 1) == pytest.approx(abs(p.mean() - y.mean()), abs=1e-14)


def test_ece_zero_for_perfect_labels_and_sample_order_free():
    rng = np.random.default_rng(4)
    p = rng.uniform(size=300)
    assert ece(p, p, 15) == 0.0
    y = rng.uniform(size=300)
    perm = rng.permutation(300)
    assert ece(p[perm], y[perm], 15) == pytest.approx(ece(p, y, 15), abs=1e-14)


def test_sigmoid_closed_forms():
    assert sigmoid(np.array([0.0]))[0] == 0.5
    x = np.linspace(-40, 40, 81)
    assert np.allclose(sigmoid(x) + sigmoid(-x), 1.0, atol=1e-15)
    assert np.allclose(sigmoid(np.log(np.array([3.0, 0.25]))), [0.75, 0.2], atol=1e-15)
    assert np.all(np.isfinite(sigmoid(np.array([-1e4, 1e4]))))


def _exact_labels(N, K, temps, seed):
    """Labels equal to the logistic law at the true temperatures: zero ECE there."""
    rng = np.random.default_rng(seed)
    a = rng.normal(1.5, 2.0, size=(N, K))
    y = sigmoid(a / np.asarray(temps)[None, :])
    return a, y


def test_fit_recovers_true_temperatures_with_zero_ece():
    grid = np.array([0.5, 0.8, 1.0, 1.3, 2.0, 3.0])
    t_true = [0.5, 1.3, 2.0, 0.8]
    a, y = _exact_labels(4000, 4, t_true, 11)
    fit = sts_fit(a, y, grid, 15)
    assert np.array_equal(fit["temps"], t_true)
    assert np.all(fit["ece"] < 1e-15)
    # every other grid point is strictly worse at every position
    for k, g in enumerate(fit["index"]):
        others = np.delete(fit["curves"][k], g)
        assert others.min() > 1e-4


def test_prefix_uses_earlier_fitted_temperatures():
    # With position 0 forced to a wrong temperature, position 1's curve no
    # longer has a zero at the true temperature: the prefix product enters.
    grid = np.array([0.5, 1.0, 2.0])
    a, y = _exact_labels(3000, 2, [2.0, 1.0], 5)
    good = sts_curves(a, y, grid, 15, [2.0, 1.0])
    bad = sts_curves(a, y, grid, 15, [0.5, 1.0])
    assert good[1, 1] < 1e-15
    assert bad[1].min() > 1e-3
    assert np.array_equal(good[0], bad[0])         # position 0 never sees temps[0]


def test_left_to_right_causality():
    rng = np.random.default_rng(8)
    a = rng.normal(1.0, 1.5, size=(2000, 5))
    y = rng.uniform(size=(2000, 5))
    grid = np.geomspace(0.2, 5.0, 40)
    base = sts_fit(a, y, grid, 10)
    a2, y2 = a.copy(), y.copy()
    a2[:, 3:] = rng.normal(-1.0, 3.0, size=(2000, 2))
    y2[:, 3:] = rng.uniform(size=(2000, 2))
    alt = sts_fit(a2, y2, grid, 10)
    assert np.array_equal(base["temps"][:3], alt["temps"][:3])


def test_overconfident_head_gets_temperature_above_one_and_lower_ece():
    grid = np.geomspace(0.25, 4.0, 64)
    grid = np.sort(np.append(grid, 1.0))
    rng = np.random.default_rng(21)
    a = rng.normal(2.0, 1.5, size=(5000, 3))
    y = sigmoid(a / 2.2 + rng.normal(0, 0.2, size=a.shape))
    fit = sts_fit(a, y, grid, 15)
    one = int(np.flatnonzero(grid == 1.0)[0])
    assert np.all(fit["temps"] > 1.0)
    assert np.all(fit["ece"] < fit["curves"][:, one])


def test_order_preserved_and_ties_take_first_grid_point():
    rng = np.random.default_rng(2)
    a = rng.normal(0, 2, size=(800, 1))
    for T in (0.3, 1.0, 4.0):
        s = sigmoid(a[:, 0] / T)
        assert np.array_equal(np.argsort(s, kind="stable"), np.argsort(a[:, 0], kind="stable"))
    y = sigmoid(a / 1.0)
    fit = sts_fit(a, y, np.array([2.0, 1.0, 1.0, 3.0]), 15)
    assert fit["index"][0] == 1
    with pytest.raises(ValueError):
        sts_fit(a, y, np.array([1.0, 0.0]), 15)


def test_generator_is_over_confident():
    from speculative_decoding_draft_block_gb300.workloads import make_sts_inputs, sts_grid
    d = make_sts_inputs(3000, 3, seed=9)
    assert d["logits"].dtype == np.float32 and d["labels"].dtype == np.float32
    assert np.all((d["labels"] >= 0) & (d["labels"] <= 1))
    fit = sts_fit(d["logits"], d["labels"], sts_grid(n=64), 15)
    assert np.all(fit["temps"] > 1.0)
