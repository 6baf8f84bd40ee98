"""Pins for the oracle's confidence head, STS and survival (CPU only)."""
import math

import numpy as np

from oracle import confidence, survival


def _setup(seed=0, B=4, K=5, V=20, r=6, d=8):
    rng = np.random.default_rng(seed)
    return dict(h=rng.normal(size=(B, K, d)), E=rng.normal(size=(V, r)),
                anchor=rng.integers(0, V, size=B), tokens=rng.integers(0, V, size=(B, K)),
                w_h=rng.normal(size=d), w_e=rng.normal(size=r))


def test_sigmoid_closed_form_points():
    a = _setup()
    a["w_h"][:] = 0.0
    a["w_e"][:] = 0.0
    K = a["h"].shape[1]
    c = confidence(bias=0.0, sts_temp=np.ones(K), **a)
    assert np.all(c == 0.5)
    c = confidence(bias=math.log(3.0), sts_temp=np.ones(K), **a)
    np.testing.assert_allclose(c, 0.75, rtol=1e-15)
    c = confidence(bias=math.log(3.0), sts_temp=np.full(K, 2.0), **a)   # sigmoid(ln3 / 2) = sqrt3/(1+sqrt3)
    np.testing.assert_allclose(c, math.sqrt(3.0) / (1.0 + math.sqrt(3.0)), rtol=1e-15)


def test_uses_previous_token_embedding():
    """Position k reads E[x_{k-1}] (anchor for k = 1), never E[x_k]."""
    a = _setup(1)
    a["w_h"][:] = 0.0
    K = a["h"].shape[1]
    c = confidence(bias=0.0, sts_temp=np.ones(K), **a)
    E, w_e = a["E"], a["w_e"]
    b = 2
    assert abs(c[b, 0] - 1 / (1 + math.exp(-(E[a["anchor"][b]] @ w_e)))) < 1e-15
    for k in range(1, K):
        assert abs(c[b, k] - 1 / (1 + math.exp(-(E[a["tokens"][b, k - 1]] @ w_e)))) < 1e-15
    # changing the last token changes nothing (no position reads it)
    t2 = a["tokens"].copy()
    t2[:, -1] = (t2[:, -1] + 1) % E.shape[0]
    assert np.array_equal(c, confidence(bias=0.0, sts_temp=np.ones(K), **{**a, "tokens": t2}))


def test_sts_preserves_order_within_position():
    a = _setup(2, B=30)
    K = a["h"].shape[1]
    c1 = confidence(bias=0.3, sts_temp=np.ones(K), **a)
    temps = np.linspace(0.5, 2.0, K)
    c2 = confidence(bias=0.3, sts_temp=temps, **a)
    for k in range(K):
        assert np.array_equal(np.argsort(c1[:, k], kind="stable"), np.argsort(c2[:, k], kind="stable"))
    # STS moves confidences toward 1/2 for T > 1, away for T < 1
    hi = temps > 1
    assert np.all(np.abs(c2[:, hi] - 0.5) <= np.abs(c1[:, hi] - 0.5) + 1e-15)


def test_survival_cumprod_and_monotone():
    c = np.array([[0.9, 0.5, 1.0, 0.2], [1.0, 1.0, 0.3, 0.7]])
    s = survival(c)
    np.testing.assert_allclose(s[0], [0.9, 0.45, 0.45, 0.09], rtol=1e-15)
    np.testing.assert_allclose(s[1], [1.0, 1.0, 0.3, 0.21], rtol=1e-15)
    rng = np.random.default_rng(3)
    s = survival(rng.random((50, 16)))
    assert np.all(np.diff(s, axis=1) <= 0)
