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


def test_hidden_state_term_reads_h_k_of_its_own_position():
    """The w_h . h_k term, pinned in closed form with w_e = 0.

    w_h is the unit vector e_j and h[b, k, j] = ln m[b, k] with m distinct for
    every (b, k); the other hidden components are random (weight 0). Then
    sigmoid(w_h . h_k) = m / (1 + m) exactly for that k, and sigmoid(ln m / T)
    = m^(1/T) / (1 + m^(1/T)) under an STS temperature T. Reading h_{k+1} or
    h_{k-1}, another request's row, or contracting the wrong axis gives
    another m (or a random value) and fails.
    """
    B, K, d = 3, 5, 7
    rng = np.random.default_rng(11)
    m = 1.0 + np.arange(B * K, dtype=np.float64).reshape(B, K) * 0.37   # distinct, > 0
    for j in (0, 4):
        a = _setup(12, B=B, K=K, d=d)
        a["w_e"][:] = 0.0
        a["h"] = rng.normal(size=(B, K, d)) * 3.0
        a["h"][:, :, j] = np.log(m)
        a["w_h"] = np.zeros(d)
        a["w_h"][j] = 1.0
        c = confidence(bias=0.0, sts_temp=np.ones(K), **a)
        for b in range(B):
            for k in range(K):
                assert abs(c[b, k] - m[b, k] / (1.0 + m[b, k])) < 1e-15, (j, b, k)
        temps = np.array([0.5, 1.0, 2.0, 4.0, 0.8])
        c = confidence(bias=0.0, sts_temp=temps, **a)
        for b in range(B):
            for k in range(K):
                mt = m[b, k] ** (1.0 / temps[k])
                assert abs(c[b, k] - mt / (1.0 + mt)) < 1e-14, (j, b, k)


def test_hidden_and_embedding_terms_add_inside_the_sigmoid():
    """Both terms and the bias together: w_h . h_k = ln a, w_e . E[x_{k-1}] = ln e,
    b = ln 2 give c = 2ae / (1 + 2ae) (a product inside one sigmoid, not two
    sigmoids or a sum of them)."""
    B, K, d, V, r = 2, 4, 5, 9, 3
    rng = np.random.default_rng(13)
    a_val = 1.0 + rng.random((B, K))
    e_val = 0.5 + rng.random(V)
    h = rng.normal(size=(B, K, d))
    h[:, :, 2] = np.log(a_val)
    w_h = np.zeros(d)
    w_h[2] = 1.0
    E = rng.normal(size=(V, r))
    E[:, 1] = np.log(e_val)
    w_e = np.zeros(r)
    w_e[1] = 1.0
    anchor = rng.integers(0, V, size=B)
    tokens = rng.integers(0, V, size=(B, K))
    c = confidence(h, E, anchor, tokens, w_h, w_e, math.log(2.0), np.ones(K))
    for b in range(B):
        for k in range(K):
            prev = anchor[b] if k == 0 else tokens[b, k - 1]
            x = 2.0 * a_val[b, k] * e_val[prev]
            assert abs(c[b, k] - x / (1.0 + x)) < 1e-15, (b, k)
