"""Pins for the oracle's hardware-aware prefix scheduler (CPU only)."""
import itertools

import numpy as np
import pytest

from oracle import schedule, sps_at, SCHED_FIXED_K, SCHED_THRESHOLD
from oracle.confidence import survival


def _J(sps, B, L, s):
    n = B + int(np.sum(L))
    a = B + sum(float(s[b, :L[b]].sum()) for b in range(B))
    return sps_at(sps, n) * a / n


def _random_s(rng, B, K):
    return survival(rng.uniform(0.3, 1.0, size=(B, K)))


def test_sps_clamp():
    sps = np.array([1.0, 2.0, 3.0])
    assert sps_at(sps, 1) == 1.0 and sps_at(sps, 3) == 3.0 and sps_at(sps, 99) == 3.0
    with pytest.raises(ValueError):
        sps_at(sps, 0)


def test_sorted_greedy_maximises_sum_for_every_size():
    """Brute force over all prefix-closed selections of tiny instances."""
    rng = np.random.default_rng(0)
    B, K = 3, 3
    for _ in range(20):
        s = _random_s(rng, B, K)
        best = {}
        for L in itertools.product(range(K + 1), repeat=B):
            m = sum(L)
            tot = sum(float(s[b, :L[b]].sum()) for b in range(B))
            best[m] = max(best.get(m, -1.0), tot)
        top = np.sort(s.ravel())[::-1]
        for m, v in best.items():
            assert abs(v - top[:m].sum()) < 1e-12


def test_early_stop_reaches_optimum_when_unimodal():
    rng = np.random.default_rng(1)
    B, K = 3, 3
    n_max = B * (K + 1)
    n = np.arange(1, n_max + 1)
    checked = 0
    for trial in range(60):
        s = _random_s(rng, B, K)
        sps = n * 9.0 / (1.0 + n / rng.uniform(1.0, 8.0))
        top = np.sort(s.ravel())[::-1]
        J = [sps_at(sps, B + m) * (B + top[:m].sum()) / (B + m) for m in range(B * K + 1)]
        m_star = int(np.argmax(J))
        unimodal = all(J[i + 1] > J[i] for i in range(m_star)) and all(
            J[i + 1] <= J[i] for i in range(m_star, len(J) - 1))
        if not unimodal:
            continue
        checked += 1
        res = schedule(s, sps)
        assert res["n_included"] == m_star
        glob = max(_J(sps, B, L, s) for L in itertools.product(range(K + 1), repeat=B))
        assert abs(res["objective"] - glob) <= 1e-12 * glob
    assert checked >= 20


def test_linear_sps_verifies_everything():
    rng = np.random.default_rng(2)
    s = _random_s(rng, 5, 7)
    sps = 3.0 * np.arange(1, 5 * 8 + 1)
    assert np.all(schedule(s, sps)["L"] == 7)


def test_fixed_and_threshold_modes():
    s = survival(np.array([[0.9, 0.9, 0.5], [0.4, 0.9, 0.9]]))
    sps = np.ones(8)
    assert np.all(schedule(s, sps, mode=SCHED_FIXED_K)["L"] == 3)
    assert list(schedule(s, sps, mode=SCHED_THRESHOLD, threshold=0.5)["L"]) == [2, 0]


def test_flat_sps_verifies_nothing():
    """Constant SPS: J = SPS * A / N falls with every candidate (s <= 1 < A/N only if...)."""
    s = np.full((4, 3), 0.999)
    sps = np.full(16, 5.0)
    assert np.all(schedule(s, sps)["L"] == 0)


def test_non_anticipation_metamorphic():
    """Changing survivals after position k never changes min(L_b, k)."""
    rng = np.random.default_rng(3)
    B, K = 6, 5
    n = np.arange(1, B * (K + 1) + 1)
    for _ in range(40):
        c = rng.uniform(0.4, 1.0, size=(B, K))
        sps = n * 5.0 / (1.0 + n / rng.uniform(2.0, 30.0))
        L = schedule(survival(c), sps)["L"]
        b = int(rng.integers(B))
        k = int(rng.integers(1, K))
        c2 = c.copy()
        c2[b, k:] = rng.uniform(0.0, 1.0, size=K - k)      # positions k+1.. of request b
        L2 = schedule(survival(c2), sps)["L"]
        assert min(L[b], k) == min(L2[b], k)


def test_global_search_would_anticipate():
    """Without early stop the choice can depend on a later position (pages' warning)."""
    sps = np.array([10.0, 12.0, 19.0])     # B = 1: J0 = 10, J1 = 6 * 1.5 = 9, J2 = 19 (1.5 + s2) / 3
    def glob(s):
        Js = [sps[m] * (1 + s[0, :m].sum()) / (1 + m) for m in range(3)]
        return int(np.argmax(Js))
    lo = np.array([[0.5, 0.05]])
    hi = np.array([[0.5, 0.45]])
    assert glob(lo) == 0 and glob(hi) == 2           # min(L, 1) flips with s_2
    assert schedule(lo, sps)["n_included"] == schedule(hi, sps)["n_included"] == 0


# ---- asynchronous scheduler (budget from two cycles back, dynamic top-k) -----

def _hyper_sps(B, K):
    n = np.arange(1, B * (K + 1) + 1)
    return n * 9e4 / (1.0 + n / 96.0)


def test_async_with_its_own_greedy_count_is_the_greedy_schedule():
    from oracle import SCHED_ASYNC
    rng = np.random.default_rng(11)
    for B, K in ((3, 4), (8, 5), (16, 8)):
        sps = _hyper_sps(B, K)
        for _ in range(10):
            s = _random_s(rng, B, K)
            g = schedule(s, sps)
            a = schedule(s, sps, SCHED_ASYNC, budget=g["n_included"])
            assert np.array_equal(a["L"], g["L"])
            assert abs(a["objective"] - g["objective"]) <= 1e-12 * g["objective"]
            assert a["greedy_count"] == g["n_included"]


def test_async_budget_edges_and_fixed_shape():
    from oracle import SCHED_ASYNC
    rng = np.random.default_rng(12)
    B, K = 5, 4
    sps = _hyper_sps(B, K)
    s = _random_s(rng, B, K)
    for budget in (-3, 0):
        r = schedule(s, sps, SCHED_ASYNC, budget=budget)
        assert (r["L"] == 0).all() and r["objective"] == sps_at(sps, B)
    for budget in (B * K, B * K + 7):
        assert (schedule(s, sps, SCHED_ASYNC, budget=budget)["L"] == K).all()
    for budget in range(B * K + 1):
        r = schedule(s, sps, SCHED_ASYNC, budget=budget)
        assert int(r["L"].sum()) == budget          # the verify batch is fixed in advance
        assert abs(r["objective"] - _J(sps, B, r["L"], s)) <= 1e-12 * r["objective"]


def test_async_top_k_is_the_best_prefix_closed_set_of_its_size():
    """Brute force: for every budget m, the selection maximises the summed
    survival over all prefix-closed selections with m candidates."""
    from oracle import SCHED_ASYNC
    rng = np.random.default_rng(13)
    B, K = 3, 3
    sps = _hyper_sps(B, K)
    for _ in range(20):
        s = _random_s(rng, B, K)
        best = {}
        for L in itertools.product(range(K + 1), repeat=B):
            tot = sum(float(s[b, :L[b]].sum()) for b in range(B))
            best[sum(L)] = max(best.get(sum(L), -1.0), tot)
        for m, v in best.items():
            L = schedule(s, sps, SCHED_ASYNC, budget=m)["L"]
            got = sum(float(s[b, :L[b]].sum()) for b in range(B))
            assert abs(got - v) < 1e-12


def test_async_budget_never_sees_the_current_cycle():
    """Causal barrier: changing cycle t's survivals leaves the budgets of
    cycles 0..t+1 unchanged (only cycle t+2 may follow it)."""
    from oracle import async_budgets
    rng = np.random.default_rng(14)
    B, K, T = 6, 5, 7
    sps = _hyper_sps(B, K)
    cycles = [_random_s(rng, B, K) for _ in range(T)]
    counts = [schedule(s, sps)["n_included"] for s in cycles]
    base = async_budgets(counts, initial=9)
    assert base[:2] == [9, 9] and base[2:] == counts[:T - 2]
    for t in range(T):
        pert = list(cycles)
        pert[t] = _random_s(rng, B, K) ** 3
        c2 = [schedule(s, sps)["n_included"] for s in pert]
        b2 = async_budgets(c2, initial=9)
        assert b2[:t + 2] == base[:t + 2]
