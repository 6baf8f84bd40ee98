"""Pins for the oracle's rejection-sampling verification (CPU only)."""
import itertools

import numpy as np
import pytest

import oracle.verify as ov
from oracle import verify_request, verify, schedule, confidence, survival, markov_logits
from oracle.draft import draft_step
from tests._exact import outcome_measures


def _accept_prob(p, q, x):
    """Measure of {u : the oracle accepts x} for one position."""
    meas = outcome_measures(lambda u: verify_request([x], 1, lambda j: p, lambda j: q,
                                                     lambda j: u, lambda j: 0.5)[0])
    return meas.get(1, 0.0)


def _rand_dist(rng, V, zeros=0.0):
    w = rng.exponential(size=V) * (rng.random(V) >= zeros)
    if w.sum() == 0:
        w[0] = 1.0
    return w / w.sum()


def test_acceptance_is_one_minus_total_variation():
    rng = np.random.default_rng(0)
    for _ in range(6):
        V = 12
        p, q = _rand_dist(rng, V, 0.2), _rand_dist(rng, V, 0.2)
        alpha = sum(q[x] * _accept_prob(p, q, x) for x in range(V) if q[x] > 0)
        tv = 0.5 * np.abs(p - q).sum()
        assert abs(alpha - (1.0 - tv)) < 1e-13
        assert abs(alpha - np.minimum(p, q).sum()) < 1e-13


def test_special_cases():
    rng = np.random.default_rng(1)
    p = _rand_dist(rng, 8)
    for x in range(8):
        assert _accept_prob(p, p, x) == 1.0           # p = q: always accept
    p = np.array([0.5, 0.5, 0.0, 0.0])
    q = np.array([0.0, 0.0, 0.3, 0.7])
    for x in (2, 3):
        assert _accept_prob(p, q, x) == 0.0           # disjoint supports: always reject


def _lossless_law(V, K, T, L_of, seed, plant=None):
    """Exact law over V^(K+1) of: draft a block, schedule, verify, then extend the
    emitted tokens to length K+1 with the exact target conditionals."""
    rng = np.random.default_rng(seed)
    r = 3
    z = rng.normal(0, 1.0, size=(K, V))
    E = rng.normal(0, 1.0, size=(V, r))
    P = rng.normal(0, 1.0, size=(r, V))
    anchor = int(rng.integers(V))
    tbl = {}

    def tgt_logits(prefix):
        if prefix not in tbl:
            tbl[prefix] = rng.normal(0, 1.5, size=V)
        return tbl[prefix]

    tcache, qcache = {}, {}

    def tprob(prefix):
        if prefix in tcache:
            return tcache[prefix]
        tcache[prefix] = _tprob(prefix)
        return tcache[prefix]

    def qprob(j, prev):
        if (j, prev) not in qcache:
            qcache[(j, prev)] = _qprob(j, prev)
        return qcache[(j, prev)]

    def _tprob(prefix):
        lg = tgt_logits(prefix)
        if T == 0:
            e = np.zeros(V); e[int(np.argmax(lg))] = 1.0
            return e
        w = np.exp(lg / T - (lg / T).max())
        return w / w.sum()

    def _qprob(j, prev):
        ell = markov_logits(z[j:j + 1], E, P, [prev])[0]
        if T == 0:
            e = np.zeros(V); e[int(np.argmax(ell))] = 1.0
            return e
        w = np.exp(ell / T - (ell / T).max())
        return w / w.sum()

    draft_law = {}

    def draft_measure(j, prev):
        key = (j, prev)
        if key not in draft_law:
            ell = markov_logits(z[j:j + 1], E, P, [prev])[0]
            draft_law[key] = outcome_measures(lambda u: draft_step(ell, T, u)[0])
        return draft_law[key]

    vr = plant or verify_request
    law = np.zeros((V,) * (K + 1))
    for xs in itertools.product(range(V), repeat=K):
        px, prev = 1.0, anchor
        for j, x in enumerate(xs):
            px *= draft_measure(j, prev).get(x, 0.0)
            prev = x
        if px == 0.0:
            continue
        L = L_of(xs)
        p_row = (lambda j, xs=xs: tgt_logits(tuple(xs[:j])) if T == 0 else tprob(tuple(xs[:j])))
        q_row = (lambda j, xs=xs: qprob(j, anchor if j == 0 else xs[j - 1]))

        # accept decisions, then the final draw, each integrated over its own u
        acc = []
        for j in range(L):
            meas = outcome_measures(lambda u, j=j: vr(
                xs, j + 1, p_row, q_row, lambda i, j=j: u if i == j else 2.0 ** -60, lambda i: 0.5,
                greedy=T == 0)[0] == j + 1)
            acc.append(meas.get(True, 0.0))
        reach = 1.0
        for a in range(L + 1):
            if a > 0:
                reach *= acc[a - 1]
            if reach == 0.0:
                break
            stop = (1.0 - acc[a]) if a < L else 1.0
            if stop == 0.0:
                continue
            ua = lambda i, a=a: 2.0 ** -60 if i < a else 1.0 - 2.0 ** -53
            final = outcome_measures(lambda u, ua=ua, a=a: vr(
                xs, L, p_row, q_row, ua, lambda i: u, greedy=T == 0)[1][a])
            for y, my in final.items():
                seq = tuple(xs[:a]) + (y,)
                w = px * reach * stop * my
                # extend to length K+1 with the exact target conditionals
                frontier = [(seq, w)]
                while len(frontier[0][0]) < K + 1:
                    nxt = []
                    for sq, wt in frontier:
                        pr = tprob(sq)
                        nxt.extend((sq + (t,), wt * pr[t]) for t in range(V) if pr[t] > 0)
                    frontier = nxt
                for sq, wt in frontier:
                    law[sq] += wt
    target = np.zeros_like(law)
    for seq in itertools.product(range(V), repeat=K + 1):
        pr = 1.0
        for j in range(K + 1):
            pr *= tprob(tuple(seq[:j]))[seq[j]]
        target[seq] = pr
    return law, target


def _sched_L(V, K, seed):
    rng = np.random.default_rng(seed + 100)
    d, r = 4, 3
    h = rng.normal(size=(1, K, d))
    E = rng.normal(size=(V, r))
    w_h, w_e = rng.normal(size=d) * 0.3, rng.normal(size=r) * 2.0
    n = np.arange(1, K + 2)
    sps = n / (1.0 + n / 2.0)

    def L_of(xs):
        c = confidence(h, E, [0], np.array([xs]), w_h, w_e, 2.0, np.ones(K))
        return int(schedule(survival(c), sps)["L"][0])
    return L_of


@pytest.mark.parametrize("T", [1.0, 0.7])
def test_lossless_with_scheduler_V8_K3(T):
    V, K = 8, 3
    L_of = _sched_L(V, K, 0)
    Ls = {L_of(xs) for xs in itertools.product(range(V), repeat=K)}
    assert len(Ls) >= 2                              # the schedule really varies with the draft
    law, target = _lossless_law(V, K, T, L_of, seed=11)
    assert abs(law.sum() - 1.0) < 1e-12
    assert np.abs(law - target).max() < 1e-12


@pytest.mark.parametrize("L", [0, 1, 2, 3])
def test_lossless_fixed_length_V8_K3(L):
    law, target = _lossless_law(8, 3, 1.0, lambda xs: L, seed=12 + L)
    assert np.abs(law - target).max() < 1e-12


def test_lossless_greedy_V8_K3():
    law, target = _lossless_law(8, 3, 0.0, lambda xs: 3, seed=20)
    assert np.abs(law - target).max() < 1e-12


def test_planted_mistake_is_caught():
    """Resampling from p instead of the residual max(0, p - q) must break losslessness."""
    from oracle.sampling import inverse_cdf

    def broken(tokens, L, p_row, q_row, u_accept, u_resample, greedy=False):
        a, out, dec = verify_request(tokens, L, p_row, q_row, u_accept, u_resample, greedy)
        if a < L:
            out[-1] = inverse_cdf(p_row(a), u_resample(a))[0]
        return a, out, dec
    law, target = _lossless_law(6, 2, 1.0, lambda xs: 2, seed=30, plant=broken)
    assert np.abs(law - target).max() > 1e-3


def test_batch_verify_uses_right_rows_and_streams():
    rng = np.random.default_rng(5)
    B, K, V, r = 3, 3, 10, 2
    tgt = rng.normal(size=(B, K + 1, V))
    base = rng.normal(size=(B, K, V))
    E, P = rng.normal(size=(V, r)), rng.normal(size=(r, V))
    anchor = np.array([0, 1, 2])
    tokens = rng.integers(0, V, size=(B, K))
    T = np.array([1.0, 1.0, 0.0], dtype=np.float32)
    L = np.array([3, 0, 2])
    out = verify(tgt, base, E, P, anchor, tokens, L, T, 5)
    assert out["num_emitted"][1] == 1 and out["accept_count"][1] == 0
    for b in range(B):
        n = out["num_emitted"][b]
        assert np.all(out["out_tokens"][b, n:] == -1)
        assert np.array_equal(out["out_tokens"][b, :n - 1], tokens[b, :n - 1])
    # greedy request: emitted tokens are target argmaxes along the accepted prefix
    b = 2
    a = out["accept_count"][b]
    for j in range(a):
        assert tokens[b, j] == np.argmax(tgt[b, j])
    assert out["out_tokens"][b, a] == np.argmax(tgt[b, a])


def test_p_token_closed_form():
    """p_k(x_k) of every scheduled position, pinned on hand-built target rows.

    Target logits T * ln(1, 2, 3, 4) give p = (0.1, 0.2, 0.3, 0.4) at any
    temperature T > 0; rows after a rejection are still reported (they are
    scheduled), positions past L are NaN. Greedy requests report the point mass
    of their argmax (token 3)."""
    V, K = 4, 3
    base = np.zeros((3, K, V))
    E = np.zeros((V, 2))
    P = np.zeros((2, V))
    temps = np.array([1.0, 2.5, 0.0], dtype=np.float32)
    tgt = np.zeros((3, K + 1, V))
    for b, T in enumerate(temps):
        tgt[b, :, :] = (T if T > 0 else 1.0) * np.log(np.arange(1.0, V + 1.0))
    tokens = np.array([[2, 0, 1], [1, 3, 3], [3, 1, 3]])
    res = verify(tgt, base, E, P, np.zeros(3, dtype=np.int64), tokens, np.array([3, 2, 3]), temps,
                 seed=5, with_p=True)
    p = res["p_token"]
    want = np.array([0.3, 0.1, 0.2])
    assert np.all(np.abs(p[0] - want) < 1e-15)
    assert np.all(np.abs(p[1, :2] - np.array([0.2, 0.4])) < 1e-15) and np.isnan(p[1, 2])
    assert p[2].tolist() == [1.0, 0.0, 1.0]
    # the accept decisions read exactly these probabilities: q = 1/4 (uniform draft)
    for j in range(res["accept_count"][0]):
        assert oracle_uniform_accept(5, 0, j) * 0.25 < p[0, j]
    assert "p_token" not in verify(tgt, base, E, P, np.zeros(3, dtype=np.int64), tokens,
                                   np.array([3, 2, 3]), temps, seed=5)


def oracle_uniform_accept(seed, b, j):
    from oracle.philox import uniform, STAGE_ACCEPT
    return uniform(seed, b, j + 1, STAGE_ACCEPT)
