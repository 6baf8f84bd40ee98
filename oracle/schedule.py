"""Hardware-aware prefix scheduler with early stop, float64 (test infrastructure only).

DSpark summary page, 방법론 › 신뢰도 기반 검증: verification length is chosen to
maximise expected system throughput. SPS(n) is the target's throughput at verify
batch n, profiled once and stored as a table. Because survival is monotone along
a block, sorting all (request, position) candidates by survival and adding them
greedily respects every request's prefix. Losslessness needs non-anticipation:
the search stops the moment throughput drops, so each truncation depends only on
the prefix seen so far (same section, and 한계와 주의사항 for unimodality).

Reading of the objective (the pages give it in words only):
    R = B               every request always verifies its bonus/next position
    N = B + sum_b L_b   verify batch in tokens
    A = B + sum of included survivals   (expected emitted tokens)
    J = SPS(N) * A / N
Start at N = B, A = B. Walk candidates by survival descending, ties by
position ascending then request ascending; include a candidate iff the new J is
strictly larger than the current J, otherwise stop. SPS(n) beyond the table is
the last entry.

Asynchronous variant (same page, 주요 결과 › 프로덕션 배포 결과, and
한계와 주의사항): the verify capacity of the coming cycle is estimated from the
confidence head two cycles back, while the current cycle's candidates are
ranked by their own (fresh) cumulative confidence, a dynamic top-k. Reading:
the budget of cycle t is the greedy early-stop count of cycle t - 2 (an initial
value for the first two cycles), and cycle t verifies the first budget-many
candidates of its own sorted order. The budget never depends on cycle t's
tokens, which is the causal barrier the page describes.
"""

import numpy as np

SCHED_GREEDY_EARLYSTOP = 0
SCHED_FIXED_K = 1
SCHED_THRESHOLD = 2
SCHED_ASYNC = 3


def sps_at(sps, n):
    """SPS(n) for n >= 1 from a table indexed n = 1..len(sps), clamped beyond."""
    n = int(n)
    if n < 1:
        raise ValueError("verify batch must be >= 1")
    return float(sps[min(n, len(sps)) - 1])


def _sorted_candidates(s):
    B, K = s.shape
    return sorted(((b, k) for b in range(B) for k in range(K)),
                  key=lambda bk: (-s[bk[0], bk[1]], bk[1], bk[0]))


def schedule(s, sps, mode=SCHED_GREEDY_EARLYSTOP, threshold=0.0, budget=0):
    """Choose per-request verify lengths L [B] from survivals s [B, K].

    Returns a dict: L (int64 [B]), objective (J at the chosen set),
    n_included, and the near-tie measures of the stop: stop_rel_gain =
    (J - J') / J for the first rejected candidate, survival_gap = relative
    survival gap between the last included and the first excluded candidate.
    """
    s = np.asarray(s, dtype=np.float64)
    B, K = s.shape
    L = np.zeros(B, dtype=np.int64)
    if mode == SCHED_FIXED_K:
        L[:] = K
        n = B + B * K
        return {"L": L, "objective": sps_at(sps, n) * (B + s.sum()) / n,
                "n_included": B * K, "stop_rel_gain": np.inf, "survival_gap": np.inf}
    if mode == SCHED_THRESHOLD:
        # Static confidence threshold (the page's threshold sweep): keep the
        # longest prefix whose survival stays at or above the threshold.
        for b in range(B):
            L[b] = int(np.sum(s[b] >= threshold))
        n = B + int(L.sum())
        a = B + sum(float(s[b, :L[b]].sum()) for b in range(B))
        return {"L": L, "objective": sps_at(sps, n) * a / n, "n_included": int(L.sum()),
                "stop_rel_gain": np.inf, "survival_gap": np.inf}
    if mode == SCHED_ASYNC:
        # dynamic top-k: the first `budget` candidates of the current order
        greedy_count = schedule(s, sps)["n_included"]
        m = min(max(int(budget), 0), B * K)
        a = float(B)
        for b, k in _sorted_candidates(s)[:m]:
            if L[b] != k:
                raise AssertionError("selection is not prefix-closed")
            L[b] += 1
            a += s[b, k]
        n = B + m
        return {"L": L, "objective": sps_at(sps, n) * a / n, "n_included": m,
                "greedy_count": greedy_count, "stop_rel_gain": np.inf, "survival_gap": np.inf}
    if mode != SCHED_GREEDY_EARLYSTOP:
        raise ValueError("unknown schedule mode")

    order = _sorted_candidates(s)
    n, a = B, float(B)
    j = sps_at(sps, n) * a / n
    stop_rel_gain = np.inf
    survival_gap = np.inf
    last_included = None
    for b, k in order:
        n1, a1 = n + 1, a + s[b, k]
        j1 = sps_at(sps, n1) * a1 / n1
        if j1 > j:
            if L[b] != k:
                raise AssertionError("selection is not prefix-closed")
            L[b] += 1
            n, a, j = n1, a1, j1
            last_included = s[b, k]
        else:
            stop_rel_gain = (j - j1) / j
            if last_included is not None and last_included > 0:
                survival_gap = (last_included - s[b, k]) / last_included
            break
    return {"L": L, "objective": j, "n_included": int(L.sum()),
            "stop_rel_gain": float(stop_rel_gain), "survival_gap": float(survival_gap)}


def async_budgets(greedy_counts, initial):
    """Budgets of cycles 0, 1, 2, ... under the asynchronous scheduler: the
    first two cycles use `initial`, cycle t >= 2 uses the greedy count of t - 2."""
    return [initial if t < 2 else int(greedy_counts[t - 2]) for t in range(len(greedy_counts))]
