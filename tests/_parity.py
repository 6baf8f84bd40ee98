"""Comparison of a GPU cycle with the oracle on the same seeded inputs.

Rules (from the parity specification):
  * token ids, accept counts and scheduled lengths are compared exactly;
  * a mismatch is allowed only at a near-tie -- a draw whose float64 CDF margin
    to u is below 1e-6 (greedy choices: top-1/top-2 logit gap below 1e-6;
    accept tests: |u - p/q| below 1e-6; schedule: relative objective change or
    survival gap at the stop below 1e-5) -- and mismatched draws must stay
    under 1e-4 of all draws;
  * probabilities -- q(x_k) of every draw, p(x_k) of every verified position --
    and confidences agree within 2e-3 relative;
  * a request whose verify outcome differs is excused only when the first
    decision on which it differs is itself a near tie.
Every draw is checked on its own: the oracle is teacher-forced with the GPU's
previous tokens, so one exempt mismatch does not cascade.
"""
import numpy as np

import oracle

NEAR_TIE = 1e-6
SCHED_NEAR_TIE = 1e-5
MISMATCH_BUDGET = 1e-4
REL_TOL = 2e-3


ROW_KEYS = ("base_logits", "target_logits", "anchor", "temperature", "h")
GPU_ROW_KEYS = ("tokens", "q_token", "conf", "survival", "L", "out_tokens", "accept_count", "p_token",
                "num_emitted", "states")


def subset(inp, g, rows):
    """Restrict inputs and GPU results to some requests (the RNG keeps global ids)."""
    rows = np.asarray(rows)
    si = dict(inp)
    for k in ROW_KEYS:
        si[k] = inp[k][rows]
    sg = dict(g)
    for k in GPU_ROW_KEYS:
        if g.get(k) is not None:
            sg[k] = g[k][rows]
    return si, sg


def compare_draft(inp, g, seed, request_ids=None):
    o = oracle.draft_block(inp["base_logits"], inp["E"], inp["P"], inp["anchor"],
                           inp["temperature"], seed, prev_tokens=g["tokens"],
                           request_ids=request_ids)
    mism = o["tokens"] != g["tokens"]
    near = o["margin"] < NEAR_TIE
    draws = mism.size
    rep = {"draws": int(draws), "mismatches": int(mism.sum()), "near_ties": int(near.sum()),
           "unexplained": int((mism & ~near).sum())}
    ok = ~mism
    rel = np.abs(g["q_token"][ok] - o["q_token"][ok]) / np.maximum(o["q_token"][ok], 1e-300)
    rep["q_max_rel"] = float(rel.max()) if rel.size else 0.0
    return rep, o


# The kernel sums each gate pre-activation in float32 over 2r + d products
# (magnitudes summing to ~10-20 for these weights: an error up to ~1e-5), and
# the gates pass it on with slope <= 1. So each stored bfloat16 state must be
# a correct rounding of a value within STATE_ABS of the float64 state:
# |s_gpu - s| <= ulp(s_gpu) / 2 + STATE_ABS. Where the rounding differs from
# the oracle's (a value near a rounding boundary, or a tiny value whose ulp is
# below the float32 error), at most STATE_DIFF_BUDGET of the elements.
STATE_ABS = 1e-5
STATE_DIFF_BUDGET = 1e-2


def compare_draft_rnn(inp, g, seed, rnn, request_ids=None):
    """RNN head: every state and every draw checked on its own.

    The oracle is teacher-forced with the GPU's tokens and states: state k is
    recomputed from the GPU's state k-1, and draw k uses the GPU's state k.
    Every stored state must be a bfloat16 rounding of a value within STATE_ABS
    of the float64 state; at most STATE_DIFF_BUDGET of them may round otherwise
    than the oracle.
    """
    from oracle.bf16 import as_f64
    o = oracle.rnn_draft_block(inp["base_logits"], inp["E"], inp["P"], inp["anchor"],
                               inp["temperature"], seed, inp["h"], rnn["w_ih"], rnn["w_hh"],
                               rnn["b_ih"], rnn["b_hh"], bf16_state=inp["bf16"],
                               prev_tokens=g["tokens"], prev_states=g["states"],
                               request_ids=request_ids)
    gs = as_f64(g["states"])
    diff = gs != o["states"]
    _, e = np.frexp(gs)
    half_ulp = np.where(gs == 0, 0.0, np.ldexp(0.5, e - 8))   # bfloat16: 8 significant bits
    excess = np.abs(gs - o["states_pre"]) - half_ulp
    mism = o["tokens"] != g["tokens"]
    near = o["margin"] < NEAR_TIE
    rep = {"draws": int(mism.size), "mismatches": int(mism.sum()), "near_ties": int(near.sum()),
           "unexplained": int((mism & ~near).sum()),
           "state_elems": int(diff.size), "state_diffs": int(diff.sum()),
           "state_unexplained": int((excess > STATE_ABS).sum()),
           "state_max_excess": float(excess.max())}
    ok = ~mism
    rel = np.abs(g["q_token"][ok] - o["q_token"][ok]) / np.maximum(o["q_token"][ok], 1e-300)
    rep["q_max_rel"] = float(rel.max()) if rel.size else 0.0
    return rep, o


def compare_schedule(inp, g):
    c = oracle.confidence(inp["h"], inp["E"], inp["anchor"], g["tokens"], inp["w_h"], inp["w_e"],
                          inp["conf_bias"], inp["sts_temp"])
    s = oracle.survival(c)
    sch = oracle.schedule(s, inp["sps"])
    rep = {
        "conf_max_rel": float(np.max(np.abs(g["conf"] - c) / c)),
        "surv_max_rel": float(np.max(np.abs(g["survival"] - s) / s)),
        "L_mismatch": int(np.sum(sch["L"] != g["L"])),
        "near_tie": bool(min(sch["stop_rel_gain"], sch["survival_gap"]) < SCHED_NEAR_TIE),
        "objective_rel": abs(g["objective"] - sch["objective"]) / abs(sch["objective"]),
    }
    return rep, sch


def first_divergence(o_accept, g_accept, o_out, g_out):
    """Index, in the oracle's decision list of one request, of the first decision
    on which the GPU's outcome differs from the oracle's, or None if none does.

    Both sides are teacher-forced on the same drafted tokens and scheduled
    length, so they take the same accept tests left to right: decision j is the
    test at position j + 1. While both accept they agree; the first position
    where one accepts and the other rejects is decision min(a_oracle, a_gpu).
    With equal accept counts, only the final draw (the last decision: residual,
    bonus or greedy argmax) can differ.
    """
    if o_accept != g_accept:
        return min(o_accept, g_accept)
    if np.any(o_out != g_out):
        return -1
    return None


def compare_verify(inp, g, seed, request_ids=None):
    o = oracle.verify(inp["target_logits"], inp["base_logits"], inp["E"], inp["P"], inp["anchor"],
                      g["tokens"], g["L"], inp["temperature"], seed, request_ids=request_ids,
                      states=g.get("states"), with_p=True)
    bad_req = np.nonzero((o["accept_count"] != g["accept_count"]) |
                         np.any(o["out_tokens"] != g["out_tokens"], axis=1))[0]
    decisions = sum(len(d) for d in o["decisions"])
    unexplained = []
    for b in bad_req:
        i = first_divergence(int(o["accept_count"][b]), int(g["accept_count"][b]),
                             o["out_tokens"][b], g["out_tokens"][b])
        # excused only when the diverging decision itself is a near tie
        if i is not None and not o["decisions"][b][i][1] < NEAR_TIE:
            unexplained.append(int(b))
    near = sum(1 for d in o["decisions"] for _, m in d if m < NEAR_TIE)
    rep = {"requests": int(len(g["L"])), "decisions": int(decisions),
           "mismatched_requests": int(len(bad_req)), "unexplained": unexplained,
           "near_ties": int(near)}
    if g.get("p_token") is not None:
        # p_k(x_k) of the positions verify evaluated, against float64: every
        # position up to and including the first rejection must be evaluated;
        # later scheduled positions may be (-1 when skipped); -1 past L_b
        K = g["tokens"].shape[1]
        pos = np.arange(K)[None, :]
        L = np.asarray(g["L"])[:, None]
        a = np.asarray(g["accept_count"])[:, None]
        sched = pos < L
        gp, op = g["p_token"], o["p_token"]
        assert np.all(gp[~sched] == -1.0), "p_token not -1 past the scheduled length"
        must = sched & (pos <= a)
        assert np.all(gp[must] != -1.0), "a position up to the first rejection was not evaluated"
        ev = sched & (gp != -1.0)
        greedy = (np.asarray(inp["temperature"]) == 0)[:, None] & ev
        assert np.array_equal(gp[greedy], op[greedy]), "greedy p_token is not the point mass"
        samp = ev & ~greedy
        rel = np.abs(gp[samp] - op[samp]) / np.maximum(op[samp], 1e-30)
        rep["p_compared"] = int(samp.sum())
        rep["p_skipped"] = int((sched & (gp == -1.0)).sum())
        rep["p_max_rel"] = float(rel.max()) if rel.size else 0.0
    return rep, o


def assert_parity(inp, g, seed, check_schedule=True, check_verify=True, rows=None, rnn=None):
    """Check a GPU cycle against the oracle; ``rows`` limits draft/verify to some requests;
    ``rnn`` (the head's weights) selects the RNN head."""
    if check_schedule:
        rs, _ = compare_schedule(inp, g)
        assert rs["conf_max_rel"] < REL_TOL and rs["surv_max_rel"] < REL_TOL, rs
        if not rs["near_tie"]:
            assert rs["L_mismatch"] == 0, rs
            assert rs["objective_rel"] < 1e-5, rs
    rid = None
    if rows is not None:
        inp, g = subset(inp, g, rows)
        rid = np.asarray(rows)
    if rnn is not None:
        rd, od = compare_draft_rnn(inp, g, seed, rnn, request_ids=rid)
        assert rd["state_unexplained"] == 0, rd
        assert rd["state_diffs"] <= STATE_DIFF_BUDGET * rd["state_elems"], rd
    else:
        rd, od = compare_draft(inp, g, seed, request_ids=rid)
    assert rd["unexplained"] == 0, rd
    assert rd["mismatches"] <= MISMATCH_BUDGET * rd["draws"], rd
    assert rd["q_max_rel"] < REL_TOL, rd
    out = {"draft": rd}
    if check_schedule:
        out["schedule"] = rs
    if check_verify:
        rv, _ = compare_verify(inp, g, seed, request_ids=rid)
        assert not rv["unexplained"], rv
        assert rv["mismatched_requests"] <= MISMATCH_BUDGET * rv["decisions"], rv
        assert rv.get("p_max_rel", 0.0) < REL_TOL, rv
        out["verify"] = rv
    return out
