"""The parity comparison's own rules, checked on the CPU against planted
differences (the "GPU" results here are the oracle's, with one entry altered)."""
import numpy as np

import oracle
from tests import _parity


def test_first_divergence_indexes():
    out = np.array([4, 7, -1])
    assert _parity.first_divergence(2, 2, out, out) is None
    assert _parity.first_divergence(2, 0, out, out) == 0     # the GPU rejected at position 1
    assert _parity.first_divergence(1, 3, out, out) == 1     # the oracle rejected at position 2
    assert _parity.first_divergence(1, 1, out, np.array([4, 8, -1])) == -1   # the final draw


def _tiny():
    from speculative_decoding_draft_block_gb300.workloads import TINY, make_inputs
    inp = make_inputs(TINY)
    o = oracle.cycle(inp, 77)
    g = {"tokens": o["draft"]["tokens"], "L": o["schedule"]["L"],
         "accept_count": o["verify"]["accept_count"].copy(),
         "out_tokens": o["verify"]["out_tokens"].copy(),
         "num_emitted": o["verify"]["num_emitted"].copy()}
    return inp, o, g


def test_identical_results_pass_and_planted_differences_are_flagged():
    inp, o, g = _tiny()
    rep, _ = _parity.compare_verify(inp, g, 77)
    assert rep["mismatched_requests"] == 0 and not rep["unexplained"]
    dec = o["verify"]["decisions"]
    # a final token changed where the final draw is not a near tie: unexplained
    b = next(i for i in range(inp["B"]) if dec[i][-1][1] >= _parity.NEAR_TIE)
    g2 = dict(g, out_tokens=g["out_tokens"].copy())
    a = int(g["accept_count"][b])
    g2["out_tokens"][b, a] = (g2["out_tokens"][b, a] + 1) % inp["V"]
    rep, _ = _parity.compare_verify(inp, g2, 77)
    assert rep["unexplained"] == [b]
    # an accept count changed: the diverging decision is an accept test, not a near tie
    g3 = dict(g, accept_count=g["accept_count"].copy())
    g3["accept_count"][b] = a + 1 if a < int(g["L"][b]) else a - 1
    if dec[b][min(a, int(g3["accept_count"][b]))][1] >= _parity.NEAR_TIE:
        rep, _ = _parity.compare_verify(inp, g3, 77)
        assert rep["unexplained"] == [b]


def test_near_tie_elsewhere_in_the_request_does_not_excuse():
    """A request with a near tie on one decision but a difference on another is
    not excused (the excuse names the diverging decision)."""
    inp, o, g = _tiny()
    dec = [list(d) for d in o["verify"]["decisions"]]
    b = 0
    a = int(g["accept_count"][b])
    # pretend an earlier accept test of this request was a near tie
    if len(dec[b]) > 1:
        dec[b][0] = (dec[b][0][0], 0.0)
    if dec[b][-1][1] < _parity.NEAR_TIE:
        return
    idx = _parity.first_divergence(a, a, g["out_tokens"][b], g["out_tokens"][b] + 1)
    assert idx == -1 and dec[b][idx][1] >= _parity.NEAR_TIE
