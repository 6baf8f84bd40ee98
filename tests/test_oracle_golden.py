"""The oracle reproduces its stored tiny-cycle output (regression pin, CPU only).

tests/golden/tiny_cycle.json was written by tests/golden/make_golden.py, which
calls only the oracle and the seeded generator.
"""
import json
import os

import numpy as np

import oracle
from speculative_decoding_draft_block_gb300.workloads import TINY, make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tiny_cycle.json")


def test_tiny_cycle_matches_golden():
    g = json.load(open(GOLDEN))
    inp = make_inputs(TINY)
    res = oracle.cycle(inp, g["philox_seed"])
    assert res["draft"]["tokens"].tolist() == g["draft_tokens"]
    np.testing.assert_allclose(res["draft"]["q_token"], g["q_token"], rtol=1e-12)
    np.testing.assert_allclose(res["conf"], g["conf"], rtol=1e-12)
    assert res["schedule"]["L"].tolist() == g["sched_len"]
    assert res["verify"]["accept_count"].tolist() == g["accept_count"]
    assert res["verify"]["out_tokens"].tolist() == g["out_tokens"]


def test_workload_generator_is_deterministic():
    a = make_inputs(TINY)
    b = make_inputs(TINY)
    for k in ("base_logits", "target_logits", "E", "P", "h", "anchor", "temperature"):
        assert np.array_equal(a[k], b[k])
    assert a["base_logits"].shape == (4, 4, 1024) and a["target_logits"].shape == (4, 5, 1024)
