"""RNN head (CUDA, through the C ABI) against the RNN oracle.

DSpark summary page, 방법론 › 반자기회귀 생성: the RNN head's state accumulates
the whole drafted prefix. The oracle is teacher-forced with the GPU's tokens
and states (tests/_parity.py, compare_draft_rnn): each state is recomputed in
float64 from the GPU's previous state, and each stored bfloat16 state must be
a rounding of a value within 1e-5 of it (at most 1 % of the elements rounding
otherwise than the oracle); each draw is compared under the usual near-tie
rule; verify rebuilds q from the GPU's states.
"""
import os

import numpy as np
import pytest

import _parity

pytestmark = pytest.mark.gpu

SEED = 0x5EED7000


@pytest.fixture(scope="module")
def ds():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_draft_block_gb300 import _lib, build
    if not os.path.exists(_lib.LIB_PATH):
        build.build()
    return _lib


def _inputs(B=37, K=5, V=3000, r=64, d=128, temps=(0.0, 0.6, 1.0), seed=21):
    from speculative_decoding_draft_block_gb300.workloads import B256, scaled, make_inputs
    w = scaled(B256, name="rnn", B=B, K=K, V=V, r=r, d=d, bf16=True, temps=temps, seed=seed)
    return make_inputs(w)


def _cycle(inp, w, seed, token_major_projection=True):
    from speculative_decoding_draft_block_gb300.cycle import DeviceCycle
    cyc = DeviceCycle(inp, rnn_weights=w, token_major_projection=token_major_projection)
    cyc.reset_status()
    cyc.run(seed)
    cyc.check_status()
    return cyc, cyc.results()


@pytest.mark.parametrize("r,d,tmp", [(64, 128, True), (128, 192, False)])
def test_rnn_ragged_cycle(ds, r, d, tmp):
    from speculative_decoding_draft_block_gb300.workloads import make_rnn_weights
    inp = _inputs(r=r, d=d, seed=21 + r)
    w = make_rnn_weights(r, d, seed=5 + r)
    _, g = _cycle(inp, w, SEED, token_major_projection=tmp)
    rep = _parity.assert_parity(inp, g, SEED, rnn=w)
    assert rep["draft"]["draws"] == 37 * 5
    assert rep["draft"]["state_elems"] == 37 * 5 * r
    # the states really move: bounded, non-zero, different across positions
    from oracle.bf16 import as_f64
    s = as_f64(g["states"])
    assert np.all(np.abs(s) <= 1.0) and np.mean(np.abs(s)) > 0.05
    assert not np.allclose(s[:, 0], s[:, -1])


def test_rnn_pack_is_exact(ds):
    import torch
    from speculative_decoding_draft_block_gb300.workloads import make_rnn_weights
    r, d = 128, 192
    w = make_rnn_weights(r, d, seed=3)
    dev = torch.device("cuda")
    wi = torch.from_numpy(w["w_ih"].view(np.int16)).to(dev).view(torch.bfloat16)
    wh = torch.from_numpy(w["w_hh"].view(np.int16)).to(dev).view(torch.bfloat16)
    out = torch.full((4 * r, 2 * r), 7.0, dtype=torch.bfloat16, device=dev)
    assert ds.ds_rnn_pack_weights(wi, wh, out) == 0
    torch.cuda.synchronize()
    got = out.cpu().view(torch.int16).numpy().view(np.uint16)
    want = np.zeros((4 * r, 2 * r), dtype=np.uint16)
    for t in range(r // 16):                 # blocks of 16 units, 64 rows each
        u = np.arange(16 * t, 16 * t + 16)
        blk = want[64 * t:64 * t + 64]
        blk[0:16, :r], blk[0:16, r:] = w["w_ih"][u, :r], w["w_hh"][u]
        blk[16:32, :r], blk[16:32, r:] = w["w_ih"][r + u, :r], w["w_hh"][r + u]
        blk[32:48, :r] = w["w_ih"][2 * r + u, :r]
        blk[48:64, r:] = w["w_hh"][2 * r + u]
    assert np.array_equal(got, want)


def test_rnn_matches_markov_draw_machinery_when_state_frozen(ds):
    """Update gate saturated open and s_0 = 0: the state stays zero, so every
    draw comes from the base logits alone (the oracle's frozen-state pin)."""
    import oracle
    from speculative_decoding_draft_block_gb300.workloads import make_rnn_weights
    inp = _inputs(seed=44)
    w = make_rnn_weights(64, 128, seed=8)
    w["b_hh"] = w["b_hh"].copy()
    w["b_hh"][64:128] = 60.0
    _, g = _cycle(inp, w, SEED + 1)
    assert np.all(g["states"] == 0)
    o = oracle.draft_block(inp["base_logits"], np.zeros_like(inp["E"]), inp["P"], inp["anchor"],
                           inp["temperature"], SEED + 1, prev_tokens=g["tokens"])
    mism = (o["tokens"] != g["tokens"]) & (o["margin"] >= _parity.NEAR_TIE)
    assert not mism.any()


def test_rnn_full_vocabulary_sampled_requests(ds):
    """Headline dimensions (B=128, K=16, V=151936, r=256, d=4096); the oracle
    checks every draw and state of a sample of requests."""
    from speculative_decoding_draft_block_gb300.workloads import B128, make_inputs, make_rnn_weights
    inp = make_inputs(B128)
    w = make_rnn_weights(256, 4096, seed=13)
    _, g = _cycle(inp, w, SEED + 2)
    rows = np.arange(0, 128, 16)
    rep = _parity.assert_parity(inp, g, SEED + 2, rows=rows, rnn=w)
    assert rep["draft"]["draws"] == len(rows) * 16
