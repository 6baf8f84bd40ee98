"""ds_verify_static (library-owned scratch) against ds_verify (caller workspace).

Collected last on purpose (file name): it must pass both alone and after the
other GPU tests, since its scratch array lives as long as the loaded module.
"""
import ctypes
import os

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

SEED = 0x5EED4000


@pytest.fixture(scope="module")
def lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_draft_block_gb300 import _lib, build
    if not os.path.exists(_lib.LIB_PATH):
        build.build()
    return _lib


def _inputs():
    from speculative_decoding_draft_block_gb300.workloads import B256, scaled, make_inputs
    w = scaled(B256, name="no_alloc", B=64, K=8, V=32768, r=64, d=128, temps=(0.0, 0.6, 1.0),
               seed=4242)
    return make_inputs(w)


def _verify_outputs(cyc, lib, seed, static):
    import torch
    t = cyc.t
    out = torch.full_like(cyc.out_tokens, -7)
    acc = torch.full_like(cyc.accept_count, -7)
    nem = torch.full_like(cyc.num_emitted, -7)
    cyc.reset_status()
    args = (t["target_logits"], t["base_logits"], t["E"], t["P"], t["anchor"], cyc.draft_tokens,
            cyc.q_token, cyc.q_stats, cyc.sched_len, t["temperature"], seed, out, acc, nem)
    if static:
        code = lib.ds_verify_static(*args, cyc.status, P_t=cyc.P_t)
    else:
        code = lib.ds_verify(*args, cyc.ws_verify, cyc.status, P_t=cyc.P_t)
    assert code == 0
    assert lib.ds_check_status(cyc.status) == 0
    return out.cpu().numpy(), acc.cpu().numpy(), nem.cpu().numpy()


def test_static_scratch_matches_workspace_entry_point(lib):
    from speculative_decoding_draft_block_gb300.cycle import DeviceCycle
    inp = _inputs()
    cyc = DeviceCycle(inp)
    cyc.reset_status()
    cyc.draft(SEED)
    cyc.schedule()
    cyc.check_status()
    want = _verify_outputs(cyc, lib, SEED, static=False)
    for _ in range(2):                      # two calls in a row reuse the same scratch
        got = _verify_outputs(cyc, lib, SEED, static=True)
        for g, w in zip(got, want):
            assert np.array_equal(g, w)     # token ids and counts: exact
    assert (want[2] == want[1] + 1).all()


def test_static_scratch_rejects_oversized_calls(lib):
    L = lib.load()
    limit = 16 << 20
    B, K, V, r = 512, 16, 129280, 256
    assert lib.ds_verify_workspace_bytes(B, K, V, r) > limit
    a = lib.VerifyArgs(B=B, K=K, V=V, r=r, dtype=1)
    assert L.ds_verify_static(ctypes.byref(a), None) == 3      # DS_ERR_WORKSPACE, nothing launched


def test_static_scratch_with_rnn_states(lib):
    """The RNN head's states reach the residual draw through the static entry point too."""
    from speculative_decoding_draft_block_gb300.cycle import DeviceCycle
    from speculative_decoding_draft_block_gb300.workloads import make_rnn_weights
    inp = _inputs()
    cyc = DeviceCycle(inp, rnn_weights=make_rnn_weights(inp["r"], inp["d"], seed=9))
    cyc.reset_status()
    cyc.draft(SEED + 1)
    cyc.schedule()
    cyc.check_status()
    import torch
    t = cyc.t
    outs = []
    for static in (False, True):
        out = torch.full_like(cyc.out_tokens, -7)
        acc = torch.full_like(cyc.accept_count, -7)
        nem = torch.full_like(cyc.num_emitted, -7)
        cyc.reset_status()
        args = (t["target_logits"], t["base_logits"], t["E"], t["P"], t["anchor"], cyc.draft_tokens,
                cyc.q_token, cyc.q_stats, cyc.sched_len, t["temperature"], SEED + 1, out, acc, nem)
        if static:
            code = lib.ds_verify_static(*args, cyc.status, P_t=cyc.P_t, states=cyc.rnn["states"])
        else:
            code = lib.ds_verify(*args, cyc.ws_verify, cyc.status, P_t=cyc.P_t, states=cyc.rnn["states"])
        assert code == 0
        assert lib.ds_check_status(cyc.status) == 0
        outs.append((out.cpu().numpy(), acc.cpu().numpy()))
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])
