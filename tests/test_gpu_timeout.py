"""A bounded device wait that runs out, through the C ABI (needs a GB300).

The failure is made without faulting or hanging anything: a test hook makes
one epilogue warp of one tile CTA withhold its arrival at the group-record
exchange of the CTA's last tile, a barrier that only epilogue threads complete.
By then every TMA copy and MMA of that CTA has completed (the epilogue already
waited for the tile's accumulator and logits), so the other threads' bounded
wait runs out, the CTA records DS_ERR_TIMEOUT, frees its tensor memory and
returns with nothing in flight. The test checks the status word, then that a
clean cycle on the same context still matches the oracle.
"""
import os

import pytest

from tests import _parity

pytestmark = pytest.mark.gpu

SEED = 0x5EED7000


@pytest.fixture(scope="module")
def lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_draft_block_gb300 import _lib, build
    if not os.path.exists(_lib.LIB_PATH):
        build.build()
    _lib.load()
    return _lib


def _inputs():
    from speculative_decoding_draft_block_gb300.workloads import B256, scaled, make_inputs
    w = scaled(B256, name="timeout", B=8, K=3, V=4096, r=64, d=64, temps=(1.0, 0.6, 0.0), seed=91)
    return make_inputs(w)


def test_withheld_arrival_times_out_and_context_survives(lib):
    import torch
    from speculative_decoding_draft_block_gb300.cycle import DeviceCycle
    inp = _inputs()
    cyc = DeviceCycle(inp)
    # the group records the timed-out CTA does not write read as zero mass
    cyc.ws_draft.zero_()
    cyc.reset_status()
    torch.cuda.synchronize()
    assert lib.ds_test_set_wait_hooks(64, 0) == 0        # ~64 polls of <= 20 us, CTA 0 withholds
    try:
        cyc.draft(SEED)
        code = lib.ds_check_status(cyc.status)
    finally:
        torch.cuda.synchronize()
        lib.ds_test_set_wait_hooks(0, -1)
    assert code == 5, lib.STATUS_NAMES.get(code, code)       # DS_ERR_TIMEOUT
    # the context is usable and the kernels are whole again: a clean cycle matches the oracle
    cyc.reset_status()
    cyc.run(SEED)
    cyc.check_status()
    _parity.assert_parity(inp, cyc.results(), SEED)


def test_hook_cleared_is_the_default(lib):
    """With the hook cleared nothing withholds: the same call reports no error."""
    from speculative_decoding_draft_block_gb300.cycle import DeviceCycle
    inp = _inputs()
    cyc = DeviceCycle(inp)
    cyc.reset_status()
    assert lib.ds_test_set_wait_hooks(0, -1) == 0
    cyc.draft(SEED)
    assert lib.ds_check_status(cyc.status) == 0
