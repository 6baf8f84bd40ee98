"""The C-ABI library builds, loads and exports every declared symbol (CPU only)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ds_draft.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ds_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_draft_block_gb300 import _lib, build
    if not os.path.exists(_lib.LIB_PATH):
        build.build()
    return _lib.load()


def test_header_declares_the_binding_exports():
    from speculative_decoding_draft_block_gb300 import _lib
    assert _declared() == sorted(_lib.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", lib._name], capture_output=True, text=True)
    if out.returncode == 0:
        syms = {l.split()[-1] for l in out.stdout.splitlines() if l.strip()}
        for name in _declared():
            assert name in syms, name


def test_host_philox_matches_oracle(lib):
    import numpy as np
    from speculative_decoding_draft_block_gb300 import _lib
    import oracle
    rng = np.random.default_rng(0)
    for _ in range(200):
        v = [int(x) for x in rng.integers(0, 2**32, size=6, dtype=np.uint64)]
        assert _lib.ds_philox4x32_10(v[:4], v[4:]) == oracle.philox4x32_10(v[:4], v[4:])
    seed = (0xDEADBEEF << 32) | 0x5EED0000
    for b in range(5):
        for k in range(1, 6):
            for s in range(3):
                assert _lib.ds_uniform(seed, b, k, s) == oracle.uniform(seed, b, k, s)


def test_workspace_sizes_and_limits(lib):
    from speculative_decoding_draft_block_gb300 import _lib
    assert _lib.ds_draft_workspace_bytes(128, 16, 151936, 256) >= 128 * 4748 * 16
    assert _lib.ds_verify_workspace_bytes(128, 16, 151936, 256) > 0
    assert _lib.ds_draft_workspace_bytes(128, 65, 151936, 256) == 0      # K > 64
    assert _lib.ds_draft_workspace_bytes(128, 16, 151937, 256) == 0      # V % 8 != 0
    assert _lib.ds_draft_workspace_bytes(1024, 17, 1024, 256) == 0       # B*K > 16384
    assert _lib.ds_sched_workspace_bytes(128, 16) == 0
    # STS fit: N samples x K positions, grid and bins within their limits
    ws = _lib.ds_sts_workspace_bytes(65536, 16, 256, 15)
    assert ws >= 4 * 4 * 65536 + 8 * 256 * 15            # prefixes + fixed-point histogram
    assert _lib.ds_sts_workspace_bytes(0, 16, 256, 15) == 0
    assert _lib.ds_sts_workspace_bytes(100, 65, 256, 15) == 0
    assert _lib.ds_sts_workspace_bytes(100, 4, 4097, 15) == 0
    assert _lib.ds_sts_workspace_bytes(100, 4, 16, 65) == 0
    assert _lib.ds_sts_workspace_bytes(1, 1, 1, 1) > 0


def test_host_validation_rejects_without_launching(lib):
    from speculative_decoding_draft_block_gb300 import _lib
    # NULL args pointer and a zeroed struct are refused on the host
    assert lib.ds_draft_block(None, None) == 1
    a = _lib.DraftArgs()
    assert lib.ds_draft_block(ctypes.byref(a), None) == 1
    assert lib.ds_verify(ctypes.byref(_lib.VerifyArgs()), None) == 1
    assert lib.ds_confidence_schedule(ctypes.byref(_lib.SchedArgs()), None) == 1
    assert lib.ds_sts_fit(ctypes.byref(_lib.StsArgs()), None) == 1
    # RNN head: checked on the host before any device work (fake, aligned, never dereferenced)
    fake = 1 << 20
    kw = dict(B=4, K=3, V=1024, r=64, base_logits=fake, E=fake, P=fake, anchor=fake,
              temperature=fake, draft_tokens=fake, q_token=fake, q_stats=fake, status=fake,
              workspace=fake, workspace_bytes=1 << 40, d=128, h=fake, rnn_w_ih=fake,
              rnn_w_step=fake, rnn_b_ih=fake, rnn_b_hh=fake, states=fake)
    assert lib.ds_draft_block(ctypes.byref(_lib.DraftArgs(dtype=0, head=1, **kw)), None) == 2
    assert lib.ds_draft_block(ctypes.byref(_lib.DraftArgs(dtype=1, head=7, **kw)), None) == 1
    kw["d"] = 100
    assert lib.ds_draft_block(ctypes.byref(_lib.DraftArgs(dtype=1, head=1, **kw)), None) == 1
    kw["d"], kw["r"] = 128, 512                  # above the tensor-core tile's r <= 256
    assert lib.ds_draft_block(ctypes.byref(_lib.DraftArgs(dtype=1, head=1, **kw)), None) == 2
    assert _lib.ds_rnn_workspace_bytes(128, 16, 512) == 0
    assert _lib.ds_rnn_workspace_bytes(128, 16, 256) >= 128 * 16 * 768 * 4 + 2 * 128 * 512 * 2
    assert _lib.ds_rnn_workspace_bytes(128, 16, 96) == 0                   # r % 64 != 0
    assert lib.ds_rnn_pack_weights(fake, fake, 64, 128, 0, fake, None) == 2  # f32 unsupported
    assert lib.ds_rnn_pack_weights(fake, fake, 96, 128, 1, fake, None) == 1
    a = _lib.StsArgs(N=4, K=2, n_grid=8, n_bins=10)      # sizes fine, pointers missing
    assert lib.ds_sts_fit(ctypes.byref(a), None) == 1
    # host staging of target rows: argument checks enqueue nothing
    lens = (ctypes.c_int32 * 4)(0, 1, 2, 3)
    n = ctypes.c_uint64(7)
    assert lib.ds_copy_scheduled_rows(None, fake, 4, 3, 64, lens, ctypes.byref(n), None) == 1
    assert lib.ds_copy_scheduled_rows(fake, None, 4, 3, 64, lens, ctypes.byref(n), None) == 1
    assert lib.ds_copy_scheduled_rows(fake, fake, 4, 3, 64, None, ctypes.byref(n), None) == 1
    assert lib.ds_copy_scheduled_rows(fake, fake, 0, 3, 64, lens, ctypes.byref(n), None) == 1
    assert lib.ds_copy_scheduled_rows(fake, fake, 4, -1, 64, lens, ctypes.byref(n), None) == 1
    assert lib.ds_copy_scheduled_rows(fake, fake, 4, 3, 0, lens, ctypes.byref(n), None) == 1
    assert n.value == 7                                  # untouched on a rejected call
    assert lib.ds_fetch_scheduled_rows(None, fake, 4, 3, 64, fake, None, None) == 1
    assert lib.ds_fetch_scheduled_rows(fake, fake, 4, 3, 24, fake, None, None) == 1  # row % 16
    assert lib.ds_fetch_scheduled_rows(fake, fake + 8, 4, 3, 64, fake, None, None) == 1  # alignment
    assert lib.ds_fetch_scheduled_rows(fake, fake, 0, 3, 64, fake, None, None) == 1
    assert _lib.ds_status_string(7) == "non-finite logit or empty distribution"
    assert _lib.ds_version() == "0.1.0"
