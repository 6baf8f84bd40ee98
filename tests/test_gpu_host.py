"""Host-resident step inputs through the C ABI (needs a GB300): the copy of the
scheduled target rows, and the pipelined host cycle against the cycle run on
resident inputs."""
import os

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

STEP_KEYS = ("base_logits", "target_logits", "anchor", "temperature", "h")


@pytest.fixture(scope="module")
def ds():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_draft_block_gb300 import _lib, build
    if not os.path.exists(_lib.LIB_PATH):
        build.build()
    _lib.load()
    import speculative_decoding_draft_block_gb300 as pkg
    return pkg


def test_copy_scheduled_rows_exact(ds):
    """Rows 0..min(max(L_b, 0), K) of each request, byte for byte; no other row."""
    import torch
    from speculative_decoding_draft_block_gb300 import _lib
    B, K, V = 6, 3, 40
    g = torch.Generator().manual_seed(3)
    src = torch.randint(-30000, 30000, (B, K + 1, V), dtype=torch.int16, generator=g).pin_memory()
    dst = torch.full((B, K + 1, V), 12345, dtype=torch.int16, device="cuda")
    lens = torch.tensor([-3, 0, 1, 2, 3, 99], dtype=torch.int32)
    code, n = _lib.ds_copy_scheduled_rows(dst, src, lens)
    assert code == 0
    torch.cuda.synchronize()
    got = dst.cpu()
    rows = [0, 0, 1, 2, 3, 3]
    assert n == sum((L + 1) * V * 2 for L in rows)
    for b, L in enumerate(rows):
        assert torch.equal(got[b, :L + 1], src[b, :L + 1])
        assert bool((got[b, L + 1:] == 12345).all())


def test_fetch_scheduled_rows_exact(ds):
    """The kernel fetch: rows 0..min(max(L_b, 0), K) of each request from pinned
    host memory, L_b read on the device, byte for byte; no other row; the
    device counter adds the bytes fetched."""
    import torch
    from speculative_decoding_draft_block_gb300 import _lib
    B, K, V = 6, 3, 40
    g = torch.Generator().manual_seed(5)
    src = torch.randint(-30000, 30000, (B, K + 1, V), dtype=torch.int16, generator=g).pin_memory()
    dst = torch.full((B, K + 1, V), 12345, dtype=torch.int16, device="cuda")
    lens = torch.tensor([-3, 0, 1, 2, 3, 99], dtype=torch.int32, device="cuda")
    counter = torch.full((1,), 7, dtype=torch.int64, device="cuda")
    assert _lib.ds_fetch_scheduled_rows(dst, src, lens, counter) == 0
    torch.cuda.synchronize()
    got = dst.cpu()
    rows = [0, 0, 1, 2, 3, 3]
    assert int(counter.item()) == 7 + sum((L + 1) * V * 2 for L in rows)
    for b, L in enumerate(rows):
        assert torch.equal(got[b, :L + 1], src[b, :L + 1])
        assert bool((got[b, L + 1:] == 12345).all())
    # a large case: several 64 KB chunks per request, a ragged last chunk
    B, K, V = 3, 4, 151936
    src = torch.randint(-30000, 30000, (B, K + 1, V), dtype=torch.int16, generator=g).pin_memory()
    dst = torch.zeros((B, K + 1, V), dtype=torch.int16, device="cuda")
    lens = torch.tensor([4, 0, 2], dtype=torch.int32, device="cuda")
    assert _lib.ds_fetch_scheduled_rows(dst, src, lens) == 0
    torch.cuda.synchronize()
    got = dst.cpu()
    for b, L in enumerate([4, 0, 2]):
        assert torch.equal(got[b, :L + 1], src[b, :L + 1])
        assert bool((got[b, L + 1:] == 0).all())


def test_fetch_of_pageable_memory(ds):
    """Pageable (not pinned) host memory: the call either refuses it before any
    launch (DS_ERR_INVALID_ARG) or, where the runtime maps it for the device,
    fetches it correctly; the context stays usable either way."""
    import ctypes
    import torch
    from speculative_decoding_draft_block_gb300 import _lib
    dst = torch.zeros((2, 2, 16), dtype=torch.int16, device="cuda")
    src = torch.arange(64, dtype=torch.int16).reshape(2, 2, 16)  # pageable
    lens = torch.zeros((2,), dtype=torch.int32, device="cuda")
    lib = _lib.load()
    code = lib.ds_fetch_scheduled_rows(ctypes.c_void_p(dst.data_ptr()), ctypes.c_void_p(src.data_ptr()),
                                       2, 1, 32, ctypes.c_void_p(lens.data_ptr()), None, None)
    torch.cuda.synchronize()
    assert code in (0, 1)
    if code == 0:
        got = dst.cpu()
        assert torch.equal(got[:, 0], src[:, 0]) and bool((got[:, 1] == 0).all())


def _group(seed_in):
    from speculative_decoding_draft_block_gb300.workloads import B256, scaled, make_inputs
    w = scaled(B256, name="host", B=37, K=5, V=3000, r=64, d=264, bf16=True,
               temps=(0.0, 0.6, 1.0), seed=seed_in)
    return make_inputs(w)


def test_host_pipeline_matches_resident_cycle(ds):
    """Two request groups served in turn, each step prefetching the next one's
    draft inputs: the emitted tokens equal those of the cycle run on fully
    resident inputs with the same key. The device buffers start as NaN, so a
    row or input the pipeline failed to copy would show."""
    import torch
    from speculative_decoding_draft_block_gb300.cycle import (DRAFT_INPUT_KEYS, DeviceCycle,
                                                               HostPipeline, to_host_pinned)
    a = _group(31)
    b = dict(a)
    other = _group(32)
    for k in STEP_KEYS:  # same weights, other requests
        b[k] = other[k]
    steps = [(a, 0x1001), (b, 0x1002), (a, 0x1003), (b, 0x1004)]

    expect = []
    for inp, seed in steps:
        ref = DeviceCycle(inp)
        ref.reset_status()
        ref.run(seed)
        ref.check_status()
        expect.append((ref.out_tokens.cpu().numpy(), ref.num_emitted.cpu().numpy()))

    cyc = DeviceCycle(a)
    pipe = HostPipeline(cyc)
    for slot in pipe.slots:
        for k in DRAFT_INPUT_KEYS:
            if slot[k].is_floating_point():
                slot[k].fill_(float("nan"))
    cyc.t["target_logits"].fill_(float("nan"))
    hosts = [{k: to_host_pinned(inp[k]) for k in STEP_KEYS} for inp, _ in steps]
    cyc.reset_status()
    for i, (_, seed) in enumerate(steps):
        nxt = hosts[i + 1] if i + 1 < len(steps) else None
        _, out, nem, done = pipe.step(hosts[i], seed, next_host=nxt)
        done.synchronize()
        out, nem = out.numpy().copy(), nem.numpy().copy()
        eo, en = expect[i]
        assert np.array_equal(nem, en), i
        for r in range(out.shape[0]):
            assert np.array_equal(out[r, :nem[r]], eo[r, :en[r]]), (i, r)
    cyc.check_status()
    assert pipe.h2d_bytes() > 0
    # the resident binding is restored after each step
    assert all(cyc.t[k] is pipe.slots[0][k] for k in DRAFT_INPUT_KEYS)
