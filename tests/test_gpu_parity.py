"""GPU cycle vs the oracle, through the C ABI (needs a GB300).

Sizes: the tiny workload and ragged multi-tile cases are compared in full; the
full-size workloads are compared on every draw (B32, B128) or on a sample of
requests (B512, B256), always with the oracle teacher-forced on the GPU's own
prefix so every draw is checked on its own.
"""
import json
import os

import numpy as np
import pytest

from tests import _parity

pytestmark = pytest.mark.gpu

SEED = 0x5EED0000


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


def _run(inp, seed=SEED, **kw):
    from speculative_decoding_draft_block_gb300.cycle import DeviceCycle
    cyc = DeviceCycle(inp, **kw)
    cyc.reset_status()
    cyc.run(seed)
    cyc.check_status()
    return cyc, cyc.results()


def test_philox_device_words(ds):
    import torch
    import oracle
    from speculative_decoding_draft_block_gb300 import _lib
    n = 1 << 20
    rng = np.random.default_rng(0)
    ctr = rng.integers(0, 2**32, size=(n, 4), dtype=np.uint64).astype(np.uint32)
    key = (0x89ABCDEF, 0x01234567)
    ct = torch.from_numpy(ctr.view(np.int32)).cuda()
    out = torch.zeros_like(ct)
    assert _lib.ds_philox_fill(ct, key[0], key[1], out) == 0
    torch.cuda.synchronize()
    got = out.cpu().numpy().view(np.uint32)
    # vectorised Philox4x32-10 in NumPy (third implementation, for the bulk)
    c = [ctr[:, i].astype(np.uint64) for i in range(4)]
    k0, k1 = np.uint64(key[0]), np.uint64(key[1])
    M = np.uint64(0xFFFFFFFF)
    for rnd in range(10):
        if rnd:
            k0 = (k0 + np.uint64(0x9E3779B9)) & M
            k1 = (k1 + np.uint64(0xBB67AE85)) & M
        p0 = np.uint64(0xD2511F53) * c[0]
        p1 = np.uint64(0xCD9E8D57) * c[2]
        c = [((p1 >> np.uint64(32)) ^ c[1] ^ k0) & M, p1 & M, ((p0 >> np.uint64(32)) ^ c[3] ^ k1) & M, p0 & M]
    want = np.stack(c, axis=1).astype(np.uint32)
    assert np.array_equal(got, want)
    for i in range(0, n, n // 500):
        assert tuple(got[i]) == oracle.philox4x32_10(ctr[i], key)


def test_tiny_cycle(ds):
    from speculative_decoding_draft_block_gb300.workloads import TINY, make_inputs
    inp = make_inputs(TINY)
    _, g = _run(inp)
    rep = _parity.assert_parity(inp, g, SEED)
    gold = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "tiny_cycle.json")))
    assert rep["draft"]["near_ties"] == 0
    assert g["tokens"].tolist() == gold["draft_tokens"]
    assert g["L"].tolist() == gold["sched_len"]
    assert g["accept_count"].tolist() == gold["accept_count"]
    assert g["out_tokens"].tolist() == gold["out_tokens"]


def _ragged(bf16, temps, seed_in, B=37, K=5, V=3000, r=48, d=264, **kw):
    from speculative_decoding_draft_block_gb300.workloads import B256, scaled, make_inputs
    w = scaled(B256, name="ragged", B=B, K=K, V=V, r=r, d=d, bf16=bf16, temps=temps,
               seed=seed_in, **kw)
    return make_inputs(w)


@pytest.mark.parametrize("bf16", [True, False])
def test_ragged_multitile_mixed_temperatures(ds, bf16):
    inp = _ragged(bf16, (0.0, 0.6, 1.0), 7)
    _, g = _run(inp)
    rep = _parity.assert_parity(inp, g, SEED)
    assert rep["draft"]["draws"] == 37 * 5


@pytest.mark.parametrize("bf16", [True, False])
def test_ragged_all_greedy(ds, bf16):
    """Every request greedy (T = 0): each draw is the exact argmax of z + b,
    first index on ties, on every row of a ragged multi-tile case."""
    inp = _ragged(bf16, (0.0,), 29)
    _, g = _run(inp)
    rep = _parity.assert_parity(inp, g, SEED)
    assert rep["draft"]["draws"] == 37 * 5


@pytest.mark.parametrize("bf16", [True, False])
def test_ragged_strided_projection(ds, bf16):
    """The draw without the token-major copy of P (r strided rows per chunk)."""
    inp = _ragged(bf16, (0.0, 0.6, 1.0), 17, r=64)
    _, g = _run(inp, token_major_projection=False)
    rep = _parity.assert_parity(inp, g, SEED)
    assert rep["draft"]["draws"] == 37 * 5


@pytest.mark.parametrize("bf16", [True, False])
def test_transpose_projection_exact(ds, bf16):
    import torch
    from speculative_decoding_draft_block_gb300 import _lib
    from speculative_decoding_draft_block_gb300.cycle import _to_device
    for r, V in ((48, 3000), (64, 4096), (16, 8), (256, 1032)):
        rng = np.random.default_rng(r * 7 + V)
        P = rng.standard_normal((r, V), dtype=np.float32)
        if bf16:
            P = P.view(np.uint32).__rshift__(16).astype(np.uint16)
        Pd = _to_device(P, "cuda")
        Pt = torch.empty((V, r), dtype=Pd.dtype, device="cuda")
        assert _lib.ds_transpose_projection(Pd, Pt) == 0
        torch.cuda.synchronize()
        got = Pt.view(torch.int16 if bf16 else torch.float32).cpu().numpy()
        want = P.T.view(np.int16) if bf16 else P.T
        assert np.array_equal(got, want)


@pytest.mark.parametrize("r,V", [(256, 4096), (64, 3000), (192, 1032), (128, 8)])
def test_pack_projection_exact(ds, r, V):
    """The tile-packed copy of P: for tile nt, k-block c, half h, row m, the
    16-byte unit u of P[c*64 + m][nt*128 + h*64 + 8u ...] sits at unit
    u ^ (m % 8) of its 128-byte row; tokens past V are zero (layout restated
    here with NumPy)."""
    import torch
    from speculative_decoding_draft_block_gb300 import _lib
    from speculative_decoding_draft_block_gb300.cycle import _to_device
    rng = np.random.default_rng(r + V)
    P = (rng.standard_normal((r, V), dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)
    nbytes = _lib.ds_packed_projection_bytes(r, V)
    n_nt = (V + 127) // 128
    assert nbytes == n_nt * (r // 64) * 16384
    out = torch.zeros((nbytes,), dtype=torch.uint8, device="cuda")
    assert _lib.ds_pack_projection(_to_device(P, "cuda"), out) == 0
    torch.cuda.synchronize()
    got = out.cpu().numpy().view(np.uint16).reshape(n_nt, r // 64, 2, 64, 8, 8)
    Pp = np.zeros((r, n_nt * 128), dtype=np.uint16)
    Pp[:, :V] = P
    # want[nt, c, h, m, u_stored, 8 tokens]
    src = Pp.reshape(r // 64, 64, n_nt, 2, 8, 8).transpose(2, 0, 3, 1, 4, 5)  # nt, c, h, m, u, e
    want = np.empty_like(src)
    for m in range(64):
        for u in range(8):
            want[:, :, :, m, u ^ (m % 8), :] = src[:, :, :, m, u, :]
    assert np.array_equal(got, want)


@pytest.mark.parametrize("bf16", [True])
def test_ragged_tensor_copies_of_projection(ds, bf16):
    """The tensor-core tile fed by per-row tensor copies of P (no packed copy)."""
    inp = _ragged(bf16, (0.0, 0.6, 1.0), 37, B=37, K=5, V=3000, r=64, d=64)
    _, g = _run(inp, packed_projection=False)
    rep = _parity.assert_parity(inp, g, SEED)
    assert rep["draft"]["draws"] == 37 * 5


def test_full_size_without_packed_projection(ds):
    from speculative_decoding_draft_block_gb300.workloads import WORKLOADS, make_inputs
    inp = make_inputs(WORKLOADS["B32_K8_V151936"])
    _, g = _run(inp, packed_projection=False)
    _parity.assert_parity(inp, g, SEED)


def test_independent_cycle_matches_oracle_cycle(ds):
    """No teacher forcing: the oracle's own cycle and the GPU's agree end to end.

    Each request's drafted tokens are compared up to its first near-tie draw
    (after it the two may diverge legitimately). The schedule is compared when
    no draft draw anywhere was a near tie (it reads every request's survivals),
    and each request's verify outcome when, in addition, none of its own verify
    decisions is a near tie."""
    import oracle
    inp = _ragged(True, (0.0, 1.0), 11, B=16, K=6, V=4096, r=64, d=128)
    _, g = _run(inp)
    o = oracle.cycle(inp, SEED)
    B, K = inp["B"], inp["K"]
    near = o["draft"]["margin"] < _parity.NEAR_TIE
    compared = 0
    for b in range(B):
        k0 = int(np.argmax(near[b])) if near[b].any() else K
        assert np.array_equal(o["draft"]["tokens"][b, :k0], g["tokens"][b, :k0]), b
        compared += k0
    assert compared >= 0.75 * B * K, compared
    if near.any():
        return
    sch = o["schedule"]
    if min(sch["stop_rel_gain"], sch["survival_gap"]) >= _parity.SCHED_NEAR_TIE:
        assert np.array_equal(sch["L"], g["L"])
    else:
        return
    checked = 0
    for b in range(B):
        if all(m >= _parity.NEAR_TIE for _, m in o["verify"]["decisions"][b]):
            assert np.array_equal(o["verify"]["out_tokens"][b], g["out_tokens"][b]), b
            checked += 1
    assert checked >= B // 2, checked


def test_masked_tokens_never_drawn(ds):
    inp = _ragged(True, (1.0, 0.6), 13, B=8, K=4, V=2048, r=32, d=64)
    mask = np.zeros(inp["V"], dtype=bool)
    mask[::3] = True
    ninf = np.uint16(0xFF80)                     # bfloat16 -inf
    inp["base_logits"][:, :, mask] = ninf
    inp["target_logits"][:, :, mask] = ninf
    _, g = _run(inp)
    assert not np.any(mask[g["tokens"]])
    emitted = g["out_tokens"][g["out_tokens"] >= 0]
    assert not np.any(mask[emitted])
    _parity.assert_parity(inp, g, SEED)


def test_schedule_modes(ds):
    from speculative_decoding_draft_block_gb300 import _lib
    import oracle
    inp = _ragged(True, (1.0,), 17, B=12, K=5, V=1024, r=32, d=64)
    _, g = _run(inp, mode=_lib.DS_SCHED_FIXED_K)
    assert np.all(g["L"] == 5)
    _parity.assert_parity(inp, g, SEED, check_schedule=False)
    _, g = _run(inp, mode=_lib.DS_SCHED_THRESHOLD, threshold=0.5)
    s = oracle.survival(oracle.confidence(inp["h"], inp["E"], inp["anchor"], g["tokens"], inp["w_h"],
                                          inp["w_e"], inp["conf_bias"], inp["sts_temp"]))
    want = oracle.schedule(s, inp["sps"], mode=oracle.SCHED_THRESHOLD, threshold=0.5)["L"]
    assert np.array_equal(g["L"], want)
    # threshold above every survival: nothing scheduled, bonus from row 1
    _, g = _run(inp, mode=_lib.DS_SCHED_THRESHOLD, threshold=2.0)
    assert np.all(g["L"] == 0) and np.all(g["num_emitted"] == 1)
    _parity.assert_parity(inp, g, SEED, check_schedule=False)


def _selection_size(survival):
    """The scheduler's selection on the host (tests/test_sched_network.py):
    how many top candidates it sorts before falling back to every key."""
    from tests.test_sched_network import _select
    surv = [float(x) for x in survival.reshape(-1)]
    B = survival.shape[0]
    cap = 256
    while cap < 4 * B and cap < 1024:
        cap *= 2
    return max(_select(surv, cap)[0], _select(surv, 1024)[0])


@pytest.mark.parametrize("case", ["stop_past_selection", "one_bin", "async_budget_past_selection",
                                  "second_tier", "async_budget_inside_selection"])
def test_schedule_sorts_every_key_past_the_selection(ds, case):
    """B*K = 2048 candidates where the early stop (or the asynchronous budget)
    lies beyond the top bins the scheduler sorts first, or every survival
    sits in one bin: the full sort runs, and its order decides sched_len.
    Also a stop past the first selection (at most 4B = 512 candidates) but
    inside the second (at most 1024), and an asynchronous budget inside the
    selection."""
    from speculative_decoding_draft_block_gb300 import _lib
    import oracle
    inp = _ragged(True, (1.0,), 29, B=128, K=16, V=1024, r=32, d=64)
    n_max = len(inp["sps"])
    if case == "one_bin":
        inp["conf_bias"] = 60.0  # c rounds to 1 in float32: every survival is 1
    elif case == "second_tier":
        # J = A while N <= 828, then 828 A / N: the stop falls near 700 candidates
        inp["sps"] = np.minimum(np.arange(1, n_max + 1), 128 + 700).astype(np.float32)
    elif case == "async_budget_inside_selection":
        pass
    else:
        # J = A while N <= 1700, then 1700 A / N: the stop falls near N = 1700,
        # past any selection of at most 1024 candidates
        inp["sps"] = np.minimum(np.arange(1, n_max + 1), 1700).astype(np.float32)
    kw = {}
    budget = {"async_budget_past_selection": 1500, "async_budget_inside_selection": 300}.get(case)
    if budget is not None:
        kw = dict(mode=_lib.DS_SCHED_ASYNC, initial_budget=budget)
    _, g = _run(inp, **kw)
    c = oracle.confidence(inp["h"], inp["E"], inp["anchor"], g["tokens"], inp["w_h"], inp["w_e"],
                          inp["conf_bias"], inp["sts_temp"])
    s = oracle.survival(c)
    if budget is not None:
        if budget == 1500:
            assert _selection_size(g["survival"]) < budget
        else:
            assert _selection_size(g["survival"]) > budget
        want = oracle.schedule(s, inp["sps"], mode=oracle.SCHED_ASYNC, budget=budget)
        assert int(g["L"].sum()) == budget
        top = np.sort(s.ravel())[::-1]
        if (top[budget - 1] - top[budget]) > _parity.SCHED_NEAR_TIE * top[budget - 1]:
            assert np.array_equal(g["L"], want["L"])
    else:
        want = oracle.schedule(s, inp["sps"])
        M = int(want["n_included"])
        if case == "one_bin":
            assert _selection_size(g["survival"]) == 0 and np.all(g["survival"] == 1.0)
            assert np.all(g["L"] == 16)
        elif case == "second_tier":
            from tests.test_sched_network import _select
            surv = [float(x) for x in g["survival"].reshape(-1)]
            assert _select(surv, 512)[0] <= M < _select(surv, 1024)[0]
        else:
            assert _selection_size(g["survival"]) < M < 2048
        if min(want["stop_rel_gain"], want["survival_gap"]) >= _parity.SCHED_NEAR_TIE:
            assert np.array_equal(g["L"], want["L"])
    _parity.assert_parity(inp, g, SEED, check_schedule=False)


def test_async_scheduler_over_cycles(ds):
    """Budget from two cycles back (device ring), dynamic top-k on the current
    survivals; each cycle compared with the oracle's asynchronous schedule."""
    from speculative_decoding_draft_block_gb300 import _lib
    from speculative_decoding_draft_block_gb300.cycle import DeviceCycle
    import oracle
    inp = _ragged(True, (1.0, 0.6), 23, B=24, K=6, V=2048, r=64, d=128)
    B, K = inp["B"], inp["K"]
    cyc = DeviceCycle(inp, mode=_lib.DS_SCHED_ASYNC, initial_budget=17)
    counts, near = [], []
    for t in range(5):
        budget = int(cyc.budget_ring.cpu()[t & 1])       # what the device will use
        want_budget = 17 if t < 2 else counts[t - 2]
        assert budget == want_budget or near[t - 2]
        cyc.reset_status()
        cyc.run(SEED + t)
        cyc.check_status()
        g = cyc.results()
        s = oracle.survival(oracle.confidence(inp["h"], inp["E"], inp["anchor"], g["tokens"],
                                              inp["w_h"], inp["w_e"], inp["conf_bias"],
                                              inp["sts_temp"]))
        greedy = oracle.schedule(s, inp["sps"])
        counts.append(greedy["n_included"])
        near.append(min(greedy["stop_rel_gain"], greedy["survival_gap"]) < _parity.SCHED_NEAR_TIE)
        want = oracle.schedule(s, inp["sps"], mode=oracle.SCHED_ASYNC, budget=budget)
        assert int(g["L"].sum()) == min(budget, B * K)        # fixed verify batch
        top = np.sort(s.ravel())[::-1]
        m = min(budget, B * K)
        boundary_tie = 0 < m < B * K and (top[m - 1] - top[m]) <= _parity.SCHED_NEAR_TIE * top[m - 1]
        if not boundary_tie:
            assert np.array_equal(g["L"], want["L"])
            assert abs(g["objective"] - want["objective"]) <= 1e-5 * want["objective"]
        _parity.assert_parity(inp, g, SEED + t, check_schedule=False)
    # the ring holds the last two cycles' early-stop counts
    ring = cyc.budget_ring.cpu().numpy().tolist()
    assert ring[2] == 5                                  # the device cycle counter
    assert sorted(ring[:2]) == sorted(counts[-2:]) or near[-1] or near[-2]


def test_cycle_replays_from_a_cuda_graph(ds):
    """A whole cycle (draft, asynchronous schedule, verify, and the key's
    advance) captured once into a CUDA graph and replayed: each replay equals a
    direct run with the same key and ring state (the per-cycle state lives on
    the device: the Philox key word and the scheduler's ring)."""
    import torch
    from speculative_decoding_draft_block_gb300 import _lib
    from speculative_decoding_draft_block_gb300.cycle import DeviceCycle
    inp = _ragged(True, (0.0, 0.6, 1.0), 31, B=24, K=6, V=4096, r=64, d=128)
    kw = dict(mode=_lib.DS_SCHED_ASYNC, initial_budget=17, device_seed=True)
    ref = DeviceCycle(inp, **kw)
    cyc = DeviceCycle(inp, **kw)
    cyc.set_seed(1)                      # one-time library set-up outside the capture
    cyc.run(0)
    torch.cuda.synchronize()
    cyc.reset_ring()
    cyc.reset_status()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            cyc.run(0)
            cyc.seed_dev[0].add_(1)
    torch.cuda.synchronize()
    cyc.set_seed(SEED)
    prev = None
    for t in range(4):
        graph.replay()
        torch.cuda.synchronize()
        got = cyc.results()
        ref.set_seed(SEED + t)
        ref.run(0)
        torch.cuda.synchronize()
        want = ref.results()
        for key in ("tokens", "L", "out_tokens", "accept_count", "q_token"):
            assert np.array_equal(got[key], want[key]), (t, key)
        assert np.array_equal(cyc.budget_ring.cpu().numpy(), ref.budget_ring.cpu().numpy())
        if prev is not None:
            assert not np.array_equal(got["tokens"], prev)  # a fresh key every replay
        prev = got["tokens"]
    cyc.check_status()
    ref.check_status()


def test_minimal_shapes(ds):
    inp = _ragged(True, (1.0,), 19, B=1, K=1, V=8, r=16, d=8)
    _, g = _run(inp)
    _parity.assert_parity(inp, g, SEED)


@pytest.mark.parametrize("B,K,V,r,bf16,rows", [
    (8, 64, 4096, 64, True, None),      # K at its limit: 64 sequential steps (tensor-core tile)
    (256, 64, 1024, 64, True, 24),      # B*K at its limit (16384 drafted tokens)
    (5, 3, 2048, 1024, True, None),     # r at its limit (SIMT tile: A rows wider than 256)
    (4, 2, 1024, 1024, False, None),    # r at its limit, float32
    (1536, 2, 1024, 64, True, 32),      # more requests than scheduler threads (sort network, no merge tree)
])
def test_limit_shapes(ds, B, K, V, r, bf16, rows):
    inp = _ragged(bf16, (0.0, 0.6, 1.0), 29 + K, B=B, K=K, V=V, r=r, d=64)
    _, g = _run(inp)
    sel = None if rows is None else np.linspace(0, B - 1, rows).astype(np.int64)
    rep = _parity.assert_parity(inp, g, SEED, rows=sel)
    assert rep["draft"]["draws"] == (B if rows is None else rows) * K


def test_device_errors_are_reported(ds):
    from speculative_decoding_draft_block_gb300 import _lib
    from speculative_decoding_draft_block_gb300.cycle import DeviceCycle
    inp = _ragged(True, (1.0,), 23, B=4, K=3, V=512, r=16, d=16)
    bad = dict(inp)
    bad["base_logits"] = inp["base_logits"].copy()
    bad["base_logits"][1, 0, 5] = np.uint16(0x7FC0)          # NaN
    cyc = DeviceCycle(bad)
    cyc.reset_status()
    cyc.run(SEED)
    assert _lib.ds_check_status(cyc.status) == 7
    bad = dict(inp)
    bad["anchor"] = inp["anchor"].copy()
    bad["anchor"][2] = inp["V"] + 5
    cyc = DeviceCycle(bad)
    cyc.reset_status()
    cyc.run(SEED)
    assert _lib.ds_check_status(cyc.status) == 6
    bad = dict(inp)
    bad["temperature"] = np.array([1.0, -1.0, 1.0, 1.0], dtype=np.float32)
    cyc = DeviceCycle(bad)
    cyc.reset_status()
    cyc.run(SEED)
    assert _lib.ds_check_status(cyc.status) == 1
    # the context is still usable: a clean cycle afterwards succeeds
    _, g = _run(inp)
    _parity.assert_parity(inp, g, SEED)


@pytest.mark.parametrize("name,rows", [
    ("B32_K8_V151936", None),
    ("B128_K16_V151936", None),
    ("B512_K16_V129280", 24),
    ("B256_K32_V151936", 24),
])
def test_full_size_workloads(ds, name, rows):
    from speculative_decoding_draft_block_gb300.workloads import WORKLOADS, make_inputs
    inp = make_inputs(WORKLOADS[name])
    _, g = _run(inp)
    sel = None
    if rows is not None:
        sel = np.linspace(0, inp["B"] - 1, rows).astype(np.int64)
    rep = _parity.assert_parity(inp, g, SEED, rows=sel)
    print(name, json.dumps(rep))


@pytest.mark.parametrize("case", ["tiny", "ragged_bf16", "ragged_f32", "k_limit", "r_limit_f32",
                                  "B128_K16_V151936"])
def test_no_write_outside_the_buffers(ds, case):
    """Every buffer the library writes (outputs, workspaces, the token-major P
    copy, the scheduler ring) sits between guard regions of sentinel bytes;
    after a cycle, and after two cycles with the asynchronous scheduler, the
    guards are intact, and the guarded cycle still matches the oracle. A
    stand-in for a memory checker, which this pool does not offer."""
    from speculative_decoding_draft_block_gb300 import _lib
    from speculative_decoding_draft_block_gb300.workloads import TINY, WORKLOADS, make_inputs
    if case == "tiny":
        inp = make_inputs(TINY)
    elif case == "ragged_bf16":
        inp = _ragged(True, (0.0, 0.6, 1.0), 41)
    elif case == "ragged_f32":
        inp = _ragged(False, (0.0, 0.6, 1.0), 43)
    elif case == "k_limit":
        inp = _ragged(True, (0.0, 1.0), 45, B=8, K=64, V=4096, r=64, d=64)
    elif case == "r_limit_f32":
        inp = _ragged(False, (0.6, 1.0), 47, B=5, K=3, V=2048, r=1024, d=64)
    else:
        inp = make_inputs(WORKLOADS[case])
    cyc, g = _run(inp, guards=True)
    assert cyc.guard_damage() == [], case
    rows = None if inp["B"] <= 64 else np.linspace(0, inp["B"] - 1, 16).astype(np.int64)
    _parity.assert_parity(inp, g, SEED, rows=rows)
    cyc, _ = _run(inp, mode=_lib.DS_SCHED_ASYNC, guards=True)
    cyc.reset_status()
    cyc.run(SEED + 1)
    cyc.check_status()
    assert cyc.guard_damage() == [], (case, "async")


def test_rnn_head_writes_nothing_outside_its_buffers(ds):
    from speculative_decoding_draft_block_gb300.workloads import make_rnn_weights
    inp = _ragged(True, (0.0, 0.6, 1.0), 49, B=20, K=4, V=4096, r=64, d=128)
    cyc, _ = _run(inp, guards=True, rnn_weights=make_rnn_weights(64, 128))
    assert cyc.guard_damage() == []
