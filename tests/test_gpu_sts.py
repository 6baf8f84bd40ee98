"""ds_sts_fit (CUDA) against the STS oracle, through the C ABI.

DSpark summary page, 방법론 › 신뢰도 기반 검증 (STS): temperatures fitted left to
right by a 1-D grid search on ECE. The oracle's curves are evaluated with the
GPU's own fitted temperatures for the earlier positions (teacher forcing), so
a near-tie resolved differently at one position does not propagate.

Tolerances: the kernel evaluates the sigmoid in float32 with the hardware
exp2 / reciprocal (relative error ~1e-6 per factor). A sample whose float64
prediction sits within EDGE of a bin edge may fall in the neighbouring bin,
moving ECE by at most 2 |lab - pred| / N <= 2 / N; every other difference is
float rounding, bounded by ECE_ABS.
"""
import numpy as np
import pytest

import oracle
from oracle.sts import sigmoid

pytestmark = pytest.mark.gpu

ECE_ABS = 2e-5
EDGE = 2e-5


@pytest.fixture(scope="module")
def lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import os
    from speculative_decoding_draft_block_gb300 import _lib, build
    if not os.path.exists(_lib.LIB_PATH):
        build.build()
    return _lib


def _fit(lib, logits, labels, grid, n_bins, expect=0):
    import torch
    N, K = logits.shape
    G = grid.shape[0]
    dev = torch.device("cuda")
    a = torch.from_numpy(np.ascontiguousarray(logits, dtype=np.float32)).to(dev)
    y = torch.from_numpy(np.ascontiguousarray(labels, dtype=np.float32)).to(dev)
    g = torch.from_numpy(np.ascontiguousarray(grid, dtype=np.float32)).to(dev)
    T = torch.full((K,), -1.0, dtype=torch.float32, device=dev)
    idx = torch.full((K,), -7, dtype=torch.int32, device=dev)
    e = torch.full((K,), -1.0, dtype=torch.float32, device=dev)
    curve = torch.full((K, G), -1.0, dtype=torch.float32, device=dev)
    ws = torch.empty((lib.ds_sts_workspace_bytes(N, K, G, n_bins),), dtype=torch.uint8, device=dev)
    status = torch.zeros((4,), dtype=torch.int32, device=dev)
    assert lib.ds_sts_fit(a, y, g, n_bins, T, idx, e, ws, status, ece_curve=curve) == 0
    assert lib.ds_check_status(status) == expect
    return T.cpu().numpy(), idx.cpu().numpy(), e.cpu().numpy(), curve.cpu().numpy()


def _edge_counts(logits, temps, grid, n_bins):
    """[K, G] count of samples whose float64 prediction is within EDGE of a bin edge."""
    a = np.asarray(logits, dtype=np.float64)
    N, K = a.shape
    out = np.zeros((K, len(grid)), dtype=np.int64)
    base = np.ones(N)
    for k in range(K):
        for gi, T in enumerate(np.asarray(grid, dtype=np.float64)):
            x = base * sigmoid(a[:, k] / T) * n_bins
            out[k, gi] = int(np.sum(np.abs(x - np.rint(x)) < EDGE * n_bins * (k + 1)))
        base = base * sigmoid(a[:, k] / float(temps[k]))
    return out


def _check(logits, labels, grid, n_bins, got):
    T, idx, e, curve = got
    N, K = logits.shape
    grid = np.asarray(grid, dtype=np.float32)
    assert np.all((idx >= 0) & (idx < len(grid)))
    assert np.array_equal(T, grid[idx])                       # T_k is the chosen grid value
    assert np.array_equal(e, curve[np.arange(K), idx])        # its ECE is the curve's value there
    assert np.array_equal(idx, np.argmin(curve, axis=1))      # first minimum of the GPU curve
    want = oracle.sts_curves(logits, labels, grid.astype(np.float64), n_bins, T.astype(np.float64))
    tol = ECE_ABS + 2.0 * _edge_counts(logits, T, grid, n_bins) / N
    assert np.all(np.abs(curve - want) <= tol), np.max(np.abs(curve - want) - tol)
    for k in range(K):
        best = want[k].min()
        assert want[k, idx[k]] <= best + 2 * tol[k].max()
        # a clear winner must be found exactly
        order = np.sort(want[k])
        if len(order) > 1 and order[1] - order[0] > 2 * tol[k].max():
            assert idx[k] == int(np.argmin(want[k]))
    return want


def test_ragged_fit_matches_oracle(lib):
    from speculative_decoding_draft_block_gb300.workloads import make_sts_inputs, sts_grid
    d = make_sts_inputs(3001, 5, seed=31)
    grid = sts_grid(0.1, 5.0, 300)                           # two grid blocks, the second ragged
    got = _fit(lib, d["logits"], d["labels"], grid, 15)
    _check(d["logits"], d["labels"], grid, 15, got)
    assert np.all(got[0] > 1.0)                              # the raw head is over-confident


def test_exact_labels_recover_true_temperatures(lib):
    rng = np.random.default_rng(12)
    grid = np.array([0.5, 0.8, 1.0, 1.3, 2.0, 3.0], dtype=np.float32)
    t_true = np.array([0.5, 1.3, 2.0, 0.8, 3.0, 1.0], dtype=np.float32)
    a = rng.normal(1.5, 2.0, size=(5000, 6)).astype(np.float32)
    y = sigmoid(a.astype(np.float64) / t_true.astype(np.float64)[None, :]).astype(np.float32)
    T, idx, e, curve = _fit(lib, a, y, grid, 15)
    assert np.array_equal(T, t_true)
    assert np.all(e < 2e-5)


def test_limits_and_degenerate_shapes(lib):
    rng = np.random.default_rng(5)
    # one sample, one position, one grid point, one bin: ECE = |y - sigmoid(a / T)|
    a = np.array([[0.7]], dtype=np.float32)
    y = np.array([[0.25]], dtype=np.float32)
    T, idx, e, curve = _fit(lib, a, y, np.array([1.5], dtype=np.float32), 1)
    assert idx[0] == 0 and T[0] == np.float32(1.5)
    assert abs(e[0] - abs(0.25 - sigmoid(np.array([0.7 / 1.5]))[0])) < 1e-6
    # maximum bins and a large grid over a sample count that is not a multiple of 256
    a = rng.normal(0.5, 2.0, size=(700, 3)).astype(np.float32)
    y = rng.uniform(size=(700, 3)).astype(np.float32)
    grid = np.geomspace(0.05, 20.0, 1100).astype(np.float32)
    got = _fit(lib, a, y, grid, 64)
    _check(a, y, grid, 64, got)


def test_bench_size_and_determinism(lib):
    from speculative_decoding_draft_block_gb300.workloads import make_sts_inputs, sts_grid
    d = make_sts_inputs(65536, 16, seed=7)
    grid = sts_grid(0.05, 5.0, 96)
    got = _fit(lib, d["logits"], d["labels"], grid, 15)
    again = _fit(lib, d["logits"], d["labels"], grid, 15)
    for x, z in zip(got, again):
        assert np.array_equal(x, z)                          # no atomically accumulated sums
    want = _check(d["logits"], d["labels"], grid, 15, got)
    one = int(np.argmin(np.abs(grid - 1.0)))
    # the calibration lowers ECE at every position against the grid point nearest T = 1
    assert np.all(want[np.arange(16), got[1]] <= want[:, one])


def test_device_reported_input_errors(lib):
    a = np.zeros((300, 2), dtype=np.float32)
    y = np.full((300, 2), 0.5, dtype=np.float32)
    grid = np.array([0.5, 1.0, 2.0], dtype=np.float32)
    bad = y.copy()
    bad[17, 1] = 1.5                                          # label outside [0, 1]
    _fit(lib, a, bad, grid, 10, expect=1)
    nan = a.copy()
    nan[299, 0] = np.nan
    _fit(lib, nan, y, grid, 10, expect=7)
    _fit(lib, a, y, np.array([0.5, 0.0, 2.0], dtype=np.float32), 10, expect=1)


def test_confidence_schedule_emits_raw_logits(lib):
    """conf_logit = w_h.h + w_e.E[x_{k-1}] + b, the STS fit's input, from the cycle."""
    from speculative_decoding_draft_block_gb300.cycle import DeviceCycle
    from speculative_decoding_draft_block_gb300.workloads import TINY, make_inputs
    inp = make_inputs(TINY)
    cyc = DeviceCycle(inp)
    cyc.reset_status()
    cyc.draft(99)
    cyc.schedule()
    cyc.check_status()
    g = cyc.results()
    from oracle.bf16 import as_f64
    tok = g["tokens"]
    prev = np.concatenate([inp["anchor"][:, None].astype(np.int64), tok[:, :-1]], axis=1)
    raw = as_f64(inp["h"]) @ as_f64(inp["w_h"]) + as_f64(inp["E"])[prev] @ as_f64(inp["w_e"]) \
        + inp["conf_bias"]
    assert np.allclose(g["conf_logit"], raw, rtol=1e-5, atol=1e-5)
    c = sigmoid(g["conf_logit"] / inp["sts_temp"][None, :].astype(np.float64))
    assert np.allclose(c, g["conf"], rtol=2e-6, atol=1e-7)
