"""ds_acceptance_rate (CUDA) against the oracle, through the C ABI, and the
STS fit supervised by it (needs a GB300).

DSpark summary page, 방법론 › 신뢰도 기반 검증: the STS temperatures are fitted
against the analytic acceptance 1 - TV(p_k, q_k) = sum_i min(p_k(i), q_k(i));
배경 gives the accept rule whose success probability that is. Tolerance: 2e-3
relative, the bar for probabilities (the kernel computes in float32).
"""
import numpy as np
import pytest

import oracle
from tests import test_gpu_sts as sts_t

pytestmark = pytest.mark.gpu

REL_TOL = 2e-3


@pytest.fixture(scope="module")
def lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import os
    from speculative_decoding_draft_block_gb300 import _lib, build
    if not os.path.exists(_lib.LIB_PATH):
        build.build()
    _lib.load()
    return _lib


def _rows(n, V, seed, bf16, temps=(0.0, 0.6, 1.0, 1.5), mask_every=0):
    """Draft rows ~ N(0, 1.5^2) with a +5 bump on a true token, target = draft +
    per-row noise of sigma in [0.2, 1.5] (the workloads' recipe), rounded to
    bfloat16 when asked."""
    rng = np.random.default_rng(seed)
    d = rng.normal(0, 1.5, size=(n, V)).astype(np.float32)
    d[np.arange(n), rng.integers(0, V, size=n)] += 5.0
    sig = rng.uniform(0.2, 1.5, size=(n, 1)).astype(np.float32)
    t = (d + rng.normal(0, 1.0, size=(n, V)).astype(np.float32) * sig).astype(np.float32)
    if mask_every:
        d[:, ::mask_every] = -np.inf
        t[:, ::mask_every] = -np.inf
    T = np.array([temps[i % len(temps)] for i in range(n)], dtype=np.float32)
    if bf16:
        def rnd(x):
            u = x.view(np.uint32).astype(np.uint64)
            u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
            return u.astype(np.uint16)
        return rnd(t), rnd(d), T
    return t, d, T


def _gpu_alpha(lib, t, d, T, expect=0):
    import torch
    from speculative_decoding_draft_block_gb300.cycle import _to_device
    tt, dd = _to_device(t, "cuda"), _to_device(d, "cuda")
    Td = torch.from_numpy(T).cuda()
    alpha = torch.full((t.shape[0],), -1.0, dtype=torch.float32, device="cuda")
    status = torch.zeros((4,), dtype=torch.int32, device="cuda")
    assert lib.ds_acceptance_rate(tt, dd, Td, alpha, status) == 0
    assert lib.ds_check_status(status) == expect
    return alpha.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("bf16,V,mask", [(True, 4096, 0), (False, 4096, 0), (True, 1000, 0),
                                         (True, 2048, 5), (False, 151936, 0)])
def test_matches_oracle(lib, bf16, V, mask):
    n = 8 if V > 100000 else 96
    t, d, T = _rows(n, V, 7 + V + mask, bf16, mask_every=mask)
    got = _gpu_alpha(lib, t, d, T)
    want = oracle.acceptance_rate(t, d, T)
    greedy = T == 0
    assert np.array_equal(got[greedy], want[greedy])
    s = ~greedy
    rel = np.abs(got[s] - want[s]) / np.maximum(want[s], 1e-6)
    assert rel.max() < REL_TOL, (rel.max(), want[s].min())
    assert np.all((got >= 0) & (got <= 1))


def test_special_rows(lib):
    V = 512
    rng = np.random.default_rng(2)
    t = rng.normal(size=(3, V)).astype(np.float32)
    d = t.copy()
    d[1] = -np.inf
    d[1, :V // 2] = 0.0
    t[1] = -np.inf
    t[1, V // 2:] = 0.0
    T = np.array([1.0, 1.0, 0.0], dtype=np.float32)
    got = _gpu_alpha(lib, t, d, T)
    assert abs(got[0] - 1.0) < 1e-5          # p = q
    assert got[1] == 0.0                     # disjoint supports
    assert got[2] == 1.0                     # same argmax


def test_device_errors(lib):
    t, d, T = _rows(4, 512, 3, False)
    t[2, 7] = np.nan
    _gpu_alpha(lib, t, d, T, expect=7)
    t, d, T = _rows(4, 512, 3, False)
    T[1] = -2.0
    _gpu_alpha(lib, t, d, T, expect=1)


def test_sts_fit_supervised_by_the_acceptance_rate(lib):
    """Soft labels from ds_acceptance_rate feed ds_sts_fit; the fit matches the
    oracle's fit on the same logits, curves compared within the STS test's
    tolerances (the oracle evaluates with the GPU's labels and temperatures)."""
    N, K, V = 2048, 4, 512
    t, d, T = _rows(N * K, V, 11, True, temps=(1.0,))
    alpha = _gpu_alpha(lib, t, d, T).reshape(N, K)
    want = oracle.acceptance_rate(t, d, T).reshape(N, K)
    assert np.max(np.abs(alpha - want) / want) < REL_TOL
    # an over-confident raw head: logits 2.2x the calibrated logit of alpha, plus noise
    rng = np.random.default_rng(12)
    a = (2.2 * np.log(alpha / np.maximum(1 - alpha, 1e-6)) + rng.normal(0, 0.3, size=(N, K))).astype(np.float32)
    labels = alpha.astype(np.float32)
    grid = np.geomspace(0.2, 5.0, 64).astype(np.float32)
    got = sts_t._fit(lib, a, labels, grid, 10)
    sts_t._check(a, labels, grid, 10, got)
    # the fitted temperatures undo the over-confidence (close to 2.2 at every position)
    assert np.all((got[0] > 1.4) & (got[0] < 3.4)), got[0]
