"""Sequential Temperature Scaling (STS) fit, float64 (test infrastructure only).

DSpark summary page, 방법론 › 신뢰도 기반 검증 (the STS paragraph), and
주요 결과 (raw confidences discriminate well but are over-confident; STS
brings the mean ECE down to about 1 %).

What the pages fix:
  * each confidence c_k models P(position k accepted | every earlier position
    accepted), so by the chain rule the probability that the prefix through k
    is accepted is the cumulative product of the c_j;
  * STS calibrates that cumulative product left to right: at position k the
    temperatures of positions 1..k-1 are held at their fitted values and a
    one-dimensional grid search picks the temperature T_k that minimises the
    Expected Calibration Error (ECE);
  * temperature scaling divides the confidence logit by T, so it preserves
    the order of the confidences;
  * the supervision is the analytic per-step acceptance rate 1 - TV(p_k, q_k).

Readings where the pages leave a step open:
  * prediction at position k for sample n:
        pred_n(T) = prod_{j<k} sigmoid(a_nj / T_j) * sigmoid(a_nk / T)
    with a_nk the raw (untempered) confidence logit;
  * label at position k: the soft prefix-acceptance probability
        lab_n = prod_{j<=k} y_nj,  y_nj in [0, 1] the per-step soft label;
  * ECE with n_bins equal-width bins on [0, 1] (bin = floor(pred * n_bins),
    clamped to the last bin), each bin weighted by its share of the N samples:
        ECE = sum_bins |bin| / N * | mean_bin(lab) - mean_bin(pred) |;
  * the grid is given by the caller; ties in the arg-min go to the first
    (lowest-index) grid point.
"""

import numpy as np


def sigmoid(x):
    """Logistic function in float64, evaluated without overflow on either side."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty_like(x)
    pos = x >= 0
    out[pos] = 1.0 / (1.0 + np.exp(-x[pos]))
    e = np.exp(x[~pos])
    out[~pos] = e / (1.0 + e)
    return out


def ece(pred, lab, n_bins):
    """Expected Calibration Error of predictions `pred` against soft labels `lab`."""
    pred = np.asarray(pred, dtype=np.float64)
    lab = np.asarray(lab, dtype=np.float64)
    n = pred.size
    if n == 0:
        return 0.0
    bins = np.minimum(np.floor(pred * n_bins).astype(np.int64), n_bins - 1)
    total = 0.0
    for b in range(n_bins):
        sel = bins == b
        cnt = int(sel.sum())
        if cnt:
            total += cnt / n * abs(lab[sel].mean() - pred[sel].mean())
    return total


def sts_curves(logits, labels, grid, n_bins, temps):
    """ECE over the grid at every position, with earlier positions held at `temps`.

    Returns an array [K, G]: row k is ECE(T) for T in `grid`, where positions
    0..k-1 use temps[0..k-1]. `temps[k]` itself is not used by row k.
    """
    a = np.asarray(logits, dtype=np.float64)
    y = np.asarray(labels, dtype=np.float64)
    grid = np.asarray(grid, dtype=np.float64)
    N, K = a.shape
    out = np.empty((K, grid.size))
    base = np.ones(N)
    lab = np.ones(N)
    for k in range(K):
        lab = lab * y[:, k]
        for g, T in enumerate(grid):
            out[k, g] = ece(base * sigmoid(a[:, k] / T), lab, n_bins)
        base = base * sigmoid(a[:, k] / float(temps[k]))
    return out


def sts_fit(logits, labels, grid, n_bins):
    """Fit one temperature per position, left to right (the STS procedure).

    Returns a dict: temps [K] (chosen grid values), index [K] (their grid
    indices), ece [K] (the minimum at each position) and curves [K, G].
    """
    a = np.asarray(logits, dtype=np.float64)
    y = np.asarray(labels, dtype=np.float64)
    grid = np.asarray(grid, dtype=np.float64)
    N, K = a.shape
    if grid.size == 0 or np.any(grid <= 0):
        raise ValueError("grid temperatures must be positive")
    temps = np.empty(K)
    index = np.empty(K, dtype=np.int64)
    best = np.empty(K)
    curves = np.empty((K, grid.size))
    base = np.ones(N)
    lab = np.ones(N)
    for k in range(K):
        lab = lab * y[:, k]
        for g, T in enumerate(grid):
            curves[k, g] = ece(base * sigmoid(a[:, k] / T), lab, n_bins)
        g = int(np.argmin(curves[k]))          # first minimum
        index[k], temps[k], best[k] = g, grid[g], curves[k, g]
        base = base * sigmoid(a[:, k] / temps[k])
    return {"temps": temps, "index": index, "ece": best, "curves": curves}
