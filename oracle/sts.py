"""Sequential temperature scaling (STS) in plain numpy, fp64.

TEST INFRASTRUCTURE ONLY, like the rest of this package: only ``tests/`` may
use it, and it shares no code with the CUDA path.

The pages ("[DeepSeek-6] DSpark" blog, section 5; the study report's answer on
calibration) describe STS as a post-hoc calibration of the confidence head on
held-out data: from left to right, position by position, a one-dimensional
grid search picks the temperature of position k so that the cumulative
product prod_{i<=k} c_i matches the empirical prefix survival, measured by the
expected calibration error.  Temperature scaling keeps the order of the
confidences.  The readings this file takes where the pages are silent:

* a sample n is one request of one round: confidence logits z[n, k] (so that
  c = sigmoid(z / T_k)), its verified length ell[n] and accepted count
  acc[n]; position k of sample n is observed when k <= ell[n], with outcome
  y = 1 if acc[n] >= k (the prefix up to k survived), else 0;
* the prediction for an observed position is P = prod_{i<k} sigmoid(z_i /
  T_i) * sigmoid(z_k / T), with T_1..T_{k-1} already fixed;
* ECE with M equal-width bins on [0, 1] (bin min(floor(P * M), M - 1)):
  sum over bins of |sum_{n in bin} (P_n - y_n)| / (number of observed
  samples), i.e. the bin-weighted |mean prediction - mean outcome|;
* the temperature is the grid value with the smallest ECE (the first on
  ties); a position that no sample observes keeps T = 1 and ECE 0.
"""
import numpy as np


def sigmoid(x):
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-x))


def ece(P, y, bins):
    """Expected calibration error of predictions P against 0/1 outcomes y."""
    if P.size == 0:
        return 0.0
    idx = np.minimum(np.floor(P * bins).astype(np.int64), bins - 1)
    total = 0.0
    for m in range(bins):
        sel = idx == m
        total += abs(float(np.sum(P[sel] - y[sel])))
    return total / P.size


def sts_fit(z, ell, acc, grid, bins=15):
    """Temperatures T [gamma] and the ECE reached at each position."""
    z = np.asarray(z, np.float64)
    ell = np.asarray(ell, np.int64)
    acc = np.asarray(acc, np.int64)
    grid = np.asarray(grid, np.float64)
    N, G = z.shape
    T = np.ones(G)
    err = np.zeros(G)
    prev = np.ones(N)                    # prod_{i<k} sigmoid(z_i / T_i)
    for k in range(1, G + 1):
        obs = ell >= k
        y = (acc >= k).astype(np.float64)
        if obs.any():
            best_e, best_g = None, 0
            for g, t in enumerate(grid):
                P = prev * sigmoid(z[:, k - 1] / t)
                e = ece(P[obs], y[obs], bins)
                if best_e is None or e < best_e:
                    best_e, best_g = e, g
            T[k - 1] = grid[best_g]
            err[k - 1] = best_e
        prev = prev * sigmoid(z[:, k - 1] / T[k - 1])
    return T, err
