"""Pins of the sequential-temperature-scaling oracle (``oracle/sts.py``):
closed-form ECE values, data generated from a known temperature (the fit must
find it, position by position along the prefix product), unobserved
positions, and order preservation."""
import numpy as np
import pytest

from oracle import sts

GRID = np.exp(np.linspace(np.log(0.25), np.log(4.0), 49)).astype(np.float32)   # holds 1.0 at index 24


def _survival_data(N, G, t_true, seed):
    """Logits z and the accepted counts of a prefix that survives position k
    with probability sigmoid(z_k / t_true) (every position verified)."""
    rng = np.random.default_rng(seed)
    z = rng.normal(1.5, 1.5, size=(N, G)).astype(np.float32)
    u = rng.random((N, G))
    ok = u < sts.sigmoid(z.astype(np.float64) / t_true)
    acc = np.where(ok.all(axis=1), G, np.argmin(ok, axis=1)).astype(np.int32)
    ell = np.full(N, G, np.int32)
    return z, ell, acc


def test_ece_closed_forms():
    assert sts.ece(np.array([0.05, 0.95]), np.array([0.0, 1.0]), 15) == pytest.approx(0.05)
    assert sts.ece(np.full(4, 0.5), np.array([0.0, 1.0, 0.0, 1.0]), 15) == pytest.approx(0.0)
    # one bin: |mean P - mean y|
    assert sts.ece(np.array([0.61, 0.62, 0.63]), np.array([1.0, 1.0, 0.0]), 10) == pytest.approx(abs(0.62 - 2 / 3))
    # P = 1 falls in the last bin
    assert sts.ece(np.array([1.0]), np.array([0.0]), 15) == pytest.approx(1.0)


@pytest.mark.parametrize("t_true,idx", [(1.0, 24), (2.0, 36)])
def test_fit_recovers_the_generating_temperature(t_true, idx):
    z, ell, acc = _survival_data(200_000, 4, t_true, seed=3)
    T, err = sts.sts_fit(z, ell, acc, GRID)
    # every position, including those behind the prefix product, within one
    # grid step of the truth, and well calibrated
    assert np.all(np.abs(np.log(T / GRID[idx])) <= np.log(GRID[1] / GRID[0]) * 1.01), T
    assert np.all(err < 0.01), err


def test_fit_is_no_worse_than_no_scaling():
    z, ell, acc = _survival_data(50_000, 3, 1.7, seed=5)
    T, err = sts.sts_fit(z, ell, acc, GRID)
    prev = np.ones(len(z))
    for k in range(3):
        obs = ell >= k + 1
        y = (acc >= k + 1).astype(np.float64)
        P1 = prev * sts.sigmoid(z[:, k].astype(np.float64))
        assert err[k] <= sts.ece(P1[obs], y[obs], 15) + 1e-15
        prev = prev * sts.sigmoid(z[:, k].astype(np.float64) / T[k])


def test_unobserved_positions_keep_unit_temperature():
    z, _, acc = _survival_data(1000, 4, 1.0, seed=7)
    ell = np.full(len(z), 2, np.int32)       # positions 3 and 4 never verified
    acc = np.minimum(acc, 2)
    T, err = sts.sts_fit(z, ell, acc, GRID)
    assert T[2] == 1.0 and T[3] == 1.0 and err[2] == 0.0 and err[3] == 0.0


def test_scaling_keeps_the_order_of_confidences():
    z, ell, acc = _survival_data(5000, 2, 3.0, seed=11)
    T, _ = sts.sts_fit(z, ell, acc, GRID)
    assert T[0] > 0
    c = sts.sigmoid(z[:, 0].astype(np.float64) / T[0])
    assert np.array_equal(np.argsort(c, kind="stable"), np.argsort(z[:, 0], kind="stable"))
