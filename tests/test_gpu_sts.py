"""Sequential temperature scaling on the GPU against the oracle (``oracle/sts.py``)
on the same synthetic held-out samples: the temperature of every position is
the oracle's (or, where fp64 sums of a different order tie, one the oracle
scores equally), and so is the ECE it reaches."""
import numpy as np
import pytest
import torch

import speculative_decoding_02_gb300 as ds
from oracle import sts

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
GRID = np.exp(np.linspace(np.log(0.25), np.log(4.0), 49)).astype(np.float32)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decoding_02_gb300 import build
    build.build()
    ds.library()


def _data(N, G, t_true, seed):
    """Logits, verified lengths (some positions unverified) and accepted counts
    of a prefix that survives position k with probability sigmoid(z_k / t_k)."""
    rng = np.random.default_rng(seed)
    z = rng.normal(1.2, 1.8, size=(N, G)).astype(np.float32)
    ok = rng.random((N, G)) < sts.sigmoid(z.astype(np.float64) / np.asarray(t_true)[None, :])
    run = np.where(ok.all(axis=1), G, np.argmin(ok, axis=1))
    ell = rng.integers(0, G + 1, size=N).astype(np.int32)
    acc = np.minimum(run, ell).astype(np.int32)
    return z, ell, acc


def _oracle_ece_at(z, ell, acc, T_prefix, k, t):
    prev = np.ones(len(z))
    for i in range(k - 1):
        prev = prev * sts.sigmoid(z[:, i].astype(np.float64) / np.float64(T_prefix[i]))
    P = prev * sts.sigmoid(z[:, k - 1].astype(np.float64) / np.float64(t))
    obs = ell >= k
    return sts.ece(P[obs], (acc >= k).astype(np.float64)[obs], 15)


@pytest.mark.parametrize("N,G", [(3000, 3), (70000, 6)])
def test_sts_matches_the_oracle(N, G):
    t_true = np.linspace(0.7, 2.2, G)
    z, ell, acc = _data(N, G, t_true, seed=N + G)
    T_o, e_o = sts.sts_fit(z, ell, acc, GRID)
    T_g, e_g = ds.sts_fit(torch.from_numpy(z).to(DEV), torch.from_numpy(ell).to(DEV),
                          torch.from_numpy(acc).to(DEV), torch.from_numpy(GRID).to(DEV))
    torch.cuda.synchronize()
    T_g, e_g = T_g.cpu().numpy().astype(np.float64), e_g.cpu().numpy().astype(np.float64)
    for k in range(1, G + 1):
        if T_g[k - 1] != T_o[k - 1]:
            # a different grid value is only acceptable if the oracle scores it
            # the same, given the GPU's own earlier temperatures
            e_alt = _oracle_ece_at(z, ell, acc, T_g, k, T_g[k - 1])
            assert e_alt <= e_o[k - 1] + 1e-12, (k, T_g[k - 1], T_o[k - 1])
        assert e_g[k - 1] == pytest.approx(e_o[k - 1], rel=1e-5, abs=1e-7), k
    assert np.all(np.isin(T_g.astype(np.float32), GRID))


def test_unobserved_positions_keep_unit_temperature():
    z, _, acc = _data(2000, 4, np.ones(4), seed=1)
    ell = np.full(len(z), 1, np.int32)
    acc = np.minimum(acc, 1).astype(np.int32)
    T_g, e_g = ds.sts_fit(torch.from_numpy(z).to(DEV), torch.from_numpy(ell).to(DEV),
                          torch.from_numpy(acc).to(DEV), torch.from_numpy(GRID).to(DEV))
    torch.cuda.synchronize()
    assert np.all(T_g.cpu().numpy()[1:] == 1.0) and np.all(e_g.cpu().numpy()[1:] == 0.0)
