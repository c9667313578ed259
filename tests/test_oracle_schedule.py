"""Pins of the oracle's prefix scheduler: a hand-worked instance, exhaustive
search over every verify-length vector on tiny batches, closed-form SPS tables
and the tie / top-K rules.  CPU only."""
import itertools
import os

import numpy as np
import pytest

import oracle
from oracle import MODE_FIXED, MODE_GREEDY, MODE_TOPK


def _theta(c, ell, sps):
    """Theta of one verify-length vector by the definitions of the blog's
    section 6: a_{r,j} = prod_{i<=j} c_{r,i}; B = sum (l_r+1);
    tau = sum (1 + sum_{j<=l_r} a_{r,j}); Theta = tau * SPS(B)."""
    R = c.shape[0]
    tau = 0.0
    for r in range(R):
        a, s = 1.0, 1.0
        for j in range(ell[r]):
            a *= c[r, j]
            s += a
        tau += s
    return tau * float(sps[R + sum(ell)])


def _read_example(golden_dir):
    d = {}
    with open(os.path.join(golden_dir, "schedule_worked_example.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            k, *v = line.split()
            d[k] = v
    return d


def test_hand_worked_example(golden_dir):
    d = _read_example(golden_dir)
    R, G = int(d["R"][0]), int(d["gamma"][0])
    c = np.array([float(t) for t in d["c"]]).reshape(R, G)
    sps = np.array([float(t) for t in d["sps"]], np.float32)
    out = oracle.schedule(c, sps, MODE_GREEDY)
    assert out["nstar"] == int(d["nstar"][0])
    assert list(out["ell"]) == [int(t) for t in d["ell"]]
    assert out["theta"] == pytest.approx(float(d["theta"][0]), rel=1e-12)


def _tables(Bmax, rng):
    b = np.arange(Bmax + 1, dtype=np.float64)
    yield "saturating", (b / (1 + b / 6.0)).astype(np.float32)           # increasing, concave
    yield "linear_dec", (1.0 + (Bmax + 1 - b) * 0.35).astype(np.float32)  # decreasing, concave
    yield "steps_per_s", (1.0 / (1.0 + b / 3.0)).astype(np.float32)      # decreasing, convex
    jag = np.sort(rng.uniform(0.2, 1.0, Bmax + 1))[::-1].copy()
    yield "jagged", jag.astype(np.float32)


@pytest.mark.parametrize("R,G", [(1, 3), (2, 2), (2, 3), (3, 2), (4, 2), (3, 3)])
def test_exhaustive_search(R, G):
    rng = np.random.default_rng(100 * R + G)
    for trial in range(25):
        c = rng.uniform(0.05, 0.999, (R, G))
        if trial % 5 == 0:
            c = np.round(c, 1)  # equal survival values exercise the tie order
        for name, sps in _tables(R * (G + 1), rng):
            out = oracle.schedule(c, sps, MODE_GREEDY)
            ell = out["ell"]
            # the reported Theta is the Theta of the reported lengths
            assert out["theta"] == pytest.approx(_theta(c, ell, sps), rel=1e-12)
            assert sum(ell) == out["nstar"]
            best = max(_theta(c, e, sps) for e in itertools.product(range(G + 1), repeat=R))
            # For a fixed number of admitted tokens the best tau is the sorted
            # prefix, so the best Theta over all vectors equals the best sorted
            # prefix; the early stop finds it whenever Theta along the sorted
            # order is unimodal, which holds for positive concave SPS tables.
            a = np.cumprod(c, axis=1).ravel()
            srt = np.sort(a)[::-1]
            prefix = [(R + srt[:n].sum()) * float(sps[R + n]) for n in range(R * G + 1)]
            assert max(prefix) == pytest.approx(best, rel=1e-12)
            d = np.diff(prefix)
            unimodal = not np.any((d[1:] > 0) & (d[:-1] <= 0))
            if name in ("saturating", "linear_dec") or unimodal:
                assert out["theta"] == pytest.approx(best, rel=1e-12)
            else:
                assert out["theta"] <= best * (1 + 1e-12)


def test_prefix_closed_and_tie_order():
    # all survival values equal: candidates are taken in (r asc, j asc) order
    R, G = 3, 2
    c = np.ones((R, G))
    b = np.arange(R * (G + 1) + 1, dtype=np.float64)
    for K in range(R * G + 1):
        out = oracle.schedule(c, np.ones(R * (G + 1) + 1, np.float32), MODE_TOPK, K=K)
        order = [(r, j) for r in range(R) for j in range(1, G + 1)]
        want = [0] * R
        for r, _ in order[:K]:
            want[r] += 1
        assert list(out["ell"]) == want
    # the candidate order itself
    out = oracle.schedule(c, np.ones(R * (G + 1) + 1, np.float32), MODE_GREEDY)
    assert list(out["order"]) == list(range(R * G))
    del b


def test_closed_form_tables():
    rng = np.random.default_rng(7)
    R, G = 5, 4
    c = rng.uniform(0.01, 0.99, (R, G))
    n = R * (G + 1) + 1
    # SPS constant: any a > 0 raises tau, so everything is admitted
    out = oracle.schedule(c, np.full(n, 3.0, np.float32), MODE_GREEDY)
    assert list(out["ell"]) == [G] * R
    # SPS(B) = B: both factors grow, everything is admitted
    out = oracle.schedule(c, np.arange(n, dtype=np.float32), MODE_GREEDY)
    assert list(out["ell"]) == [G] * R
    # a zero survival probability leaves Theta equal under a constant table: a tie stops
    c2 = c.copy()
    c2[:, 1] = 0.0
    out = oracle.schedule(c2, np.full(n, 3.0, np.float32), MODE_GREEDY)
    assert list(out["ell"]) == [1] * R
    # fixed mode never truncates
    out = oracle.schedule(c, None, MODE_FIXED)
    assert list(out["ell"]) == [G] * R


def test_topk_admits_exactly_k_prefix_closed():
    rng = np.random.default_rng(3)
    R, G = 6, 5
    c = rng.uniform(0.1, 0.99, (R, G))
    sps = (1.0 / (1.0 + np.arange(R * (G + 1) + 1) / 8.0)).astype(np.float32)
    greedy = oracle.schedule(c, sps, MODE_GREEDY)
    a = np.cumprod(c, axis=1)
    for K in [0, 1, 7, R * G, R * G + 5, -3]:
        out = oracle.schedule(c, sps, MODE_TOPK, K=K)
        assert out["ell"].sum() == min(max(K, 0), R * G)
        assert out["nstar"] == greedy["nstar"]  # the greedy count is still reported
        # prefix-closed and made of the K largest survival values
        thr = np.sort(a.ravel())[::-1][out["ell"].sum() - 1] if out["ell"].sum() else np.inf
        for r in range(R):
            assert np.all(a[r, :out["ell"][r]] >= thr)


def test_sps_table_too_short_is_rejected():
    c = np.full((2, 3), 0.5)
    with pytest.raises(RuntimeError):
        oracle.schedule(c, np.ones(8, np.float32), MODE_GREEDY)  # needs B up to 8
