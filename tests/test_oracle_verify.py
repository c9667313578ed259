"""Pins of the oracle's rejection-sampling verification.

* Exact output law by enumeration (V = 8, gamma <= 3): drafting with the
  semi-autoregressive Markov head, verifying with the oracle's acceptance ratio
  and residual, then continuing with plain target sampling up to gamma + 1
  tokens must give exactly the target's sequential law (the losslessness of
  speculative sampling, digest item 2), also when the verify lengths come from
  the confidence head and the scheduler (the non-anticipating property, blog
  section 7).  Planted mistakes in the test's own copy (a reversed residual, a
  peeking verify length) must break it.
* Monte-Carlo chi-square on the oracle's full sampled path (its own RNG).
* Eq.8 of the study report: the expected single-position acceptance equals
  sum_v min(p_d, p_t) = 1 - 0.5 * ||p_d - p_t||_1.
CPU only."""
import itertools
import math

import numpy as np
import pytest
from scipy import stats

import oracle
from oracle import MODE_GREEDY, MODE_TOPK


class TinyModel:
    """A drafter (backbone logits U + Markov head W1/W2) and a target whose
    logits depend on the whole emitted prefix (a seeded table)."""

    def __init__(self, V=8, G=3, seed=0, tgt_noise=0.9):
        rng = np.random.default_rng(seed)
        self.V, self.G, self.seed = V, G, seed
        self.U = rng.normal(0, 1.2, (1, G, V)).astype(np.float32)
        r = 6
        self.W1 = rng.normal(0, 0.8, (V, r)).astype(np.float32)
        self.W2 = rng.normal(0, 0.8, (V, r)).astype(np.float32)
        self.anchor = np.array([3], np.int32)
        self.tgt_noise = tgt_noise
        self._pd, self._tl, self._comp = {}, {}, {}
        # confidence head inputs
        H = 5
        self.h = rng.normal(0, 1, (1, G, H)).astype(np.float32)
        self.w = rng.normal(0, 0.6, H + r).astype(np.float32)

    def target_logits(self, prefix):
        prefix = tuple(int(t) for t in prefix)
        if prefix not in self._tl:
            m = len(prefix)
            base = self.U[0, m] if m < self.G else np.zeros(self.V, np.float32)
            noise = np.random.default_rng([self.seed, 99, m] + list(prefix)).normal(0, self.tgt_noise, self.V)
            self._tl[prefix] = (base + noise).astype(np.float32)
        return self._tl[prefix]

    def p_t(self, prefix):
        l = self.target_logits(prefix).astype(np.float64)
        e = np.exp(l - l.max())
        return e / e.sum()

    def p_d(self, k, prev):  # k is 0-based position
        key = (k, int(prev))
        if key not in self._pd:
            self._pd[key] = oracle.draft_probs(self.U[0, k], self.W1, self.W2, prev)
        return self._pd[key]

    def completion(self, seq):
        """Target law of the continuation of `seq` up to G+1 tokens."""
        seq = tuple(seq)
        if len(seq) == self.G + 1:
            return np.float64(1.0)
        if seq not in self._comp:
            pt = self.p_t(seq)
            self._comp[seq] = np.stack([pt[v] * self.completion(seq + (v,)) for v in range(self.V)])
        return self._comp[seq]

    def T_rows(self, x):
        return np.stack([self.target_logits(x[:m]) for m in range(self.G + 1)])


def exact_law(M, ell_fn, residual=oracle.residual):
    V, G = M.V, M.G
    out = np.zeros((V,) * (G + 1))

    def add(seq, w):
        out[tuple(seq)] += w * M.completion(seq)

    for x in itertools.product(range(V), repeat=G):
        prev, Px, pds = int(M.anchor[0]), 1.0, []
        for k in range(G):
            pd = M.p_d(k, prev)
            pds.append(pd)
            Px *= pd[x[k]]
            prev = x[k]
        L = int(ell_fn(x))
        stay = 1.0
        for k in range(L):
            pt = M.p_t(x[:k])
            acc = min(1.0, pt[x[k]] / pds[k][x[k]])
            rej = stay * (1.0 - acc)
            if rej > 0:
                rho = residual(pt, pds[k])
                rho = rho / rho.sum()
                for y in range(V):
                    if rho[y] > 0:
                        add(x[:k] + (y,), Px * rej * rho[y])
            stay *= acc
        if stay > 0:
            pt = M.p_t(x[:L])
            for y in range(V):
                add(x[:L] + (y,), Px * stay * pt[y])
    return out


@pytest.mark.parametrize("G", [1, 2, 3])
def test_exact_law_fixed_length(G):
    M = TinyModel(G=G, seed=G)
    law = exact_law(M, lambda x: G)
    np.testing.assert_allclose(law, M.completion(()), rtol=0, atol=1e-12)
    assert law.sum() == pytest.approx(1.0, abs=1e-12)


@pytest.mark.parametrize("G", [2, 3])
def test_exact_law_every_fixed_length(G):
    M = TinyModel(G=G, seed=10 + G)
    for L in range(G + 1):
        law = exact_law(M, lambda x: L)
        np.testing.assert_allclose(law, M.completion(()), rtol=0, atol=1e-12)


def _scheduled_lengths(M, mode, other_c=None, K=-1):
    """Verify length of request 0 chosen by the oracle's confidence head and
    scheduler from its own draft (and a second request with fixed confidences)."""
    R = 1 if other_c is None else 2
    nb = R * (M.G + 1) + 1
    sps = (1.0 / (1.0 + np.arange(nb) / 6.0)).astype(np.float32)  # steps/s falls with batch

    def ell(x):
        c = oracle.confidence(M.h, M.W1, M.w, M.anchor, np.array([x], np.int32))
        if other_c is not None:
            c = np.vstack([c, other_c])
        return oracle.schedule(c, sps, mode, K=K)["ell"][0]

    return ell


@pytest.mark.parametrize("G", [2, 3])
def test_exact_law_scheduled_lengths(G):
    M = TinyModel(G=G, seed=20 + G)
    ell = _scheduled_lengths(M, MODE_GREEDY)
    lengths = {int(ell(x)) for x in itertools.product(range(M.V), repeat=G)}
    assert len(lengths) > 1  # the schedule really truncates, differently per draft
    law = exact_law(M, ell)
    np.testing.assert_allclose(law, M.completion(()), rtol=0, atol=1e-12)


def test_exact_law_scheduled_with_competing_request():
    G = 3
    M = TinyModel(G=G, seed=46)
    other = np.array([[0.8, 0.7, 0.3]])
    for mode, K in [(MODE_GREEDY, -1), (MODE_TOPK, 2), (MODE_TOPK, 4)]:
        ell = _scheduled_lengths(M, mode, other_c=other, K=K)
        lengths = {int(ell(x)) for x in itertools.product(range(M.V), repeat=G)}
        assert len(lengths) > 1
        law = exact_law(M, ell)
        np.testing.assert_allclose(law, M.completion(()), rtol=0, atol=1e-12)


def test_planted_mistakes_break_the_law():
    G = 2
    M = TinyModel(G=G, seed=41)
    target = M.completion(())
    # residual with the operands swapped
    bad = exact_law(M, lambda x: G, residual=lambda pt, pd: oracle.residual(pd, pt))
    assert np.abs(bad - target).max() > 1e-4
    # a verify length that peeks at the token it admits (anticipating)
    bad = exact_law(M, lambda x: G if x[0] % 2 == 0 else 0)
    assert np.abs(bad - target).max() > 1e-4


def _mc_round(M, B, seed, rnd, ell_value):
    V, G = M.V, M.G
    U = np.broadcast_to(M.U, (B, G, V)).copy()
    anchor = np.full(B, M.anchor[0], np.int32)
    d = oracle.draft(U, M.W1, M.W2, anchor, seed, rnd)
    x = d["x"]
    T = np.stack([M.T_rows(tuple(x[b])) for b in range(B)])
    ell = np.full(B, ell_value, np.int32)
    v = oracle.verify(T, U, M.W1, M.W2, anchor, x, ell, seed, rnd)
    return x, v


def test_monte_carlo_first_two_tokens_chi_square():
    G = 2
    M = TinyModel(G=G, seed=51)
    B = 20000
    x, v = _mc_round(M, B, seed=2024, rnd=1, ell_value=G)
    rng = np.random.default_rng(5)
    s = np.empty((B, 2), np.int64)
    for b in range(B):
        n, y = int(v["n"][b]), int(v["y"][b])
        emitted = list(x[b, :n]) + [y]
        while len(emitted) < 2:
            emitted.append(int(rng.choice(M.V, p=M.p_t(tuple(emitted)))))
        s[b] = emitted[:2]
    law = M.completion(()).sum(axis=2).ravel()  # marginal of the first two tokens
    cnt = np.bincount(s[:, 0] * M.V + s[:, 1], minlength=M.V ** 2)
    e = law * B
    keep = e > 5
    chi2 = ((cnt[keep] - e[keep]) ** 2 / e[keep]).sum()
    assert stats.chi2.sf(chi2, keep.sum() - 1) > 1e-4


def test_eq8_identity_and_first_position_acceptance():
    rng = np.random.default_rng(8)
    for _ in range(20):
        V = int(rng.integers(2, 50))
        pd = rng.dirichlet(np.ones(V))
        pt = rng.dirichlet(np.ones(V))
        lab = oracle.acceptance_label(pd, pt)
        assert lab == pytest.approx(np.minimum(pd, pt).sum(), abs=1e-12)
        assert lab == pytest.approx(1 - 0.5 * np.abs(pd - pt).sum(), abs=1e-12)
    assert oracle.acceptance_label(pd, pd) == pytest.approx(1.0, abs=1e-15)
    # the Monte-Carlo acceptance rate of position 1 matches the label
    G = 1
    M = TinyModel(G=G, seed=61)
    B = 30000
    x, v = _mc_round(M, B, seed=99, rnd=3, ell_value=1)
    rate = float(np.mean(v["n"] >= 1))
    lab = oracle.acceptance_label(M.p_d(0, M.anchor[0]), M.p_t(()))
    se = math.sqrt(lab * (1 - lab) / B)
    assert abs(rate - lab) < 3.3 * se  # 99.9 % two-sided


def test_decisions_follow_uniform_below_ratio():
    G, V, B = 4, 8, 64
    M = TinyModel(V=V, G=G, seed=71)
    seed, rnd = 17, 6
    x, v = _mc_round(M, B, seed, rnd, ell_value=G)
    for b in range(B):
        n = int(v["n"][b])
        for k in range(1, n + 2):
            if k > G:
                break
            u = oracle.u01(oracle.rng_word(seed, rnd, 1, b, k, 0))
            ratio = v["ratio"][b, k - 1]
            assert v["umargin"][b, k - 1] == pytest.approx(abs(u - ratio), abs=1e-15)
            assert (u < ratio) == (k <= n)
        for k in range(n + 2, G + 1):
            assert math.isnan(v["ratio"][b, k - 1])
        if n < G:
            assert v["flags"][b] & 2
            pt = M.p_t(tuple(x[b, :n]))
            prev = M.anchor[0] if n == 0 else x[b, n - 1]
            rho = oracle.residual(pt, M.p_d(n, prev))
            assert rho[v["y"][b]] > 0
        else:
            assert v["flags"][b] == 1


def test_identical_distributions_always_accept_and_bonus_row():
    # W2 = 0 and T rows equal to U rows: p_t == p_d exactly, ratio 1 > u always
    B, G, V = 8, 3, 32
    rng = np.random.default_rng(1)
    U = rng.normal(0, 2, (B, G, V)).astype(np.float32)
    W1 = rng.normal(0, 1, (V, 4)).astype(np.float32)
    W2 = np.zeros((V, 4), np.float32)
    T = np.concatenate([U, rng.normal(0, 2, (B, 1, V)).astype(np.float32)], axis=1)
    anchor = rng.integers(0, V, B).astype(np.int32)
    d = oracle.draft(U, W1, W2, anchor, 5, 0)
    ell = np.array([0, 1, 2, 3, 3, 2, 1, 0], np.int32)
    out = oracle.verify(T, U, W1, W2, anchor, d["x"], ell, 5, 0)
    np.testing.assert_array_equal(out["n"], ell)
    assert np.all(out["flags"] == 1)
    for b in range(B):
        want, _ = oracle.softmax_draw(T[b, ell[b]].astype(np.float64), 5, 0, 3, b, int(ell[b]) + 1)
        assert out["y"][b] == want


def test_residual_uses_stream2_at_rejected_position():
    G, V, B = 3, 8, 200
    M = TinyModel(V=V, G=G, seed=81, tgt_noise=2.0)
    seed, rnd = 23, 9
    x, v = _mc_round(M, B, seed, rnd, ell_value=G)
    checked = 0
    for b in range(B):
        n = int(v["n"][b])
        if n == G:
            continue
        pt = M.p_t(tuple(x[b, :n]))
        prev = M.anchor[0] if n == 0 else x[b, n - 1]
        rho = oracle.residual(pt, M.p_d(n, prev))
        want, _ = oracle.block_draw(rho, seed, rnd, 2, b, n + 1)
        assert v["y"][b] == want
        checked += 1
    assert checked > 50


def test_out_of_range_tokens_are_refused():
    # a drafted token outside the vocabulary is an error, not a read past W1
    rng = np.random.default_rng(3)
    B, G, V, r = 2, 2, 16, 4
    U = rng.normal(0, 1, (B, G, V)).astype(np.float32)
    T = rng.normal(0, 1, (B, G + 1, V)).astype(np.float32)
    W1 = rng.normal(0, 0.3, (V, r)).astype(np.float32)
    W2 = rng.normal(0, 0.3, (V, r)).astype(np.float32)
    anchor = np.array([1, 2], np.int32)
    ell = np.array([2, 2], np.int32)
    for bad in (V, -1):
        x = np.array([[3, 4], [5, bad]], np.int32)
        with pytest.raises(RuntimeError):
            oracle.verify(T, U, W1, W2, anchor, x, ell, 1, 0)
    bad_anchor = np.array([1, V + 3], np.int32)
    with pytest.raises(RuntimeError):
        oracle.verify(T, U, W1, W2, bad_anchor, np.array([[3, 4], [5, 6]], np.int32), ell, 1, 0)
