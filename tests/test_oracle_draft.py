"""Pins of the oracle's Markov draft and confidence head against cases whose
answer is fixed by construction, by closed forms or by the textbook law of
Gumbel-max sampling.  CPU only."""
import math

import numpy as np
import pytest
from scipy import stats

import oracle


def _bf16_bits(a):
    a = np.ascontiguousarray(a, dtype=np.float32)
    return (a.view(np.uint32) >> 16).astype(np.uint16)


# ---------------------------------------------------------------------------
# Markov chain by construction: with W1 = identity the embedding of the previous
# token is a unit vector, so the bias of vocabulary entry v is W2[v, prev].
# A +60 entry at v = succ(prev) forces x_k = succ(x_{k-1}) with x_0 = anchor.
# A swapped operand (W1 indexed by v, W2 by prev) or an off-by-one previous
# token would walk a different chain.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("bf16", [False, True])
def test_draft_follows_planted_markov_chain(bf16):
    V, G, B = 16, 6, 3
    succ = lambda i: (3 * i + 5) % V
    W1 = np.eye(V, dtype=np.float32)
    W2 = np.zeros((V, V), np.float32)
    for prev in range(V):
        W2[succ(prev), prev] = 60.0
    rng = np.random.default_rng(0)
    U = rng.normal(0, 1, (B, G, V)).astype(np.float32)
    anchor = np.array([0, 7, 11], np.int32)
    if bf16:
        W1, W2 = _bf16_bits(W1), _bf16_bits(W2)
    out = oracle.draft(U, W1, W2, anchor, seed=3, rnd=0)
    for b in range(B):
        t = int(anchor[b])
        for k in range(G):
            t = succ(t)
            assert out["x"][b, k] == t
    # the planted entry holds all of its block's mass: the block race is won by
    # about 60 nats and the margin left is the inverse-CDF distance of the
    # block's uniform from the ends of [0, 1]
    assert np.all(out["margin"] > 1e-3)


def test_draft_uniform_logits_closed_form():
    # W2 = 0 (no Markov bias) and constant U: p = 1/V exactly, lse = c + log V
    V, G, B = 1000, 3, 2
    U = np.full((B, G, V), 1.25, np.float32)
    W1 = np.ones((V, 4), np.float32)
    W2 = np.zeros((V, 4), np.float32)
    out = oracle.draft(U, W1, W2, np.array([1, 2], np.int32), seed=0, rnd=0)
    np.testing.assert_allclose(out["p"], 1.0 / V, rtol=1e-14)
    np.testing.assert_allclose(out["lse"], 1.25 + math.log(V), rtol=1e-14)


def _constructed_case(V=6, G=3, seed=0):
    """U_k = log q_k and a one-hot embedding with W2[v, prev] = log A[prev, v], so
    p_k(v | prev) = q_k(v) A[prev, v] / sum_u q_k(u) A[prev, u] by construction."""
    rng = np.random.default_rng(seed)
    q = rng.dirichlet(np.ones(V), size=G)          # [G, V]
    A = rng.dirichlet(np.ones(V) * 0.7, size=V)    # [V(prev), V]
    A = np.maximum(A, 1e-3)
    U = np.log(q).astype(np.float32)
    W1 = np.eye(V, dtype=np.float32)
    W2 = np.ascontiguousarray(np.log(A).T.astype(np.float32))  # W2[v, prev] = log A[prev, v]
    # the law the oracle must reproduce, from the float32-rounded inputs
    qf = np.exp(U.astype(np.float64))
    Af = np.exp(W2.astype(np.float64).T)
    return U, W1, W2, qf, Af


def test_draft_probability_and_lse_by_construction():
    V, G = 6, 3
    U, W1, W2, q, A = _constructed_case(V, G)
    B = 4
    Ub = np.broadcast_to(U, (B, G, V)).copy()
    anchor = np.array([0, 1, 2, 5], np.int32)
    out = oracle.draft(Ub, W1, W2, anchor, seed=9, rnd=1)
    for b in range(B):
        prev = anchor[b]
        for k in range(G):
            w = q[k] * A[prev]
            x = out["x"][b, k]
            assert out["p"][b, k] == pytest.approx(w[x] / w.sum(), rel=1e-12)
            assert out["lse"][b, k] == pytest.approx(math.log(w.sum()), rel=1e-12, abs=1e-12)
            prev = x


def test_draft_sequence_law_chi_square():
    # the sampler's law (an exact draw from softmax(l)) over the whole
    # semi-autoregressive chain: P(x1,x2,x3) = prod_k q_k(x_k) A[x_{k-1},x_k] / Z_k
    V, G = 4, 3
    U, W1, W2, q, A = _constructed_case(V, G, seed=5)
    B = 30000
    Ub = np.broadcast_to(U, (B, G, V)).copy()
    anchor = np.full(B, 2, np.int32)
    out = oracle.draft(Ub, W1, W2, anchor, seed=123, rnd=4)
    idx = out["x"][:, 0] * V * V + out["x"][:, 1] * V + out["x"][:, 2]
    counts = np.bincount(idx, minlength=V ** 3)
    law = np.zeros(V ** 3)
    for x1 in range(V):
        p1 = q[0] * A[2]
        p1 = p1[x1] / p1.sum()
        for x2 in range(V):
            p2 = q[1] * A[x1]
            p2 = p2[x2] / p2.sum()
            for x3 in range(V):
                p3 = q[2] * A[x2]
                law[x1 * V * V + x2 * V + x3] = p1 * p2 * p3[x3] / p3.sum()
    exp_ = law * B
    keep = exp_ > 5
    chi2 = ((counts[keep] - exp_[keep]) ** 2 / exp_[keep]).sum()
    dof = keep.sum() - 1
    assert stats.chi2.sf(chi2, dof) > 1e-4
    assert counts[~keep].sum() <= max(20, 3 * exp_[~keep].sum())


def test_markov_free_draft_is_parallel_drafter():
    # With W2 = 0 the bias vanishes and each position is an independent draw
    # from softmax(U_k) (the parallel-drafter special case).
    V, G, B = 5, 2, 40000
    rng = np.random.default_rng(2)
    Urow = rng.normal(0, 1, (G, V)).astype(np.float32)
    U = np.broadcast_to(Urow, (B, G, V)).copy()
    W1 = rng.normal(0, 1, (V, 3)).astype(np.float32)
    W2 = np.zeros((V, 3), np.float32)
    out = oracle.draft(U, W1, W2, np.zeros(B, np.int32), seed=77, rnd=0)
    P = np.exp(Urow.astype(np.float64))
    P /= P.sum(1, keepdims=True)
    joint = np.bincount(out["x"][:, 0] * V + out["x"][:, 1], minlength=V * V)
    law = np.outer(P[0], P[1]).ravel()
    chi2 = ((joint - law * B) ** 2 / (law * B)).sum()
    assert stats.chi2.sf(chi2, V * V - 1) > 1e-4


def test_draft_teacher_forcing_uses_forced_previous_token():
    V, G = 16, 4
    succ = lambda i: (5 * i + 1) % V
    W1 = np.eye(V, dtype=np.float32)
    W2 = np.zeros((V, V), np.float32)
    for prev in range(V):
        W2[succ(prev), prev] = 60.0
    U = np.zeros((1, G, V), np.float32)
    forced = np.array([[9, 3, 12, 0]], np.int32)
    out = oracle.draft(U, W1, W2, np.array([4], np.int32), seed=0, rnd=0, x_force=forced)
    assert out["x"][0, 0] == succ(4)
    for k in range(1, G):
        assert out["x"][0, k] == succ(forced[0, k - 1])


def _block_sample_by_hand(l, seed, rnd, req, k):
    """The two-level draw restated from raw Philox words: Gumbel-max over
    blocks of 4 on their log-mass (stream 0, word j of the call sequence), then
    the inverse CDF inside the winner (stream 4)."""
    V = l.size
    m = np.max(l)
    best, second, jb = -np.inf, -np.inf, -1
    for j in range((V + 3) // 4):
        s_ = np.exp(l[4 * j:4 * j + 4] - m).sum()
        if s_ == 0:
            continue
        w = oracle.rng_word(seed, rnd, 0, req, k, j)
        u = ((w >> 9) + 0.5) / 2.0 ** 23
        z = m + math.log(s_) - math.log(-math.log(u))
        if z > best:
            best, second, jb = z, best, j
        elif z > second:
            second = z
    u2 = ((oracle.rng_word(seed, rnd, 4, req, k, jb) >> 9) + 0.5) / 2.0 ** 23
    e = np.exp(l[4 * jb:4 * jb + 4] - m)
    cum = np.cumsum(e) / e.sum()
    x = 4 * jb + int(np.argmax(cum > u2))
    inner = [abs(u2 - c) for i, c in enumerate(cum[:-1]) if e[i] > 0 and e[i + 1:].sum() > 0]
    return x, min([best - second] + inner)


def _block_draw_by_hand(w, seed, rnd, stream, req, k):
    """The generic two-level draw from weights w, restated from raw words."""
    V = w.size
    best, second, jb = -np.inf, -np.inf, -1
    for j in range((V + 3) // 4):
        s_ = w[4 * j:4 * j + 4].sum()
        if s_ <= 0:
            continue
        u = ((oracle.rng_word(seed, rnd, stream, req, k, j) >> 9) + 0.5) / 2.0 ** 23
        z = math.log(s_) - math.log(-math.log(u))
        if z > best:
            best, second, jb = z, best, j
        elif z > second:
            second = z
    if jb < 0:
        return -1
    u2 = ((oracle.rng_word(seed, rnd, stream + 4, req, k, jb) >> 9) + 0.5) / 2.0 ** 23
    e = w[4 * jb:4 * jb + 4]
    cum = np.cumsum(e) / e.sum()
    return 4 * jb + int(np.argmax(cum > u2))


@pytest.mark.parametrize("stream", [2, 3])
def test_block_draw_definition_and_law(stream):
    rng = np.random.default_rng(stream)
    # definition, with zero weights and a short last block
    for t in range(30):
        V = [9, 16, 30][t % 3]
        w = rng.uniform(0, 1, V) * (rng.uniform(0, 1, V) > 0.3)
        x, _ = oracle.block_draw(w, 7 + t, 3, stream, 2, 5)
        assert x == _block_draw_by_hand(w, 7 + t, 3, stream, 2, 5)
        assert x < 0 or w[x] > 0
    assert oracle.block_draw(np.zeros(8), 1, 1, stream, 0, 1)[0] == -1
    # law over seeds: w / sum w
    w = np.array([0.5, 0.0, 2.0, 0.1, 0.0, 0.0, 1.4, 0.3, 0.9, 0.2])
    n = 30000
    counts = np.bincount([oracle.block_draw(w, s, 0, stream, 1, 2)[0] for s in range(n)], minlength=w.size)
    p = w / w.sum()
    assert np.all(counts[p == 0] == 0)
    keep = p > 0
    chi2 = ((counts[keep] - n * p[keep]) ** 2 / (n * p[keep])).sum()
    assert stats.chi2.sf(chi2, keep.sum() - 1) > 1e-4
    # a softmax draw is the block draw of exp(score - max)
    sc = rng.normal(0, 2, 24)
    sc[5] = -np.inf
    assert oracle.softmax_draw(sc, 3, 1, stream, 4, 2)[0] == \
        oracle.block_draw(np.exp(sc - sc.max()), 3, 1, stream, 4, 2)[0]


def test_block_sample_definition_and_margin():
    rng = np.random.default_rng(4)
    for V in (64, 10, 4, 3):
        for t in range(20):
            l = rng.normal(0, 2, V)
            if t % 4 == 1:
                l[rng.integers(0, V)] = -np.inf
            x, mg = oracle.block_sample(l, 5 + t, 6, 1, 2)
            xh, mh = _block_sample_by_hand(l, 5 + t, 6, 1, 2)
            assert x == xh
            assert mg == pytest.approx(mh, abs=1e-12)
            assert l[x] > -np.inf
    assert oracle.block_sample(np.full(4, -np.inf), 1, 1, 0, 1)[0] == -1


@pytest.mark.parametrize("V", [8, 10, 13])
def test_block_sample_law_chi_square(V):
    # over seeds the two-level draw follows softmax(l), also with a short
    # last block and a -inf entry
    rng = np.random.default_rng(V)
    l = rng.normal(0, 1, V)
    l[3] = -np.inf
    p = np.exp(l - l[np.isfinite(l)].max())
    p /= p.sum()
    n = 30000
    counts = np.bincount([oracle.block_sample(l, s, 0, 0, 1)[0] for s in range(n)], minlength=V)
    assert counts[3] == 0
    keep = p > 0
    chi2 = ((counts[keep] - n * p[keep]) ** 2 / (n * p[keep])).sum()
    assert stats.chi2.sf(chi2, keep.sum() - 1) > 1e-4


# ---------------------------------------------------------------------------
# confidence head c_k = sigmoid(w^T [h_k ; W1[x_{k-1}]] / T_k)
# ---------------------------------------------------------------------------
def test_confidence_zero_weight_and_infinite_temperature():
    B, G, H, V, r = 2, 3, 8, 10, 4
    rng = np.random.default_rng(0)
    h = rng.normal(0, 1, (B, G, H)).astype(np.float32)
    W1 = rng.normal(0, 1, (V, r)).astype(np.float32)
    x = rng.integers(0, V, (B, G)).astype(np.int32)
    anchor = np.array([1, 2], np.int32)
    c = oracle.confidence(h, W1, np.zeros(H + r, np.float32), anchor, x)
    assert np.all(c == 0.5)
    w = rng.normal(0, 1, H + r).astype(np.float32)
    c = oracle.confidence(h, W1, w, anchor, x, sts_T=np.full(G, 1e30, np.float32))
    np.testing.assert_allclose(c, 0.5, atol=1e-15)


def test_confidence_one_hot_closed_form():
    # one-hot h_k and one-hot embeddings pick single weights: the logit is
    # w[i] + w[H + prev] where i is the hot hidden unit and prev the previous token
    B, G, H, V = 1, 3, 4, 5
    W1 = np.eye(V, dtype=np.float32)           # r = V
    w = np.array([0.5, -1.0, 2.0, 0.25, 1.0, -2.0, 0.75, 3.0, -0.5], np.float32)
    h = np.zeros((B, G, H), np.float32)
    hot = [2, 0, 3]
    for k in range(G):
        h[0, k, hot[k]] = 1.0
    anchor = np.array([4], np.int32)
    x = np.array([[1, 3, 0]], np.int32)
    T = np.array([1.0, 2.0, 0.5], np.float32)
    c = oracle.confidence(h, W1, w, anchor, x, sts_T=T)
    prevs = [4, 1, 3]
    for k in range(G):
        z = (float(w[hot[k]]) + float(w[H + prevs[k]])) / float(T[k])
        assert c[0, k] == pytest.approx(1.0 / (1.0 + math.exp(-z)), rel=1e-15)
    # z = 2 reference value of the logistic function
    c1 = oracle.confidence(np.zeros((1, 1, 1), np.float32), np.eye(2, dtype=np.float32),
                           np.array([0.0, 0.0, 2.0], np.float32), np.array([1], np.int32),
                           np.zeros((1, 1), np.int32))
    assert c1[0, 0] == pytest.approx(0.8807970779778823, rel=1e-15)


def test_confidence_bf16_inputs_match_float_values():
    B, G, H, V, r = 2, 2, 16, 12, 8
    rng = np.random.default_rng(1)
    hf = rng.normal(0, 1, (B, G, H)).astype(np.float32)
    Wf = rng.normal(0, 1, (V, r)).astype(np.float32)
    hb, Wb = _bf16_bits(hf), _bf16_bits(Wf)
    # the bf16 values, widened back to float32 exactly
    h_r = (hb.astype(np.uint32) << 16).view(np.float32)
    W_r = (Wb.astype(np.uint32) << 16).view(np.float32)
    w = rng.normal(0, 0.3, H + r).astype(np.float32)
    x = rng.integers(0, V, (B, G)).astype(np.int32)
    a = np.array([3, 4], np.int32)
    np.testing.assert_array_equal(oracle.confidence(hb, Wb, w, a, x),
                                  oracle.confidence(h_r, W_r, w, a, x))


def test_draft_uses_stream0_counter_layout():
    # x_k = the two-level draw from softmax(l) with (request b, position k)
    V, G, B = 40, 3, 3
    rng = np.random.default_rng(12)
    U = rng.normal(0, 1, (B, G, V)).astype(np.float32)
    W1 = rng.normal(0, 0.5, (V, 4)).astype(np.float32)
    W2 = rng.normal(0, 0.5, (V, 4)).astype(np.float32)
    anchor = np.array([1, 5, 9], np.int32)
    seed, rnd = (1 << 40) + 3, 2
    out = oracle.draft(U, W1, W2, anchor, seed, rnd)
    for b in range(B):
        prev = anchor[b]
        for k in range(1, G + 1):
            l = oracle.draft_logits(U[b, k - 1], W1, W2, prev)
            x, mg = _block_sample_by_hand(l, seed, rnd, b, k)
            assert out["x"][b, k - 1] == x
            assert out["margin"][b, k - 1] == pytest.approx(mg, abs=1e-12)
            prev = out["x"][b, k - 1]


def test_thread_count_leaves_results_unchanged():
    # the request loops run in parallel; one thread must give the same rounds
    rng = np.random.default_rng(17)
    B, G, V, r = 6, 3, 96, 16
    U = rng.normal(0, 2, (B, G, V)).astype(np.float32)
    T = rng.normal(0, 2, (B, G + 1, V)).astype(np.float32)
    W1 = rng.normal(0, 0.3, (V, r)).astype(np.float32)
    W2 = rng.normal(0, 0.3, (V, r)).astype(np.float32)
    anchor = rng.integers(0, V, B).astype(np.int32)
    ell = np.array([0, 1, 2, 3, 3, 2], np.int32)

    def one_round():
        d = oracle.draft(U, W1, W2, anchor, 9, 4)
        v = oracle.verify(T, U, W1, W2, anchor, d["x"], ell, 9, 4)
        return d, v

    many = one_round()
    thr = oracle.num_threads()
    oracle.set_num_threads(1)
    try:
        assert oracle.num_threads() == 1
        single = one_round()
    finally:
        oracle.set_num_threads(thr)
    assert oracle.num_threads() == thr
    for a, b in zip(many, single):
        for k in a:
            assert np.array_equal(a[k], b[k], equal_nan=a[k].dtype.kind == "f"), k
