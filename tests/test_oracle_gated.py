"""Pins of the oracle's gated recurrent Markov head (the head the DSpark pages
name without equations: [blog] section 4 and [digest] item 8; its plain design
is e_k = W1[x_{k-1}], a_k = sigmoid(g * e_k + c), s_0 = 0,
s_k = e_k + a_k * s_{k-1}, bias_k(v) = s_k . W2[v]).  Each pin checks the
recurrence against a different statement of it: the Markov head when the gate
is shut, a geometric sum for a constant gate, the unrolled product form for
input-dependent gates, and a two-step example worked by hand."""
import numpy as np
import pytest

import oracle


def _weights(V, r, seed, scale=0.5):
    rng = np.random.default_rng(seed)
    W1 = (rng.standard_normal((V, r)) * scale).astype(np.float32)
    W2 = (rng.standard_normal((V, r)) * scale).astype(np.float32)
    return rng, W1, W2


def _sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def test_two_steps_by_hand():
    # r = 1, W1 = [[1], [2]], g = 0, c = 0: every gate is 1/2.  Prefix: anchor
    # 0, then x_1 = 1: s_1 = W1[0] = 1, s_2 = W1[1] + s_1 / 2 = 2.5.
    W1 = np.array([[1.0], [2.0]], np.float32)
    s = oracle.gated_states(W1, np.zeros(1, np.float32), np.zeros(1, np.float32), 0, [1], 2)
    assert s[:, 0].tolist() == [1.0, 2.5]


def test_constant_gate_is_a_geometric_sum():
    V, r, G = 50, 8, 6
    rng, W1, _ = _weights(V, r, 1)
    alpha = 0.3
    c = np.full(r, np.log(alpha / (1 - alpha)), np.float32)
    toks = rng.integers(0, V, G)            # anchor, then x_1 .. x_{G-1}
    s = oracle.gated_states(W1, np.zeros(r, np.float32), c, int(toks[0]), toks[1:], G)
    a = float(_sigmoid(np.float64(c[0])))   # the float32 c, as the oracle reads it
    e = W1[toks].astype(np.float64)
    for k in range(1, G + 1):
        want = sum(a ** (k - i) * e[i - 1] for i in range(1, k + 1))
        np.testing.assert_allclose(s[k - 1], want, rtol=1e-12, atol=1e-14)


def test_input_gates_match_the_unrolled_products():
    V, r, G = 40, 6, 5
    rng, W1, _ = _weights(V, r, 2)
    g = rng.standard_normal(r).astype(np.float32)
    c = rng.standard_normal(r).astype(np.float32)
    toks = rng.integers(0, V, G)
    s = oracle.gated_states(W1, g, c, int(toks[0]), toks[1:], G)
    e = W1[toks].astype(np.float64)
    a = _sigmoid(g.astype(np.float64) * e + c.astype(np.float64))   # a_j gates s_{j-1} at step j
    for k in range(1, G + 1):
        want = np.zeros(r)
        for i in range(1, k + 1):
            want += np.prod(a[i:k], axis=0) * e[i - 1]
        np.testing.assert_allclose(s[k - 1], want, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("bf16", [False, True])
def test_shut_gate_is_the_markov_head(bf16):
    B, G, V, r = 3, 4, 300, 8
    rng, W1, W2 = _weights(V, r, 3)
    if bf16:
        W1 = (W1.view(np.uint32) >> 16).astype(np.uint16)
        W2 = (W2.view(np.uint32) >> 16).astype(np.uint16)
    U = rng.standard_normal((B, G, V)).astype(np.float32)
    T = rng.standard_normal((B, G + 1, V)).astype(np.float32)
    anchor = rng.integers(0, V, B).astype(np.int32)
    g = rng.standard_normal(r).astype(np.float32)
    c = np.full(r, -1e4, np.float32)        # sigmoid underflows to exactly 0
    m = oracle.draft(U, W1, W2, anchor, 5, 2)
    q = oracle.gated_draft(U, W1, W2, g, c, anchor, 5, 2)
    assert np.array_equal(m["x"], q["x"])
    assert np.array_equal(m["p"], q["p"]) and np.array_equal(m["lse"], q["lse"])
    ell = np.full(B, G, np.int32)
    mv = oracle.verify(T, U, W1, W2, anchor, m["x"], ell, 5, 2)
    qv = oracle.gated_verify(T, U, W1, W2, g, c, anchor, m["x"], ell, 5, 2)
    assert np.array_equal(mv["n"], qv["n"]) and np.array_equal(mv["y"], qv["y"])


def test_gated_draft_scores_each_position_with_its_state():
    B, G, V, r = 2, 4, 200, 8
    rng, W1, W2 = _weights(V, r, 4)
    U = rng.standard_normal((B, G, V)).astype(np.float32)
    anchor = rng.integers(0, V, B).astype(np.int32)
    g = rng.standard_normal(r).astype(np.float32)
    c = (rng.standard_normal(r) + 1.0).astype(np.float32)
    d = oracle.gated_draft(U, W1, W2, g, c, anchor, 9, 0)
    for b in range(B):
        s = oracle.gated_states(W1, g, c, int(anchor[b]), d["x"][b], G)
        for k in range(G):
            l = U[b, k].astype(np.float64) + W2.astype(np.float64) @ s[k]
            lse = np.log(np.exp(l - l.max()).sum()) + l.max()
            assert d["lse"][b, k] == pytest.approx(lse, rel=1e-12)
            assert d["p"][b, k] == pytest.approx(np.exp(l[d["x"][b, k]] - lse), rel=1e-10)
    # an open gate changes the distribution of every position after the first
    m = oracle.draft(U, W1, W2, anchor, 9, 0, x_force=d["x"])
    assert np.array_equal(m["lse"][:, 0], d["lse"][:, 0])
    assert np.all(np.abs(m["lse"][:, 1:] - d["lse"][:, 1:]) > 1e-9)


def _bf16_rne(x):
    # nearest bf16 (ties to even) of float64 values, through their float32 bits
    u = np.asarray(x, np.float64).astype(np.float32).view(np.uint32).astype(np.uint64)
    u = ((u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000).astype(np.uint32)
    return u.view(np.float32).astype(np.float64)


def test_bf16_state_rounds_each_step():
    # the tensor-core precision option: every state rounded to bf16 as it is
    # formed, then carried; checked against an independent rounding
    V, r, G = 60, 16, 6
    rng, W1, _ = _weights(V, r, 5)
    W1b = (W1.view(np.uint32) >> 16).astype(np.uint16)           # bf16 bits
    e_all = (W1b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    g = rng.standard_normal(r).astype(np.float32)
    c = rng.standard_normal(r).astype(np.float32)
    toks = rng.integers(0, V, G)
    s = oracle.gated_states(W1b, g, c, int(toks[0]), toks[1:], G, bf16_state=True)
    want = np.zeros(r)
    for k in range(G):
        e = e_all[toks[k]]
        a = 1.0 / (1.0 + np.exp(-(g.astype(np.float64) * e + c.astype(np.float64))))
        want = _bf16_rne(e + a * want)
        assert np.array_equal(s[k], want), k
    exact = oracle.gated_states(W1b, g, c, int(toks[0]), toks[1:], G)
    # each step rounds to 2^-9 relative; the gate (below 1) carries the error on
    np.testing.assert_allclose(s, exact, rtol=0, atol=G * 2.0 ** -9 * np.abs(exact).max())
    assert not np.array_equal(s, exact)
