"""The gated recurrent Markov head on the GPU (dspark_gated_markov_draft and
dspark_verify_ex with DSPARK_GATED_STATES) against the oracle, teacher-forced
on the GPU's own tokens.

The kernel keeps each state s_k in bf16, as the tensor cores read it, so the
decisions are compared with the oracle run in that same state precision
(bf16_state=True: each state rounded to bf16 as it is formed; the exact
fp64 recurrence is pinned on the CPU).  The two states can still differ where
the GPU's fp32 value of e + a*s and the oracle's fp64 value fall on different
sides of a bf16 rounding boundary: the values are a few fp32 ulps apart, so
this is rare, and each such element moves a logit by at most
2^-8 * max|s| * max|W2|.  SLACK allows four of them per position on top of
the usual 1e-4 decision margin."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_02_gb300 as ds
from speculative_decoding_02_gb300 import workloads as wl

from _parity import MARGIN, host

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decoding_02_gb300 import build
    build.build()
    ds.library()


def _inputs(w):
    inp = wl.make_inputs(w, 0, DEV)
    inp.update(wl.make_gates(w, DEV))
    return inp


def _own_ws(w):
    n = ds.workspace_size(w.B, w.gamma, w.V)
    buf = torch.zeros(n + 256, dtype=torch.uint8, device=DEV)
    return buf[(-buf.data_ptr()) % 256:][:n]


def test_shut_gate_is_the_markov_head():
    # a = sigmoid(g*e - 30) ~ 1e-13: s_k = e_k exactly after the bf16
    # rounding, so draft and verification equal the Markov head bit for bit
    w = wl.custom(B=40, gamma=5, V=8200, r=256, H=64, wdtype=torch.bfloat16, u_sigma=2.0, weight_sigma=0.1, seed=21)
    inp = _inputs(w)
    shut = torch.full_like(inp["gate_c"], -30.0)
    ws_m, ws_g = _own_ws(w), _own_ws(w)
    xm, pm, lm = ds.markov_draft(inp["U"], inp["W1"], inp["W2"], inp["anchor"], w.seed, 3, ws=ws_m)
    xg, pg, lg = ds.gated_markov_draft(inp["U"], inp["W1"], inp["W2"], inp["gate_g"], shut, inp["anchor"], w.seed, 3,
                                       ws=ws_g)
    torch.cuda.synchronize()
    assert torch.equal(xm, xg) and torch.equal(pm, pg) and torch.equal(lm, lg)
    ell = torch.full((w.B,), w.gamma, dtype=torch.int32, device=DEV)
    nm, tm = ds.verify(inp["T"], inp["U"], inp["W1"], inp["W2"], inp["anchor"], xm, pm, lm, ell, w.seed, 3, ws_m)
    ng, tg = ds.verify(inp["T"], inp["U"], inp["W1"], inp["W2"], inp["anchor"], xg, pg, lg, ell, w.seed, 3, ws_g,
                       gated=True)
    torch.cuda.synchronize()
    assert torch.equal(nm, ng) and torch.equal(tm, tg)
    assert ds.read_status(ws_m) == ds.OK and ds.read_status(ws_g) == ds.OK


def _check(w, inp, x, p, lse, n, tok, reqs, rnd):
    h = host(inp)
    g, c = h["gate_g"], h["gate_c"]
    x, p, lse, n, tok = (t.cpu().numpy() for t in (x, p, lse, n, tok))
    ell = np.full(w.B, w.gamma, np.int32)
    b0, b1 = min(reqs), max(reqs) + 1
    d = oracle.gated_draft(h["U"], h["W1"], h["W2"], g, c, h["anchor"], w.seed, rnd, x_force=x, b0=b0, b1=b1,
                           bf16_state=True)
    v = oracle.gated_verify(h["T"], h["U"], h["W1"], h["W2"], g, c, h["anchor"], x, ell, w.seed, rnd, b0=b0, b1=b1,
                            bf16_state=True)
    W2 = (h["W2"].astype(np.uint32) << 16).view(np.float32)
    checked = 0
    for b in reqs:
        s = oracle.gated_states(h["W1"], g, c, int(h["anchor"][b]), x[b], w.gamma, bf16_state=True)
        slack = 4 * 2.0 ** -8 * np.abs(s).max() * np.abs(W2).max()
        sure = d["margin"][b] > MARGIN + slack
        assert sure.mean() > 0.5
        assert np.array_equal(d["x"][b][sure], x[b][sure]), (b, x[b].tolist(), d["x"][b].tolist())
        # bf16 weights: lse_k and the drafted token's logit l_k(x_k) within 2e-2
        np.testing.assert_allclose(lse[b], d["lse"][b], rtol=0, atol=2e-2)
        np.testing.assert_allclose(np.log(p[b]) + lse[b], np.log(d["p"][b]) + d["lse"][b], rtol=0, atol=2e-2)
        um = v["umargin"][b]
        um = um[~np.isnan(um)]
        ratio = v["ratio"][b][~np.isnan(v["ratio"][b])]
        if um.size and np.all(um > MARGIN + 4 * slack * np.maximum(ratio, 1.0)):
            assert n[b] == v["n"][b], (b, n[b], v["n"][b])
            if v["ymargin"][b] > MARGIN + 2 * slack:
                assert tok[b] == v["y"][b], (b, tok[b], v["y"][b])
            checked += 1
    return checked


@pytest.mark.parametrize("B", [24, 130])
def test_gated_draft_and_verify_match_the_oracle(B):
    # B = 24: replicated 32-row tiles; B = 130: two 128-row tiles; V = 8200
    # ends in a ragged tile; weight_sigma = 0.1 makes the head's bias matter
    w = wl.custom(B=B, gamma=6, V=8200, r=256, H=64, wdtype=torch.bfloat16, u_sigma=1.5, t_sigma=(0.5, 1.5),
                  weight_sigma=0.1, seed=31)
    inp = _inputs(w)
    ws = _own_ws(w)
    x, p, lse = ds.gated_markov_draft(inp["U"], inp["W1"], inp["W2"], inp["gate_g"], inp["gate_c"], inp["anchor"],
                                      w.seed, 5, ws=ws, T_early=inp["T"])
    ell = torch.full((w.B,), w.gamma, dtype=torch.int32, device=DEV)
    n, tok = ds.verify(inp["T"], inp["U"], inp["W1"], inp["W2"], inp["anchor"], x, p, lse, ell, w.seed, 5, ws,
                       early_stats=True, gated=True)
    torch.cuda.synchronize()
    assert ds.read_status(ws) == ds.OK
    assert _check(w, inp, x, p, lse, n, tok, range(w.B), 5) >= w.B // 2
    # the state carries the prefix: the Markov head scores the same drafted
    # tokens (l_k(x_k) = log p + lse) differently, by more than the tolerance,
    # from position 2 on, and identically at position 1 (s_1 = e_1)
    h = host(inp)
    m = oracle.draft(h["U"], h["W1"], h["W2"], h["anchor"], w.seed, 5, x_force=x.cpu().numpy(), b0=0, b1=8)
    lg = (np.log(p.cpu().numpy()) + lse.cpu().numpy())[:8]
    lm = np.log(m["p"][:8]) + m["lse"][:8]
    assert np.abs(lm[:, 0] - lg[:, 0]).max() < 2e-2
    assert np.abs(lm[:, 1:] - lg[:, 1:]).max() > 0.05


def test_gated_full_vocabulary_sampled():
    w = wl.WORKLOADS["batch128"]
    inp = _inputs(w)
    ws = _own_ws(w)
    x, p, lse = ds.gated_markov_draft(inp["U"], inp["W1"], inp["W2"], inp["gate_g"], inp["gate_c"], inp["anchor"],
                                      w.seed, 2, ws=ws, T_early=inp["T"])
    ell = torch.full((w.B,), w.gamma, dtype=torch.int32, device=DEV)
    n, tok = ds.verify(inp["T"], inp["U"], inp["W1"], inp["W2"], inp["anchor"], x, p, lse, ell, w.seed, 2, ws,
                       early_stats=True, gated=True)
    torch.cuda.synchronize()
    assert ds.read_status(ws) == ds.OK
    _check(w, inp, x, p, lse, n, tok, [0, 1, 64, 127], 2)
