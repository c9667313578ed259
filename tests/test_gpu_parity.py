"""GPU parity: the CUDA path against the CPU oracle on the same seeded inputs,
through the C ABI.  Small cases are checked element by element (several tiles
and a ragged tail); the full-size workloads on sampled requests."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_02_gb300 as ds
from speculative_decoding_02_gb300 import workloads as wl

from _parity import (MARGIN, check_confidence, check_draft, check_schedule, check_status, check_verify, host,
                     is_bf16, run_round)

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decoding_02_gb300 import build
    build.build()
    ds.library()


def full_check(w, inp, out, rnd=0, reqs=None, chain=True):
    h = host(inp)
    o = {k: v.cpu().numpy() for k, v in out.as_dict().items()}
    bf16 = is_bf16(inp)
    sd = check_draft(h, o["x"], o["p"], o["lse"], w.seed, rnd, bf16, reqs)
    c = check_confidence(h, o["x"], o["c"])
    sps = None if inp["sps"] is None else inp["sps"].cpu().numpy()
    check_schedule(o["c"], sps, w.mode if w.mode != wl.MODE_TOPK else wl.MODE_GREEDY, o["ell"], int(o["nstar"][0]),
                   float(o["theta"][0]))
    sv = check_verify(h, o["x"], o["ell"], o["n"], o["tok"], w.seed, rnd, reqs)
    if chain:
        # the whole chain on the oracle alone, compared up to the first
        # low-margin decision of each request
        B = h["U"].shape[0]
        for b in (range(B) if reqs is None else reqs):
            d = oracle.draft(h["U"], h["W1"], h["W2"], h["anchor"], w.seed, rnd, b0=b, b1=b + 1)
            for k in range(w.gamma):
                if d["margin"][b, k] <= MARGIN:
                    break
                assert d["x"][b, k] == o["x"][b, k]
    return sd, sv, c


def test_tiny_workload_round():
    w = wl.WORKLOADS["tiny"]
    inp = wl.make_inputs(w, 0, DEV)
    out = run_round(inp, w)
    check_status(w, DEV)
    sd, sv, _ = full_check(w, inp, out)
    assert sd["checked"] >= 6 and sv["checked"] >= 1


SMALL = [
    # (B, gamma, V, r, H, dtype, mode) -- several row tiles / vocab slices and ragged tails
    (40, 5, 5000, 64, 128, torch.float32, wl.MODE_GREEDY),
    (40, 5, 5000, 64, 128, torch.bfloat16, wl.MODE_GREEDY),
    (33, 3, 9216, 32, 64, torch.bfloat16, wl.MODE_FIXED),
    (7, 8, 2056, 16, 32, torch.float32, wl.MODE_GREEDY),
    (3, 32, 1032, 256, 256, torch.bfloat16, wl.MODE_FIXED),
    # r = 256 with bf16 weights runs the tensor-core draft: ragged last vocab
    # tile, two M tiles with a ragged second one, several tiles per CTA
    (40, 5, 5000, 256, 128, torch.bfloat16, wl.MODE_GREEDY),
    (130, 3, 2056, 256, 64, torch.bfloat16, wl.MODE_FIXED),
    (33, 2, 16384, 256, 64, torch.bfloat16, wl.MODE_GREEDY),
    (128, 4, 65536, 256, 64, torch.bfloat16, wl.MODE_FIXED),
]


@pytest.mark.parametrize("B,G,V,r,H,dt,mode", SMALL)
def test_small_cases(B, G, V, r, H, dt, mode):
    w = wl.custom(B=B, gamma=G, V=V, r=r, H=H, wdtype=dt, mode=mode, seed=B + G, u_sigma=2.5,
                  t_sigma=(0.4, 1.5), sps_b0=float(4 * B) if mode == wl.MODE_GREEDY else None,
                  sps_kind="steps", w_sigma=0.05)
    inp = wl.make_inputs(w, 0, DEV)
    out = run_round(inp, w)
    check_status(w, DEV)
    full_check(w, inp, out)


def test_degenerate_sizes():
    # one request, one position, the smallest vocabulary
    w = wl.custom(B=1, gamma=1, V=8, r=16, H=8, seed=5)
    inp = wl.make_inputs(w, 0, DEV)
    out = run_round(inp, w)
    check_status(w, DEV)
    full_check(w, inp, out)


def test_verify_zero_lengths_draws_bonus_from_first_row():
    w = wl.custom(B=6, gamma=3, V=2048, r=16, H=16, seed=9)
    inp = wl.make_inputs(w, 0, DEV)
    x, p, lse = ds.markov_draft(inp["U"], inp["W1"], inp["W2"], inp["anchor"], w.seed, 0)
    ell = torch.zeros(w.B, dtype=torch.int32, device=DEV)
    n, tok = ds.verify(inp["T"], inp["U"], inp["W1"], inp["W2"], inp["anchor"], x, p, lse, ell, w.seed, 0)
    torch.cuda.synchronize()
    assert torch.all(n == 0)
    T = inp["T"].cpu().numpy()
    for b in range(w.B):
        y, m = oracle.softmax_draw(T[b, 0].astype(np.float64), w.seed, 0, 3, b, 1)
        if m > MARGIN:
            assert int(tok[b]) == y


def test_identical_distributions_accept_everything():
    # W2 = 0 and target rows equal to the backbone rows: p_t == p_d, every
    # drafted token is accepted and the bonus row is used
    w = wl.custom(B=5, gamma=4, V=4096, r=16, H=16, seed=11)
    inp = wl.make_inputs(w, 0, DEV)
    inp["W2"].zero_()
    inp["T"][:, :w.gamma] = inp["U"]
    x, p, lse = ds.markov_draft(inp["U"], inp["W1"], inp["W2"], inp["anchor"], w.seed, 0)
    ell = torch.tensor([4, 3, 0, 2, 4], dtype=torch.int32, device=DEV)
    n, tok = ds.verify(inp["T"], inp["U"], inp["W1"], inp["W2"], inp["anchor"], x, p, lse, ell, w.seed, 0)
    torch.cuda.synchronize()
    assert torch.equal(n, ell)


def test_bad_anchor_and_nonfinite_logits_set_status():
    w = wl.custom(B=2, gamma=2, V=1024, r=16, H=8, seed=1)
    inp = wl.make_inputs(w, 0, DEV)
    ws = ds.workspace(w.B, w.gamma, w.V, DEV)
    ds.read_status(ws)
    bad = inp["anchor"].clone()
    bad[1] = w.V + 5
    ds.markov_draft(inp["U"], inp["W1"], inp["W2"], bad, w.seed, 0, ws=ws)
    assert ds.read_status(ws) == ds.ERR_INVALID
    U = inp["U"].clone()
    U[0, 1, 17] = float("nan")
    ds.markov_draft(U, inp["W1"], inp["W2"], inp["anchor"], w.seed, 0, ws=ws)
    assert ds.read_status(ws) == ds.ERR_NONFINITE
    ds.markov_draft(inp["U"], inp["W1"], inp["W2"], inp["anchor"], w.seed, 0, ws=ws)
    assert ds.read_status(ws) == ds.OK


@pytest.mark.parametrize("R,G", [(1, 1), (3, 4), (128, 16), (512, 5), (256, 32), (64, 8)])
def test_schedule_parity(R, G):
    rng = np.random.default_rng(R * 100 + G)
    n = R * (G + 1) + 1
    b = np.arange(n, dtype=np.float64)
    tables = [(b / (1 + b / 256.0)), 1.0 / (1.0 + b / (R * 2.0)), np.maximum(1.0 - b / (2.0 * n), 0.05)]
    for trial in range(4):
        c = rng.uniform(0.0, 1.0, (R, G)).astype(np.float32)
        if trial == 1:
            c = (1.0 / (1.0 + np.exp(-rng.normal(0, 5, (R, G))))).astype(np.float32)
        if trial == 2:
            c = np.round(c, 1)
        if trial == 3:
            c[:] = 1.0
        for sps in tables:
            sps = sps.astype(np.float32)
            for mode, K in [(wl.MODE_GREEDY, -1), (wl.MODE_FIXED, -1)]:
                ell, nstar, theta = ds.schedule(torch.from_numpy(c).to(DEV), torch.from_numpy(sps).to(DEV), mode)
                torch.cuda.synchronize()
                check_schedule(c, sps, mode, ell.cpu().numpy(), int(nstar[0]), float(theta[0]))


def test_topk_history_ring():
    R, G = 64, 5
    rng = np.random.default_rng(0)
    sps = (1.0 / (1.0 + np.arange(R * (G + 1) + 1) / 100.0)).astype(np.float32)
    sps_d = torch.from_numpy(sps).to(DEV)
    khist = torch.zeros(2, dtype=torch.int32, device=DEV)
    greedy = []
    for t in range(6):
        c = rng.uniform(0.2, 1.0, (R, G)).astype(np.float32)
        ell, nstar, theta = ds.schedule(torch.from_numpy(c).to(DEV), sps_d, wl.MODE_TOPK, rnd=t, khist=khist)
        torch.cuda.synchronize()
        g = oracle.schedule(c.astype(np.float64), sps, oracle.MODE_GREEDY)
        greedy.append(g["nstar"])
        assert int(nstar[0]) == g["nstar"]
        if t < 2:
            assert np.array_equal(ell.cpu().numpy(), g["ell"])
        else:
            o = oracle.schedule(c.astype(np.float64), sps, oracle.MODE_TOPK, K=greedy[t - 2])
            assert np.array_equal(ell.cpu().numpy(), o["ell"])
            assert int(ell.sum()) == min(greedy[t - 2], R * G)


def test_gpu_sampling_law_chi_square():
    # V = 8 with a peaked Markov bias: the GPU's first emitted token (draft,
    # then verification against a different target) follows the target law
    B, G, V, r = 40000, 2, 8, 16
    gen = torch.Generator(device="cpu").manual_seed(3)
    U1 = torch.randn(1, G, V, generator=gen) * 1.2
    T1 = torch.randn(1, G + 1, V, generator=gen) * 1.2
    W1 = (torch.randn(V, r, generator=gen) * 0.5)
    W2 = (torch.randn(V, r, generator=gen) * 0.5)
    U = U1.expand(B, G, V).contiguous().to(DEV)
    T = T1.expand(B, G + 1, V).contiguous().to(DEV)
    anchor = torch.full((B,), 2, dtype=torch.int32, device=DEV)
    W1d, W2d = W1.to(DEV), W2.to(DEV)
    x, p, lse = ds.markov_draft(U, W1d, W2d, anchor, 77, 5)
    ell = torch.full((B,), 1, dtype=torch.int32, device=DEV)
    n, tok = ds.verify(T, U, W1d, W2d, anchor, x, p, lse, ell, 77, 5)
    torch.cuda.synchronize()
    first = torch.where(n >= 1, x[:, 0], tok).cpu().numpy()
    # T here does not depend on the drafted prefix, so the first emitted token
    # must follow softmax(T row 0)
    pt = torch.softmax(T1[0, 0].double(), 0).numpy()
    cnt = np.bincount(first, minlength=V)
    from scipy import stats
    chi2 = ((cnt - pt * B) ** 2 / (pt * B)).sum()
    assert stats.chi2.sf(chi2, V - 1) > 1e-4
    # acceptance rate of position 1 matches sum_v min(p_d, p_t) (Eq.8)
    pd = oracle.draft_probs(U1[0, 0].numpy(), W1.numpy(), W2.numpy(), 2)
    lab = oracle.acceptance_label(pd, pt)
    rate = float((n >= 1).float().mean())
    assert abs(rate - lab) < 3.3 * np.sqrt(lab * (1 - lab) / B)
    # the first two emitted tokens at ell = 2: a request that stops short is
    # extended by sampling the target on the host, and since T does not depend
    # on the prefix the pair follows softmax(T row 0) x softmax(T row 1)
    ell2 = torch.full((B,), 2, dtype=torch.int32, device=DEV)
    n2, tok2 = ds.verify(T, U, W1d, W2d, anchor, x, p, lse, ell2, 77, 5)
    torch.cuda.synchronize()
    n2, tok2, xh = n2.cpu().numpy(), tok2.cpu().numpy(), x.cpu().numpy()
    pt1 = torch.softmax(T1[0, 1].double(), 0).numpy()
    ext = np.random.default_rng(11).choice(V, size=B, p=pt1)
    s1 = np.where(n2 >= 1, xh[:, 0], tok2)
    s2 = np.where(n2 >= 2, xh[:, 1], np.where(n2 == 1, tok2, ext))
    e = np.outer(pt, pt1).ravel() * B
    cnt2 = np.bincount(s1 * V + s2, minlength=V * V)
    assert e.min() > 5
    assert stats.chi2.sf(((cnt2 - e) ** 2 / e).sum(), V * V - 1) > 1e-4


FULL = ["qwen3_4b", "batch128", "large_vocab", "serving512"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_workload_sampled(name):
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w, 0, DEV)
    out = run_round(inp, w)
    check_status(w, DEV)
    reqs = sorted({0, 1, w.B // 2, w.B - 1})
    sd, sv, _ = full_check(w, inp, out, reqs=reqs, chain=False)
    assert sd["checked"] > 0 and sv["checked"] + sv["low_margin"] == len(reqs)
    # properties over every request
    o = out.as_dict()
    assert torch.all((o["x"] >= 0) & (o["x"] < w.V))
    assert torch.all((o["n"] >= 0) & (o["n"] <= o["ell"]))
    assert torch.all((o["tok"] >= 0) & (o["tok"] < w.V))
    assert torch.all((o["p"] > 0) & (o["p"] <= 1))
    del inp
    torch.cuda.empty_cache()
