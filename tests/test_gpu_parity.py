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
                     is_bf16, ranges, run_round)

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
        # the whole chain on the oracle alone (no teacher forcing), compared up
        # to the first low-margin decision of each request
        B = h["U"].shape[0]
        for b0, b1 in ranges(reqs, B):
            d = oracle.draft(h["U"], h["W1"], h["W2"], h["anchor"], w.seed, rnd, b0=b0, b1=b1)
            for b in range(b0, b1):
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


CHAIN = [
    # (B, gamma, V, r, dtype): tensor-core and CUDA-core drafts, a ragged last
    # segment (V % 2048), several lists deep, gamma = 1
    (40, 5, 5000, 256, torch.bfloat16),
    (130, 8, 9000, 256, torch.bfloat16),
    (33, 6, 4104, 64, torch.float32),
    (9, 1, 2056, 16, torch.float32),
]


@pytest.mark.parametrize("B,G,V,r,dt", CHAIN)
def test_chain_verification_equals_the_full_row_pass(B, G, V, r, dt):
    # verification along the accept chains reads only the rows its tests
    # reach; the full row pass reads every row j < ell first.  The accept
    # tests, the residual and the bonus draws are the same, and so are the
    # results (the two passes sum a row's softmax in different segments, so
    # they agree to float rounding, far inside every decision's margin here)
    w = wl.custom(B=B, gamma=G, V=V, r=r, H=64, wdtype=dt, mode=wl.MODE_GREEDY, seed=B + 5 * G, u_sigma=2.5,
                  t_sigma=(0.4, 1.5), sps_b0=float(4 * B), sps_kind="steps", w_sigma=0.05)
    inp = wl.make_inputs(w, 0, DEV)
    chain = run_round(inp, w)
    check_status(w, DEV)
    full = run_round(inp, w, all_row_stats=True)
    check_status(w, DEV)
    for name in ("x", "p", "lse", "c", "ell", "n", "tok"):
        assert torch.equal(chain.as_dict()[name], full.as_dict()[name]), name
    n, ell = chain.n.cpu().numpy(), chain.ell.cpu().numpy()
    assert (n < ell).any() and (n == ell).any()   # rejections and whole accepts
    full_check(w, inp, chain, chain=False)


def test_chain_verification_reads_no_row_past_a_rejection():
    # every target row past each request's rejected position is set to +inf:
    # verification along the accept chains never reads one, so it returns the
    # same results with no error; the full row pass reads them and reports a
    # non-finite logit
    w = wl.custom(B=48, gamma=6, V=6000, r=256, H=64, wdtype=torch.bfloat16, mode=wl.MODE_FIXED, seed=29,
                  u_sigma=2.5, t_sigma=(0.4, 1.5), sps_b0=None)
    inp = wl.make_inputs(w, 0, DEV)
    ws = ds.workspace(w.B, w.gamma, w.V, DEV)
    x, p, lse = ds.markov_draft(inp["U"], inp["W1"], inp["W2"], inp["anchor"], w.seed, 0, ws=ws)
    ell = torch.full((w.B,), w.gamma, dtype=torch.int32, device=DEV)
    args = (inp["U"], inp["W1"], inp["W2"], inp["anchor"], x, p, lse, ell, w.seed, 0, ws)
    n0, tok0 = ds.verify(inp["T"], *args)
    torch.cuda.synchronize()
    assert ds.read_status(ws) == ds.OK
    n_host = n0.cpu().numpy()
    assert (n_host < w.gamma - 1).sum() >= w.B // 4   # most requests leave rows unread
    T = inp["T"].clone()
    for b in range(w.B):
        if n_host[b] < w.gamma:
            T[b, n_host[b] + 1:w.gamma] = float("inf")
    n1, tok1 = ds.verify(T, *args)
    torch.cuda.synchronize()
    assert ds.read_status(ws) == ds.OK
    assert torch.equal(n0, n1) and torch.equal(tok0, tok1)
    ds.verify(T, *args, all_row_stats=True)
    torch.cuda.synchronize()
    assert ds.read_status(ws) == ds.ERR_NONFINITE


CHAIN_STATS = [
    # (B, gamma, V): replicated 64- and 32-row tiles, two 128-row tiles,
    # one and several statistics segments per row with a ragged last one,
    # gamma = 16
    (40, 5, 5000),
    (24, 6, 40000),
    (130, 8, 9000),
    (128, 16, 33000),
]


@pytest.mark.parametrize("B,G,V", CHAIN_STATS)
def test_chain_statistics_round_equals_the_early_round(B, G, V):
    # the draft takes the statistics only of the rows the accept tests can
    # reach (it runs those tests itself as their inputs come out and skips a
    # row once its request is certain to stop before it); the rows it takes
    # get the same partials as when it takes every row j < gamma, so the
    # round's results are the early round's bit for bit
    w = wl.custom(B=B, gamma=G, V=V, r=256, H=64, wdtype=torch.bfloat16, mode=wl.MODE_GREEDY, seed=B + 7 * G,
                  u_sigma=2.5, t_sigma=(0.4, 1.5), sps_b0=float(4 * B), sps_kind="steps", w_sigma=0.05)
    inp = wl.make_inputs(w, 0, DEV)
    ws = ds.workspace(w.B, w.gamma, w.V, DEV)
    early = run_round(inp, w, early_stats=True, ws=ws)
    assert ds.read_status(ws) == ds.OK
    # another round on the same workspace first, so that every partial the
    # round under test reads too early would be a different round's
    run_round(inp, w, rnd=3, chain_stats=True, ws=ws)
    lazy = run_round(inp, w, chain_stats=True, ws=ws)
    assert ds.read_status(ws) == ds.OK
    for name in ("x", "p", "lse", "c", "ell", "n", "tok"):
        assert torch.equal(lazy.as_dict()[name], early.as_dict()[name]), name
    n, ell = lazy.n.cpu().numpy(), lazy.ell.cpu().numpy()
    assert (n < ell).any() and (n == ell).any()   # rejections and whole accepts


def test_chain_statistics_round_skips_rows_past_a_rejection():
    # every target row past each request's rejected position is set to +inf.
    # The draft that takes the chains' rows reads few of them (any it reads
    # ahead of a decision are not used) and verification checks only the rows
    # its tests use, so the round returns the same results with no error; the
    # draft that takes every row reports the non-finite logits; the label call
    # refuses the chains' statistics, which do not cover every row
    w = wl.custom(B=48, gamma=6, V=6000, r=256, H=64, wdtype=torch.bfloat16, mode=wl.MODE_FIXED, seed=29,
                  u_sigma=2.5, t_sigma=(0.4, 1.5), sps_b0=None)
    inp = wl.make_inputs(w, 0, DEV)
    ws = ds.workspace(w.B, w.gamma, w.V, DEV)
    ref = run_round(inp, w, chain_stats=True, ws=ws)
    assert ds.read_status(ws) == ds.OK
    n_host = ref.n.cpu().numpy()
    assert (n_host < w.gamma - 1).sum() >= w.B // 4   # most requests leave rows unread
    T = inp["T"].clone()
    for b in range(w.B):
        if n_host[b] < w.gamma:
            T[b, n_host[b] + 1:w.gamma] = float("inf")
    lazy = run_round(inp, w, chain_stats=True, T=T, ws=ws)
    assert ds.read_status(ws) == ds.OK
    for name in ("x", "p", "lse", "c", "ell", "n", "tok"):
        assert torch.equal(lazy.as_dict()[name], ref.as_dict()[name]), name
    ds.acceptance_label(T, inp["U"], inp["W1"], inp["W2"], inp["anchor"], lazy.x, lazy.lse, lazy.ell, ws=ws,
                        stats="early")
    assert ds.read_status(ws) == ds.ERR_INVALID
    run_round(inp, w, early_stats=True, T=T, ws=ws)
    assert ds.read_status(ws) == ds.ERR_NONFINITE


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


EARLY = [
    # (B, gamma, V, r, dtype, mode): tensor-core draft (persistent launch, the
    # statistics warps), CUDA-core draft (statistics after the draft), a
    # truncating schedule (rows past ell read but not used)
    (40, 5, 5000, 256, torch.bfloat16, wl.MODE_GREEDY),
    (128, 4, 65536, 256, torch.bfloat16, wl.MODE_FIXED),
    (130, 3, 2056, 256, torch.bfloat16, wl.MODE_FIXED),
    (40, 5, 5000, 64, torch.float32, wl.MODE_GREEDY),
]


@pytest.mark.parametrize("B,G,V,r,dt,mode", EARLY)
def test_stages_called_one_by_one_equal_the_round(B, G, V, r, dt, mode):
    # markov_draft(T_early) + confidence + schedule + verify(early_stats) on
    # one workspace, each call separate (verification clears its own scratch):
    # the same bits as the round, whose first stage clears that scratch and
    # leaves T at the drafted tokens and the row statistics for verification
    w = wl.custom(B=B, gamma=G, V=V, r=r, H=64, wdtype=dt, mode=mode, u_sigma=2.0, seed=71, sps_b0=float(B))
    inp = wl.make_inputs(w, 0, DEV)
    ref = run_round(inp, w, rnd=4, early_stats=True)
    ws = ds.workspace(w.B, w.gamma, w.V, DEV)
    x, p, lse = ds.markov_draft(inp["U"], inp["W1"], inp["W2"], inp["anchor"], w.seed, 4, ws=ws, T_early=inp["T"])
    c = ds.confidence(inp["h"], inp["W1"], inp["w"], inp["anchor"], x)
    khist = torch.zeros(2, dtype=torch.int32, device=DEV) if mode == wl.MODE_TOPK else None
    ell, _, _ = ds.schedule(c, inp["sps"], mode, 4, khist, ws)
    # twice on the same workspace: each call starts its scratch (the bonus
    # list, the keys) afresh
    for _ in range(2):
        n, tok = ds.verify(inp["T"], inp["U"], inp["W1"], inp["W2"], inp["anchor"], x, p, lse, ell, w.seed, 4, ws,
                           early_stats=True)
        torch.cuda.synchronize()
        assert ds.read_status(ws) == ds.OK
        for name, got in (("x", x), ("p", p), ("lse", lse), ("c", c), ("ell", ell), ("n", n), ("tok", tok)):
            assert torch.equal(ref.as_dict()[name], got), name


@pytest.mark.parametrize("B,G,V,r,dt,mode", EARLY)
def test_early_target_stats_round(B, G, V, r, dt, mode):
    w = wl.custom(B=B, gamma=G, V=V, r=r, H=64, wdtype=dt, mode=mode, seed=B + 3 * G, u_sigma=2.5,
                  t_sigma=(0.4, 1.5), sps_b0=float(4 * B) if mode == wl.MODE_GREEDY else None,
                  sps_kind="steps", w_sigma=0.05)
    inp = wl.make_inputs(w, 0, DEV)
    base = run_round(inp, w)
    check_status(w, DEV)
    early = run_round(inp, w, early_stats=True)
    check_status(w, DEV)
    # the draft, confidence and schedule do not change; verification reads
    # statistics taken earlier by other warps
    for name in ("x", "p", "lse", "c", "ell"):
        assert torch.equal(base.as_dict()[name], early.as_dict()[name]), name
    full_check(w, inp, early, chain=False)


def test_early_target_stats_fallback_launch():
    # 153 M tiles of 128 requests: more CTAs than SMs, so the tensor-core draft
    # runs one launch per position and the statistics follow it
    w = wl.custom(B=153 * 128, gamma=2, V=256, r=256, H=8, wdtype=torch.bfloat16, mode=wl.MODE_FIXED, seed=21,
                  u_sigma=2.0, t_sigma=(0.5,), sps_b0=None)
    inp = wl.make_inputs(w, 0, DEV)
    out = run_round(inp, w, early_stats=True)
    check_status(w, DEV)
    reqs = list(range(16)) + list(range(w.B - 16, w.B))
    full_check(w, inp, out, reqs=reqs, chain=False)


def test_verify_with_missing_early_stats_is_reported():
    # verify(early_stats=True) after a draft that did not take the statistics
    w = wl.custom(B=8, gamma=3, V=1024, r=256, H=8, wdtype=torch.bfloat16, seed=2)
    inp = wl.make_inputs(w, 0, DEV)
    ws = ds.workspace(w.B, w.gamma, w.V, DEV)
    ds.read_status(ws)
    x, p, lse = ds.markov_draft(inp["U"], inp["W1"], inp["W2"], inp["anchor"], w.seed, 0, ws=ws)
    ell = torch.full((w.B,), w.gamma, dtype=torch.int32, device=DEV)
    ds.verify(inp["T"], inp["U"], inp["W1"], inp["W2"], inp["anchor"], x, p, lse, ell, w.seed, 0, ws=ws,
              early_stats=True)
    assert ds.read_status(ws) == ds.ERR_INVALID
    # with the statistics taken by the draft the same call is clean
    x, p, lse = ds.markov_draft(inp["U"], inp["W1"], inp["W2"], inp["anchor"], w.seed, 0, ws=ws, T_early=inp["T"])
    ds.verify(inp["T"], inp["U"], inp["W1"], inp["W2"], inp["anchor"], x, p, lse, ell, w.seed, 0, ws=ws,
              early_stats=True)
    assert ds.read_status(ws) == ds.OK


def test_gpu_sampling_law_chi_square_tensor_cores():
    # The product path: bf16 W1/W2 of rank 256, V = 256 (four 64-column
    # tiles), 152 M tiles of 128 requests (the persistent cooperative draft
    # with its 16-bit block screen, the tensor-core residual).  The mass sits
    # on eight tokens in different blocks; the first emitted token must follow
    # softmax(T row 0) and the first two the product of rows 0 and 1.
    from scipy import stats
    B, G, V, r = 152 * 128, 2, 256, 256
    heavy = np.array([3, 37, 70, 101, 130, 166, 200, 250])
    gen = torch.Generator(device="cpu").manual_seed(8)

    def rows(n, sd):
        t = torch.full((n, V), -6.0) + torch.randn(n, V, generator=gen) * 0.5
        t[:, heavy] = torch.randn(n, len(heavy), generator=gen) * sd
        return t

    U1, T1 = rows(G, 1.0), rows(G + 1, 0.7)
    W1 = (torch.randn(V, r, generator=gen) * 0.25).to(torch.bfloat16)
    W2 = (torch.randn(V, r, generator=gen) * 0.25).to(torch.bfloat16)
    U = U1.unsqueeze(0).expand(B, G, V).contiguous().to(DEV)
    T = T1.unsqueeze(0).expand(B, G + 1, V).contiguous().to(DEV)
    anchor = torch.full((B,), 5, dtype=torch.int32, device=DEV)
    W1d, W2d = W1.to(DEV), W2.to(DEV)

    def cell(tok):
        c = np.full(tok.shape, len(heavy))
        for i, hv in enumerate(heavy):
            c[tok == hv] = i
        return c

    def probs(row):
        p = torch.softmax(row.double(), 0).numpy()
        return np.append(p[heavy], 1.0 - p[heavy].sum())

    pt0, pt1 = probs(T1[0]), probs(T1[1])
    firsts, pairs, accepted = [], [], 0
    ext_rng = np.random.default_rng(17)
    for rnd in (5, 6):
        x, p, lse = ds.markov_draft(U, W1d, W2d, anchor, 91, rnd)
        ell = torch.full((B,), 2, dtype=torch.int32, device=DEV)
        n, tok = ds.verify(T, U, W1d, W2d, anchor, x, p, lse, ell, 91, rnd)
        torch.cuda.synchronize()
        n, tok, xh = n.cpu().numpy(), tok.cpu().numpy(), x.cpu().numpy()
        s1 = np.where(n >= 1, xh[:, 0], tok)
        ext = ext_rng.choice(V, size=B, p=torch.softmax(T1[1].double(), 0).numpy())
        s2 = np.where(n >= 2, xh[:, 1], np.where(n == 1, tok, ext))
        firsts.append(cell(s1))
        pairs.append(cell(s1) * (len(heavy) + 1) + cell(s2))
        accepted += int((n >= 1).sum())
    first, pair = np.concatenate(firsts), np.concatenate(pairs)
    N = first.size
    cnt = np.bincount(first, minlength=len(heavy) + 1)
    e = pt0 * N
    assert e.min() > 5
    assert stats.chi2.sf(((cnt - e) ** 2 / e).sum(), len(heavy)) > 1e-4
    e2 = np.outer(pt0, pt1).ravel() * N
    cnt2 = np.bincount(pair, minlength=e2.size)
    assert e2.min() > 5
    assert stats.chi2.sf(((cnt2 - e2) ** 2 / e2).sum(), e2.size - 1) > 1e-4
    # position 1 is accepted at the rate sum_v min(p_d, p_t) (Eq.8)
    pd = oracle.draft_probs(U1[0].numpy(), wl.to_numpy(W1), wl.to_numpy(W2), 5)
    lab = oracle.acceptance_label(pd, torch.softmax(T1[0].double(), 0).numpy())
    rate = accepted / N
    assert abs(rate - lab) < 3.3 * np.sqrt(lab * (1 - lab) / N)


FULL = ["qwen3_4b", "batch128", "large_vocab", "serving512"]


@pytest.mark.parametrize("name", ["batch128", "serving512"])
def test_full_size_chain_statistics_round(name):
    # the benchmark's headline form at full size: the draft taking the rows
    # the accept chains reach gives the early round's results bit for bit
    # (after a different round on the same workspace), which the test below
    # holds against the oracle on sampled requests
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w, 0, DEV)
    ws = ds.workspace(w.B, w.gamma, w.V, DEV)
    early = run_round(inp, w, early_stats=True, ws=ws)
    assert ds.read_status(ws) == ds.OK
    run_round(inp, w, rnd=5, chain_stats=True, ws=ws)
    lazy = run_round(inp, w, chain_stats=True, ws=ws)
    assert ds.read_status(ws) == ds.OK
    for name_ in ("x", "p", "lse", "c", "ell", "n", "tok"):
        assert torch.equal(lazy.as_dict()[name_], early.as_dict()[name_]), name_
    del inp, ws
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", FULL)
def test_full_size_workload_sampled(name):
    # the round as the benchmark runs it: the draft takes the target rows'
    # statistics on the tensor-core path
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w, 0, DEV)
    out = run_round(inp, w, early_stats=True)
    check_status(w, DEV)
    # 16 requests (two runs of 8 at both ends of the batch), teacher-forced
    # and as a whole chain
    reqs = list(range(8)) + list(range(w.B - 8, w.B)) if w.B > 16 else list(range(w.B))
    if name == "batch128":
        sig = inp["target_sigma"].cpu().numpy().astype(np.float64)[reqs]
        assert set(np.round(sig, 3).tolist()) == {0.3, 1.0, 2.0}, "every target-noise class among the checked requests"
    sd, sv, _ = full_check(w, inp, out, reqs=reqs, chain=True)
    assert sd["checked"] > 0 and sv["checked"] + sv["low_margin"] == len(reqs)
    # properties over every request
    o = out.as_dict()
    assert torch.all((o["x"] >= 0) & (o["x"] < w.V))
    assert torch.all((o["n"] >= 0) & (o["n"] <= o["ell"]))
    assert torch.all((o["tok"] >= 0) & (o["tok"] < w.V))
    assert torch.all((o["p"] > 0) & (o["p"] <= 1))
    del inp
    torch.cuda.empty_cache()
