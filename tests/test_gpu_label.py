"""Acceptance labels on the GPU (the study report's confidence-head label, Eq.8:
the probability that rejection sampling accepts a drafted position is the
mass the draft and target distributions share, sum_v min(p_d, p_t)), against
the oracle's draft distribution and acceptance label for the GPU's own drafted
prefix, position by position."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_02_gb300 as ds
from speculative_decoding_02_gb300 import workloads as wl

from _parity import host

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decoding_02_gb300 import build
    build.build()
    ds.library()


def _check(w, inp, out, label, reqs):
    h = host(inp)
    x, ell = out.x.cpu().numpy(), out.ell.cpu().numpy()
    lab = label.cpu().numpy()
    checked = 0
    for b in reqs:
        for k in range(1, w.gamma + 1):
            if k > ell[b]:
                assert lab[b, k - 1] == 0.0, (b, k)
                continue
            prev = int(h["anchor"][b]) if k == 1 else int(x[b, k - 2])
            pd = oracle.draft_probs(h["U"][b, k - 1], h["W1"], h["W2"], prev)
            pt = oracle.softmax(h["T"][b, k - 1])
            want = oracle.acceptance_label(pd, pt)
            assert abs(lab[b, k - 1] - want) <= 2e-4 + 1e-3 * want, (b, k, lab[b, k - 1], want)
            checked += 1
    return checked


def _round(w, inp):
    out = ds.round(inp["U"], inp["T"], inp["W1"], inp["W2"], inp["h"], inp["w"], inp["anchor"], seed=w.seed, rnd=0,
                   sps=inp["sps"], mode=w.mode)
    return out


@pytest.mark.parametrize("B", [24, 130])
def test_labels_match_the_oracle(B):
    # a falling steps-per-second curve makes ell vary across requests; B = 130
    # takes two 128-row tiles, B = 24 replicated rows
    w = wl.custom(B=B, gamma=4, V=8200, r=256, H=64, wdtype=torch.bfloat16, u_sigma=2.5, t_sigma=(0.4, 1.5),
                  seed=17, sps_b0=float(2 * B), sps_kind="steps")
    inp = wl.make_inputs(w, 0, DEV)
    out = _round(w, inp)
    ws = ds.workspace(w.B, w.gamma, w.V, DEV)
    label = ds.acceptance_label(inp["T"], inp["U"], inp["W1"], inp["W2"], inp["anchor"], out.x, out.lse, out.ell,
                                ws=ws)
    torch.cuda.synchronize()
    assert ds.read_status(ws) == ds.OK
    ell = out.ell.cpu().numpy()
    assert 0 < ell.sum() < w.B * w.gamma   # both verified and unverified positions
    assert _check(w, inp, out, label, range(w.B)) == int(ell.sum())
    lab = label.cpu().numpy()
    assert np.all((lab >= 0.0) & (lab <= 1.0 + 1e-5))


def test_labels_full_vocabulary_sampled():
    w = wl.WORKLOADS["batch128"]
    inp = wl.make_inputs(w, 0, DEV)
    out = _round(w, inp)
    ws = ds.workspace(w.B, w.gamma, w.V, DEV)
    label = ds.acceptance_label(inp["T"], inp["U"], inp["W1"], inp["W2"], inp["anchor"], out.x, out.lse, out.ell,
                                ws=ws)
    torch.cuda.synchronize()
    assert ds.read_status(ws) == ds.OK
    assert _check(w, inp, out, label, [0, w.B - 1]) > 0
    del inp
    torch.cuda.empty_cache()
