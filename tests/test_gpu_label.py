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


def _round(w, inp, ws=None, early=False, all_rows=False):
    return ds.round(inp["U"], inp["T"], inp["W1"], inp["W2"], inp["h"], inp["w"], inp["anchor"], seed=w.seed, rnd=0,
                    sps=inp["sps"], mode=w.mode, ws=ws, early_stats=early, all_row_stats=all_rows)


def _labels(w, inp, stats):
    # stats None: the label call streams the target rows' statistics itself;
    # "early": the round's draft took them; "verify": the round's verification
    # did, over every row j < ell (both on the workspace the label call is
    # given)
    ws = ds.workspace(w.B, w.gamma, w.V, DEV)
    out = _round(w, inp, ws=ws if stats else None, early=stats == "early", all_rows=stats == "verify")
    label = ds.acceptance_label(inp["T"], inp["U"], inp["W1"], inp["W2"], inp["anchor"], out.x, out.lse, out.ell,
                                ws=ws, stats=stats)
    torch.cuda.synchronize()
    assert ds.read_status(ws) == ds.OK
    return out, label


@pytest.mark.parametrize("stats", [None, "early", "verify"])
@pytest.mark.parametrize("B", [24, 60, 130])
def test_labels_match_the_oracle(B, stats):
    # a falling steps-per-second curve makes ell vary across requests; B = 130
    # takes two 128-row tiles, B = 24 and 60 replicated rows (32 and 64 per
    # tile); V = 8200 ends in a ragged 8-column tile
    w = wl.custom(B=B, gamma=4, V=8200, r=256, H=64, wdtype=torch.bfloat16, u_sigma=2.5, t_sigma=(0.4, 1.5),
                  seed=17, sps_b0=float(2 * B), sps_kind="steps")
    inp = wl.make_inputs(w, 0, DEV)
    out, label = _labels(w, inp, stats)
    ell = out.ell.cpu().numpy()
    assert 0 < ell.sum() < w.B * w.gamma   # both verified and unverified positions
    assert _check(w, inp, out, label, range(w.B)) == int(ell.sum())
    lab = label.cpu().numpy()
    assert np.all((lab >= 0.0) & (lab <= 1.0 + 1e-5))


def test_label_sources_agree():
    # the three sources of the target rows' statistics give labels within
    # float rounding of one another (the partials differ only in segment size)
    w = wl.custom(B=40, gamma=3, V=40000, r=256, H=64, wdtype=torch.bfloat16, u_sigma=2.0, t_sigma=(0.5, 1.2),
                  seed=5, sps_b0=1e6)
    inp = wl.make_inputs(w, 0, DEV)
    labs = [_labels(w, inp, s)[1] for s in (None, "early", "verify")]
    for lab in labs[1:]:
        torch.testing.assert_close(lab, labs[0], rtol=1e-4, atol=1e-6)


def test_missing_early_statistics_are_reported():
    # a round whose draft did not take the statistics leaves the draft's count
    # of row segments at zero: the label call with stats="early" reports it
    w = wl.custom(B=8, gamma=2, V=4096, r=256, H=64, wdtype=torch.bfloat16, seed=3, sps_b0=1e6)
    inp = wl.make_inputs(w, 0, DEV)
    ws = ds.workspace(w.B, w.gamma, w.V, DEV)
    out = _round(w, inp, ws=ws, early=False)
    ds.acceptance_label(inp["T"], inp["U"], inp["W1"], inp["W2"], inp["anchor"], out.x, out.lse, out.ell, ws=ws,
                        stats="early")
    torch.cuda.synchronize()
    assert ds.read_status(ws) == ds.ERR_INVALID


def test_statistics_of_a_chain_verification_are_refused():
    # a verification along the accept chains reads only the rows its tests
    # reach: the label call that would reuse its statistics reports it
    w = wl.custom(B=8, gamma=3, V=4096, r=256, H=64, wdtype=torch.bfloat16, seed=3, sps_b0=1e6)
    inp = wl.make_inputs(w, 0, DEV)
    ws = ds.workspace(w.B, w.gamma, w.V, DEV)
    out = _round(w, inp, ws=ws)
    ds.acceptance_label(inp["T"], inp["U"], inp["W1"], inp["W2"], inp["anchor"], out.x, out.lse, out.ell, ws=ws,
                        stats="verify")
    torch.cuda.synchronize()
    assert ds.read_status(ws) == ds.ERR_INVALID


def test_labels_full_vocabulary_sampled():
    w = wl.WORKLOADS["batch128"]
    inp = wl.make_inputs(w, 0, DEV)
    out, label = _labels(w, inp, "early")
    assert _check(w, inp, out, label, [0, 37, 64, 101, w.B - 1]) > 0
    del inp
    torch.cuda.empty_cache()
