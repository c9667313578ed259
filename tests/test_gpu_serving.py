"""The serving loop on the GPU: 100 consecutive rounds of the high-concurrency
workload (B = 512, gamma = 5, V = 129280) with the asynchronous top-K schedule
([blog] section 7: round t admits the K_t = n*_{t-2} best candidates, n* being
the greedy count of round t - 2, kept in a two-entry device ring).  Every
round's schedule is checked against the oracle on the GPU's own confidences;
rounds 0-3 and 99 are checked end to end on sampled requests."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_02_gb300 as ds
from speculative_decoding_02_gb300 import workloads as wl

from _parity import check_confidence, check_draft, check_verify, host, is_bf16

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decoding_02_gb300 import build
    build.build()
    ds.library()


def test_hundred_rounds_topk_from_two_rounds_back():
    # a falling steps-per-second curve, so that the greedy count truncates
    w = dataclasses.replace(wl.WORKLOADS["serving512"], name="serving512_steps", sps_kind="steps")
    weights = wl.make_weights(w, DEV)
    sps_d = wl.sps_table(w).to(DEV)
    sps = sps_d.cpu().numpy()
    khist = torch.zeros(2, dtype=torch.int32, device=DEV)
    out = ds.RoundOutputs(w.B, w.gamma, DEV)
    ws = ds.workspace(w.B, w.gamma, w.V, DEV)
    greedy = []
    full = {0, 1, 2, 3, 99}
    reqs = [0, 1, w.B // 2, w.B - 1]
    for rnd in range(100):
        rin = wl.make_round_inputs(w, rnd, DEV)
        ds.round(rin["U"], rin["T"], weights["W1"], weights["W2"], rin["h"], weights["w"], weights["anchor"],
                 seed=w.seed, rnd=rnd, sps=sps_d, mode=wl.MODE_TOPK, khist=khist, out=out, ws=ws)
        torch.cuda.synchronize()
        assert ds.read_status(ws) == ds.OK, f"round {rnd}"
        c = out.c.cpu().numpy().astype(np.float64)
        ell = out.ell.cpu().numpy()
        g = oracle.schedule(c, sps, oracle.MODE_GREEDY)
        greedy.append(g["nstar"])
        assert int(out.nstar.cpu()[0]) == g["nstar"], f"round {rnd}: greedy count"
        if rnd < 2:
            assert np.array_equal(ell, g["ell"]), f"round {rnd}: synchronous greedy"
        else:
            o = oracle.schedule(c, sps, oracle.MODE_TOPK, K=greedy[rnd - 2])
            assert np.array_equal(ell, o["ell"]), f"round {rnd}: top-K from round {rnd - 2}"
            assert int(ell.sum()) == min(greedy[rnd - 2], w.B * w.gamma)
        if rnd in full:
            # draft, confidence and verification of sampled requests against
            # the oracle, each teacher-forced on the GPU's upstream outputs
            inp = dict(weights)
            inp.update(rin)
            h = host(inp)
            o = {k: v.cpu().numpy() for k, v in out.as_dict().items()}
            sd = check_draft(h, o["x"], o["p"], o["lse"], w.seed, rnd, is_bf16(inp), reqs)
            check_confidence(h, o["x"], o["c"])
            sv = check_verify(h, o["x"], o["ell"], o["n"], o["tok"], w.seed, rnd, reqs)
            assert sd["checked"] > 0 and sv["checked"] + sv["low_margin"] == len(reqs)
        del rin
    # the schedule really truncates on this curve, and the history moved
    assert min(greedy) < w.B * w.gamma
    assert len(set(greedy)) > 1
