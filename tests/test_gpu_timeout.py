"""Failure detection on the GPU without a fault: a kernel whose wait nothing
satisfies gives up after the library's bounded-wait limit, records
DSPARK_ERR_TIMEOUT in the workspace status word and returns, and the CUDA
context stays usable for the next round."""
import time

import pytest
import torch

import speculative_decoding_02_gb300 as ds
from speculative_decoding_02_gb300 import workloads as wl

from _parity import check_status, host, check_draft, run_round

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decoding_02_gb300 import build
    build.build()
    ds.library()


@pytest.mark.parametrize("mode", [0, 1], ids=["mbarrier", "grid_barrier"])
def test_bounded_wait_gives_up_and_context_survives(mode):
    ws = ds.workspace(8, 4, 1024, DEV)
    assert ds.read_status(ws) == ds.OK
    t0 = time.perf_counter()
    ds.selftest_wait_timeout(mode, ws)
    st = ds.read_status(ws)          # synchronises the stream
    dt = time.perf_counter() - t0
    assert st == ds.ERR_TIMEOUT
    assert 0.9 < dt < 30.0, f"the wait gave up after {dt:.2f} s"
    assert ds.read_status(ws) == ds.OK   # reading clears the word
    # the context still runs a round that matches the oracle
    w = wl.WORKLOADS["tiny"]
    inp = wl.make_inputs(w, 0, DEV)
    out = run_round(inp, w)
    check_status(w, DEV)
    o = {k: v.cpu().numpy() for k, v in out.as_dict().items()}
    st = check_draft(host(inp), o["x"], o["p"], o["lse"], w.seed, 0, False)
    assert st["checked"] > 0
