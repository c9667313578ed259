"""A whole round is stream-ordered with no host synchronisation, so it can be
captured into a CUDA graph: the captured round, replayed, gives exactly the
outputs of the same round run eagerly (same seed and round: the random
numbers are counter-based, and every reduction in the path has a fixed
order or is a maximum)."""
import pytest
import torch

import speculative_decoding_02_gb300 as ds
from speculative_decoding_02_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decoding_02_gb300 import build
    build.build()
    ds.library()


def _round(inp, w, rnd, out, ws):
    return ds.round(inp["U"], inp["T"], inp["W1"], inp["W2"], inp["h"], inp["w"], inp["anchor"], seed=w.seed,
                    rnd=rnd, sps=inp["sps"], mode=w.mode, out=out, ws=ws)


@pytest.mark.parametrize("wdtype,r", [(torch.bfloat16, 256), (torch.float32, 64)])
def test_round_replayed_from_a_graph_matches_eager(wdtype, r):
    # bf16 rank 256 runs the persistent tensor-core draft (a cooperative
    # launch) and the tensor-core residual; fp32 the CUDA-core kernels
    w = wl.custom(B=24, gamma=4, V=8192, r=r, H=64, wdtype=wdtype, u_sigma=3.0, seed=13, sps_b0=48.0,
                  sps_kind="steps")
    inp = wl.make_inputs(w, 0, DEV)
    eager = _round(inp, w, 3, ds.RoundOutputs(w.B, w.gamma, DEV), ds.workspace(w.B, w.gamma, w.V, DEV))
    torch.cuda.synchronize()

    out = ds.RoundOutputs(w.B, w.gamma, DEV)
    ws = ds.workspace(w.B, w.gamma, w.V, DEV)
    side = torch.cuda.Stream(DEV)
    side.wait_stream(torch.cuda.current_stream(DEV))
    with torch.cuda.stream(side):
        _round(inp, w, 3, out, ws)   # first calls (tensor maps, attributes) outside the capture
    torch.cuda.current_stream(DEV).wait_stream(side)
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _round(inp, w, 3, out, ws)
    for t in out.as_dict().values():
        t.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert ds.read_status(ws) == ds.OK
    e, g = eager.as_dict(), out.as_dict()
    for name in e:
        assert torch.equal(e[name], g[name]), f"{name} differs between the replayed graph and the eager round"
    # a second replay of the same graph gives the same outputs again
    graph.replay()
    torch.cuda.synchronize()
    for name in e:
        assert torch.equal(e[name], out.as_dict()[name]), name
