"""A whole round is stream-ordered with no host synchronisation, so it can be
captured into a CUDA graph: the captured round, replayed, gives exactly the
outputs of the same round run eagerly (same seed and round: the random
numbers are counter-based, and every reduction in the path has a fixed
order or is a maximum).  With the round index in device memory, advanced by
the round's last kernel, one captured graph serves consecutive rounds."""
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


def _own_workspace(w):
    # a workspace of its own (the binding's cached one would be shared with
    # the eager rounds)
    n = ds.workspace_size(w.B, w.gamma, w.V)
    buf = torch.zeros(n + 256, dtype=torch.uint8, device=DEV)
    off = (-buf.data_ptr()) % 256
    return buf[off:off + n]


@pytest.mark.parametrize("early", [False, True])
def test_one_graph_serves_consecutive_rounds(early):
    # The round index lives in device memory and the round's last kernel adds
    # 1 to it, so ten replays of ONE captured graph are rounds 0..9: each must
    # equal the eager round with that host index bit for bit, top-K history
    # included (rounds 2.. admit the greedy count of two rounds earlier).
    w = wl.custom(B=24, gamma=4, V=8192, r=256, H=64, wdtype=torch.bfloat16, mode=wl.MODE_TOPK, u_sigma=3.0,
                  seed=17, sps_b0=48.0, sps_kind="steps")
    inp = wl.make_inputs(w, 0, DEV)
    kh_e = torch.zeros(2, dtype=torch.int32, device=DEV)
    ws_e = _own_workspace(w)
    eager = []
    for i in range(10):
        out = ds.round(inp["U"], inp["T"], inp["W1"], inp["W2"], inp["h"], inp["w"], inp["anchor"], seed=w.seed,
                       rnd=i, sps=inp["sps"], mode=w.mode, khist=kh_e, ws=ws_e, early_stats=early)
        eager.append({k: v.clone() for k, v in out.as_dict().items()})
    torch.cuda.synchronize()
    assert ds.read_status(ws_e) == ds.OK
    assert len({int(e["nstar"][0]) for e in eager}) >= 1

    round_dev = torch.zeros(1, dtype=torch.int64, device=DEV)
    kh_g = torch.zeros(2, dtype=torch.int32, device=DEV)
    ws_g = _own_workspace(w)
    out = ds.RoundOutputs(w.B, w.gamma, DEV)

    def rnd_call():
        ds.round(inp["U"], inp["T"], inp["W1"], inp["W2"], inp["h"], inp["w"], inp["anchor"], seed=w.seed, rnd=0,
                 sps=inp["sps"], mode=w.mode, khist=kh_g, out=out, ws=ws_g, early_stats=early, round_dev=round_dev,
                 advance_round=True)

    side = torch.cuda.Stream(DEV)
    side.wait_stream(torch.cuda.current_stream(DEV))
    with torch.cuda.stream(side):
        rnd_call()   # first calls (tensor maps, attributes) outside the capture
    torch.cuda.current_stream(DEV).wait_stream(side)
    torch.cuda.synchronize()
    assert int(round_dev[0]) == 1
    round_dev.zero_()
    kh_g.zero_()
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        rnd_call()
    for i in range(10):
        for t in out.as_dict().values():
            t.zero_()
        graph.replay()
        torch.cuda.synchronize()
        g = out.as_dict()
        for name in eager[i]:
            assert torch.equal(eager[i][name], g[name]), f"replay {i}: {name} differs from eager round {i}"
    assert int(round_dev[0]) == 10
    assert torch.equal(kh_g, kh_e)
    assert ds.read_status(ws_g) == ds.OK
