"""The allocation-free draft entry point (dspark_markov_draft_noalloc).

Some callers cannot allocate device memory when they call the library (an
engine whose pool allocator owns all of HBM, a plugin given no allocator, a
decode loop that must not call cudaMalloc).  This entry point uses a fixed
scratch array inside the library instead of a caller workspace.  The test calls
it through the C ABI, twice in a row, and checks that it returns what the
workspace entry point returns.  It lives in its own file so that pytest collects
it last."""
import ctypes

import pytest
import torch

import speculative_decoding_02_gb300 as ds
from speculative_decoding_02_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def _entry():
    from speculative_decoding_02_gb300 import build
    build.build()
    L = ds.library()
    f = L.dspark_markov_draft_noalloc
    vp, i32, u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64
    f.argtypes = [vp, vp, vp, i32, vp, i32, i32, i32, i32, u64, u64, vp, vp, vp, vp]
    f.restype = i32
    return f


def _call(f, inp, w, rnd, B=None, G=None, V=None):
    B = w.B if B is None else B
    G = w.gamma if G is None else G
    V = w.V if V is None else V
    x = torch.empty((w.B, w.gamma), dtype=torch.int32, device=DEV)
    p = torch.empty((w.B, w.gamma), dtype=torch.float32, device=DEV)
    lse = torch.empty((w.B, w.gamma), dtype=torch.float32, device=DEV)
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())
    dt = ds.BF16 if inp["W1"].dtype == torch.bfloat16 else ds.F32
    st = f(ptr(inp["U"]), ptr(inp["W1"]), ptr(inp["W2"]), dt, ptr(inp["anchor"]), B, G, V, w.r, w.seed, rnd,
           ptr(x), ptr(p), ptr(lse), ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream))
    torch.cuda.synchronize()
    return st, x, p, lse


@pytest.mark.parametrize("name", ["small", "batch128"])
def test_noalloc_draft_matches_workspace_draft(name):
    f = _entry()
    if name == "small":
        w = wl.custom(B=40, gamma=5, V=5000, r=64, H=16, wdtype=torch.bfloat16, seed=3)
    else:
        w = wl.WORKLOADS["batch128"]
    weights = wl.make_weights(w, DEV)
    rin = wl.make_round_inputs(w, 0, DEV)
    inp = dict(U=rin["U"], W1=weights["W1"], W2=weights["W2"], anchor=weights["anchor"])
    del rin
    for rnd in (0, 1):  # two calls in a row share the scratch array
        st, x, p, lse = _call(f, inp, w, rnd)
        assert st == ds.OK, ds._strerror(st)
        rx, rp, rl = ds.markov_draft(inp["U"], inp["W1"], inp["W2"], inp["anchor"], w.seed, rnd)
        torch.cuda.synchronize()
        assert torch.equal(x, rx)
        torch.testing.assert_close(p, rp, rtol=1e-5, atol=0)
        torch.testing.assert_close(lse, rl, rtol=1e-5, atol=0)


def _read_status():
    L = ds.library()
    L.dspark_noalloc_read_status.argtypes = [ctypes.POINTER(ctypes.c_int), ctypes.c_void_p]
    L.dspark_noalloc_read_status.restype = ctypes.c_int
    v = ctypes.c_int(-1)
    assert L.dspark_noalloc_read_status(ctypes.byref(v), ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)) \
        == ds.OK
    return int(v.value)


def test_noalloc_reports_kernel_errors():
    # an anchor outside [0, V) is caught by the kernels and shows in the
    # scratch array's status word; a clean call after it reads OK
    f = _entry()
    L = ds.library()
    L.dspark_noalloc_init.argtypes = []
    L.dspark_noalloc_init.restype = ctypes.c_int
    assert L.dspark_noalloc_init() == ds.OK
    w = wl.custom(B=40, gamma=5, V=5000, r=64, H=16, wdtype=torch.bfloat16, seed=3)
    weights = wl.make_weights(w, DEV)
    rin = wl.make_round_inputs(w, 0, DEV)
    inp = dict(U=rin["U"], W1=weights["W1"], W2=weights["W2"], anchor=weights["anchor"].clone())
    inp["anchor"][7] = w.V + 3
    st, _, _, _ = _call(f, inp, w, 0)
    assert st == ds.OK
    assert _read_status() == ds.ERR_INVALID
    inp["anchor"] = weights["anchor"]
    st, _, _, _ = _call(f, inp, w, 1)
    assert st == ds.OK
    assert _read_status() == ds.OK
