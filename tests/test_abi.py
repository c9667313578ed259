"""The C-ABI library loads without a GPU, exports every symbol its header
declares, and rejects bad arguments on the host before touching the device."""
import ctypes
import os
import re

import pytest

import speculative_decoding_02_gb300 as ds

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_02_gb300 import build

    build.build()
    return ds.library()


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names |= set(re.findall(r"\b(dspark_[a-z_0-9]+)\s*\(", txt))
    return names


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert {"dspark_markov_draft", "dspark_confidence", "dspark_schedule", "dspark_verify",
            "dspark_round", "dspark_workspace_size", "dspark_read_status", "dspark_strerror"} <= names
    for n in sorted(names):
        assert hasattr(lib, n), f"{n} declared but not exported"


def _prototypes():
    """name -> number of parameters, from every prototype in include/*.h."""
    protos = {}
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            for name, params in re.findall(r"\b(dspark_[a-z_0-9]+)\s*\(([^)]*)\)\s*;", txt, flags=re.S):
                params = params.strip()
                protos[name] = 0 if params in ("", "void") else params.count(",") + 1
    return protos


def test_binding_argument_counts_match_the_header(lib):
    # ctypes cannot see the C signatures: a parameter added on one side only
    # would shift every later argument, so the counts are compared here
    protos = _prototypes()
    assert set(protos) == _declared()
    bound = [n for n in protos if getattr(lib, n).argtypes is not None]
    assert {"dspark_markov_draft", "dspark_verify", "dspark_round", "dspark_sts_fit"} <= set(bound)
    for n in bound:
        assert len(getattr(lib, n).argtypes) == protos[n], n


def test_strerror_and_workspace_size(lib):
    for code in range(7):
        assert ds._strerror(code)
    assert ds._strerror(99) == "unknown status"
    assert lib.dspark_workspace_size(0, 4, 1024) == 0
    a = lib.dspark_workspace_size(2, 4, 1024)
    b = lib.dspark_workspace_size(128, 16, 151936)
    assert a > 0 and b > a and b % 256 == 0


def _fake(addr=0x10000):
    return ctypes.c_void_p(addr)


def test_host_side_argument_errors(lib):
    p = _fake()
    ws = _fake(0x100000)
    big = 1 << 30
    # null pointers
    assert lib.dspark_markov_draft(None, p, p, 1, p, 2, 4, 1024, 16, 0, 0, p, p, p, ws, big, None) == ds.ERR_INVALID
    # unsupported sizes: B > 65535, gamma > 32, V % 8, r % 16, r > 256
    assert lib.dspark_markov_draft(p, p, p, 1, p, 65536, 4, 1024, 16, 0, 0, p, p, p, ws, big, None) == ds.ERR_UNSUPPORTED
    assert lib.dspark_markov_draft(p, p, p, 1, p, 2, 33, 1024, 16, 0, 0, p, p, p, ws, big, None) == ds.ERR_UNSUPPORTED
    assert lib.dspark_markov_draft(p, p, p, 1, p, 2, 4, 1020, 16, 0, 0, p, p, p, ws, big, None) == ds.ERR_UNSUPPORTED
    assert lib.dspark_markov_draft(p, p, p, 1, p, 2, 4, 1024, 24, 0, 0, p, p, p, ws, big, None) == ds.ERR_UNSUPPORTED
    assert lib.dspark_markov_draft(p, p, p, 1, p, 2, 4, 1024, 512, 0, 0, p, p, p, ws, big, None) == ds.ERR_UNSUPPORTED
    # bad dtype, workspace too small / misaligned, round out of range
    assert lib.dspark_markov_draft(p, p, p, 7, p, 2, 4, 1024, 16, 0, 0, p, p, p, ws, big, None) == ds.ERR_INVALID
    assert lib.dspark_markov_draft(p, p, p, 1, p, 2, 4, 1024, 16, 0, 0, p, p, p, ws, 64, None) == ds.ERR_WORKSPACE
    assert lib.dspark_markov_draft(p, p, p, 1, p, 2, 4, 1024, 16, 0, 0, p, p, p, _fake(0x100010), big,
                                   None) == ds.ERR_WORKSPACE
    assert lib.dspark_markov_draft(p, p, p, 1, p, 2, 4, 1024, 16, 0, 1 << 29, p, p, p, ws, big,
                                   None) == ds.ERR_INVALID
    # scheduler: SPS table too short, B*gamma above 8192, bad mode, top-K without history
    assert lib.dspark_schedule(p, 2, 4, p, 10, 1, 0, None, p, p, p, ws, big, None) == ds.ERR_INVALID
    assert lib.dspark_schedule(p, 512, 32, p, 99999, 1, 0, None, p, p, p, ws, big, None) == ds.ERR_UNSUPPORTED
    assert lib.dspark_schedule(p, 2, 4, p, 11, 5, 0, None, p, p, p, ws, big, None) == ds.ERR_INVALID
    assert lib.dspark_schedule(p, 2, 4, p, 11, 2, 0, None, p, p, p, ws, big, None) == ds.ERR_INVALID
    # verify: null target logits
    assert lib.dspark_verify(None, p, p, p, 1, p, p, p, p, p, 2, 4, 1024, 16, 0, 0, p, p, ws, big,
                             None) == ds.ERR_INVALID
    # confidence: bad dtype
    assert lib.dspark_confidence(p, 3, p, 1, p, None, p, p, 2, 4, 64, 16, 1024, p, None) == ds.ERR_INVALID
    # confidence: more requests than the grid arithmetic allows, gamma past 32
    assert lib.dspark_confidence(p, 1, p, 1, p, None, p, p, 65536, 32, 64, 16, 1024, p, None) == ds.ERR_UNSUPPORTED
    assert lib.dspark_confidence(p, 1, p, 1, p, None, p, p, 2, 33, 64, 16, 1024, p, None) == ds.ERR_UNSUPPORTED
    # bounded-wait self-test: unknown mode, missing / small / misaligned workspace
    assert lib.dspark_selftest_wait_timeout(2, ws, big, None) == ds.ERR_INVALID
    assert lib.dspark_selftest_wait_timeout(0, None, big, None) == ds.ERR_WORKSPACE
    assert lib.dspark_selftest_wait_timeout(1, ws, 128, None) == ds.ERR_WORKSPACE
    assert lib.dspark_selftest_wait_timeout(0, _fake(0x100010), big, None) == ds.ERR_WORKSPACE


def test_noalloc_argument_errors(lib):
    f = lib.dspark_markov_draft_noalloc
    vp, i32, u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64
    f.argtypes = [vp, vp, vp, i32, vp, i32, i32, i32, i32, u64, u64, vp, vp, vp, vp]
    f.restype = i32
    p = _fake(0x100000)
    assert f(None, p, p, 1, p, 2, 4, 1024, 16, 0, 0, p, p, p, None) == ds.ERR_INVALID
    assert f(p, p, p, 1, p, 2, 33, 1024, 16, 0, 0, p, p, p, None) == ds.ERR_UNSUPPORTED
    assert f(p, p, p, 1, p, 65536, 4, 1024, 16, 0, 0, p, p, p, None) == ds.ERR_UNSUPPORTED
    # more elements than the 2^40 the kernels' offsets are sized for
    assert f(p, p, p, 1, p, 1000, 32, 1 << 30, 16, 0, 0, p, p, p, None) == ds.ERR_UNSUPPORTED
    # scratch larger than the library's fixed array
    assert f(p, p, p, 1, p, 4096, 32, 1024, 16, 0, 0, p, p, p, None) == ds.ERR_WORKSPACE


def test_noalloc_status_argument_error(lib):
    f = lib.dspark_noalloc_read_status
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    assert f(None, None) == ds.ERR_INVALID


def test_product_path_never_loads_the_oracle():
    # the package (binding, kernels, library build) imports, links and runs
    # nothing under oracle/: a reference to it may only appear in prose
    pkg = os.path.join(ROOT, "speculative_decoding_02_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                txt = open(os.path.join(dirpath, fn)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", txt, flags=re.M), fn
                assert "liboracle" not in txt and "dspark_oracle" not in txt, fn
                assert not re.search(r"#include\s*[<\"][^>\"]*oracle", txt), fn


def test_missing_library_raises(monkeypatch):
    # no CPU fallback: without the built library every call fails loudly
    monkeypatch.setattr(ds, "_lib", None)
    monkeypatch.setattr(ds, "LIB_PATH", os.path.join(ROOT, "no_such_dir", "libdspark.so"))
    with pytest.raises(ds.DSparkError):
        ds.library()
    with pytest.raises(ds.DSparkError):
        ds.workspace_size(2, 4, 1024)


def test_binding_requires_cuda_tensors():
    import torch
    U = torch.zeros(2, 4, 1024)
    with pytest.raises(ValueError):
        ds.markov_draft(U, U, U, torch.zeros(2, dtype=torch.int32), 0)


def test_binding_shape_checks():
    # the kernels index every tensor from the sizes alone: a W1 with fewer rows
    # than the vocabulary, or per-request tensors of the wrong length, must be
    # refused before anything reaches the device
    import torch
    ds._sized(torch.zeros(8, 16), "W1", (8, 16))
    ds._sized(None, "sts_T", (4,))
    for t, shape in [(torch.zeros(7, 16), (8, 16)), (torch.zeros(8, 16), (16, 8)), (torch.zeros(2, 1), (2,)),
                     (torch.zeros(3), (2,))]:
        with pytest.raises(ValueError):
            ds._sized(t, "t", shape)
    out = ds.RoundOutputs(2, 3, "cpu")
    with pytest.raises(ValueError):
        out.check(2, 3, torch.device("cpu"))   # CPU buffers are refused first


def test_gated_draft_argument_errors(lib):
    p = _fake()
    ws = _fake(0x100000)
    big = 1 << 30
    # missing or misaligned gates; fp32 weights (tensor-core path only)
    assert lib.dspark_gated_markov_draft(p, None, p, p, 1, None, p, p, 2, 4, 1024, 256, 0, 0, None, p, p, p, ws,
                                         big, None) == ds.ERR_INVALID
    assert lib.dspark_gated_markov_draft(p, None, p, p, 1, _fake(0x10004), p, p, 2, 4, 1024, 256, 0, 0, None, p, p,
                                         p, ws, big, None) == ds.ERR_INVALID
    assert lib.dspark_gated_markov_draft(p, None, p, p, 0, p, p, p, 2, 4, 1024, 256, 0, 0, None, p, p, p, ws, big,
                                         None) == ds.ERR_UNSUPPORTED
    assert lib.dspark_gated_markov_draft(p, None, p, p, 1, p, p, p, 2, 4, 1024, 64, 0, 0, None, p, p, p, ws, big,
                                         None) == ds.ERR_UNSUPPORTED
    # verification of a gated draft on the CUDA-core path
    assert lib.dspark_verify_ex(p, p, p, p, 0, p, p, p, p, p, 2, 4, 1024, 64, 0, 0, None, ds.GATED_STATES, p, p,
                                ws, big, None) == ds.ERR_UNSUPPORTED


def test_row_statistics_flags(lib):
    p = _fake()
    ws = _fake(0x100000)
    big = 1 << 30
    # statistics taken by the draft (of every row or along the accept
    # chains) and a full row pass by verification exclude one another, in
    # verify_ex and in round_ex; an unknown bit is refused; verify_ex takes
    # the draft's chain statistics as early ones, not by the chain flag
    both = ds.EARLY_TARGET_STATS | ds.ALL_ROW_STATS
    for flags in (both, 128, ds.CHAIN_TARGET_STATS):
        assert lib.dspark_verify_ex(p, p, p, p, 1, p, p, p, p, p, 2, 4, 1024, 256, 0, 0, None, flags, p, p, ws, big,
                                    None) == ds.ERR_INVALID
    for flags in (both, 128, ds.CHAIN_TARGET_STATS | ds.EARLY_TARGET_STATS,
                  ds.CHAIN_TARGET_STATS | ds.ALL_ROW_STATS):
        assert lib.dspark_round_ex(p, p, p, p, 1, p, 1, p, None, p, 2, 4, 1024, 256, 64, p, 11, 1, None, 0, 0, None,
                                   flags, p, p, p, p, p, p, p, p, p, ws, big, None) == ds.ERR_INVALID
    # draft_schedule_ex: the chain flag needs T_early; other bits are refused
    for t_early, flags in ((None, ds.CHAIN_TARGET_STATS), (p, ds.EARLY_TARGET_STATS), (p, 128)):
        assert lib.dspark_draft_schedule_ex(p, t_early, p, p, 1, p, 1, p, None, p, 2, 4, 1024, 256, 64, p, 11, 1,
                                            None, 0, 0, None, flags, p, p, p, p, p, p, p, ws, big,
                                            None) == ds.ERR_INVALID


def test_acceptance_label_and_sts_argument_errors(lib):
    p = _fake()
    ws = _fake(0x100000)
    big = 1 << 30
    # acceptance labels: a null output, fp32 weights (tensor-core path only),
    # a workspace that is too small
    assert lib.dspark_acceptance_label(p, p, p, p, 1, p, p, p, p, 2, 4, 1024, 256, None, ws, big,
                                       None) == ds.ERR_INVALID
    assert lib.dspark_acceptance_label(p, p, p, p, 0, p, p, p, p, 2, 4, 1024, 256, p, ws, big,
                                       None) == ds.ERR_UNSUPPORTED
    assert lib.dspark_acceptance_label(p, p, p, p, 1, p, p, p, p, 2, 4, 1024, 256, p, ws, 16,
                                       None) == ds.ERR_WORKSPACE
    # the statistics-source flags: not both, no other bits
    for flags in (ds.EARLY_TARGET_STATS | ds.TARGET_STATS_FROM_VERIFY, 8, ds.ADVANCE_ROUND):
        assert lib.dspark_acceptance_label_ex(p, p, p, p, 1, p, p, p, p, 2, 4, 1024, 256, flags, p, ws, big,
                                              None) == ds.ERR_INVALID
    # STS: workspace size grows with the samples and the grid; bad arguments
    assert lib.dspark_sts_workspace_size(0, 4, 8) == 0
    assert lib.dspark_sts_workspace_size(10000, 4, 49) > lib.dspark_sts_workspace_size(100, 4, 49) > 0
    assert lib.dspark_sts_fit(None, p, p, 100, 4, p, 49, p, p, ws, big, None) == ds.ERR_INVALID
    assert lib.dspark_sts_fit(p, p, p, 0, 4, p, 49, p, p, ws, big, None) == ds.ERR_INVALID
    assert lib.dspark_sts_fit(p, p, p, 100, 33, p, 49, p, p, ws, big, None) == ds.ERR_UNSUPPORTED
    assert lib.dspark_sts_fit(p, p, p, 100, 4, p, 257, p, p, ws, big, None) == ds.ERR_UNSUPPORTED
    assert lib.dspark_sts_fit(p, p, p, 100, 4, p, 49, p, p, ws, 8, None) == ds.ERR_WORKSPACE
    assert lib.dspark_sts_fit(p, p, p, 100, 4, p, 49, p, p, _fake(0x100010), big, None) == ds.ERR_WORKSPACE
