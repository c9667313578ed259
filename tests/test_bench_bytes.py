"""The bench's algorithmic byte counts and launch counts (CPU only): they follow
the per-unit figures stated for the roofline, term by term, and agree with the
committed profile of the draft kernel."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from speculative_decoding_02_gb300 import workloads as wl  # noqa: E402

# round totals with ell = gamma, every position accepted (gamma verified rows
# and the bonus row of each request) and no residual, in MB, as tabulated by
# hand from U + T rows + W2 + h (+ the small terms)
ROUND_MB = {"qwen3_4b": 722.5, "batch128": 2656.4, "large_vocab": 1279.3, "serving512": 3000.9}


@pytest.mark.parametrize("name", sorted(ROUND_MB))
def test_round_bytes_match_the_tabulated_totals(name):
    w = wl.WORKLOADS[name]
    assert bench.round_bytes(w, w.B * (w.gamma + 1), 0) / 1e6 == pytest.approx(ROUND_MB[name], abs=0.1)


def test_round_bytes_terms():
    w = wl.WORKLOADS["batch128"]
    base = bench.round_bytes(w, 1000, 0)
    assert bench.round_bytes(w, 1001, 0) - base == 4 * w.V        # one more T row
    assert bench.round_bytes(w, 1000, 1) - base == 8 * w.V        # a rejection re-reads a U and a T row


def test_target_rows_per_form():
    # 3 requests, gamma 4, every l_r = 4: n = (1, 4, 0) accepted, so request 1
    # accepted everything (its bonus row is read) and 0 and 2 rejected
    B, G, ell_sum, n_acc, n_full = 3, 4, 12, 5, 1
    # along the accept chains: rows 0..n_r of each request (2 + 5 + 1)
    assert bench.t_rows("chain", B, G, ell_sum, n_acc, n_full) == 8
    # the draft took the rows the accept chains reach: the same rows
    assert bench.t_rows("lazy", B, G, ell_sum, n_acc, n_full) == 8
    # the draft took every row j < gamma; plus the bonus row
    assert bench.t_rows("early", B, G, ell_sum, n_acc, n_full) == 13
    # verification's pass over every row j < l_r; plus the bonus row
    assert bench.t_rows("all", B, G, ell_sum, n_acc, n_full) == 13
    # a truncating schedule: l = (2, 1, 0), n = (1, 1, 0): the chain reads
    # rows 0-1, 0-1 (bonus row 1) and 0 (bonus row 0); the pass over j < l_r
    # reads 3 rows and the two bonus rows; the early draft all 12 and the bonus rows
    assert bench.t_rows("chain", 3, 4, 3, 2, 2) == 5
    assert bench.t_rows("all", 3, 4, 3, 2, 2) == 5
    assert bench.t_rows("early", 3, 4, 3, 2, 2) == 14


def test_draft_bytes_match_the_profile():
    w = wl.WORKLOADS["batch128"]
    d = bench.draft_bytes_per_launch(w)
    # U once (1244.7 MB), W2 once (77.8 MB), the W1 gathers and x/p/lse
    assert d == 4 * 128 * 16 * 151936 + 2 * 256 * 151936 + 2 * 128 * 16 * 256 + 12 * 128 * 16
    # with the target rows j < gamma taken along: those rows once more (1244.7 MB)
    fd = bench.fused_draft_bytes_per_launch(w)
    assert fd - d == 4 * 128 * 16 * 151936
    # the round's first stage adds the hidden states h (bf16, 10.5 MB), the
    # head's w, the confidences and the verified lengths
    sd = bench.stage_bytes_per_launch(w, early=True)
    assert sd - fd == 2 * 128 * 16 * 2560 + 4 * (2560 + 256) + 4 * 128 * 16 + 4 * 128
    assert bench.stage_bytes_per_launch(w, early=False) == sd - 4 * 128 * 16 * 151936
    # the rows the accept chains reach, taken along instead: those rows once
    assert bench.stage_bytes_per_launch(w, rows=517) - bench.stage_bytes_per_launch(w, early=False) == 517 * 4 * w.V
    recs = bench.profile_records(bench.DRAFT_PROFILE)
    assert {(r["early_target_stats"], bool(r.get("chain_target_stats"))) for r in recs} == \
        {(True, False), (False, False), (True, True)}
    for rec in recs:
        assert rec["workload"] == "batch128"
        if rec.get("chain_target_stats"):
            alg = bench.stage_bytes_per_launch(w, rows=rec["chain_rows"])
        else:
            alg = bench.stage_bytes_per_launch(w, rec["early_target_stats"])
        assert int(rec["algorithmic_bytes_per_launch"]) == alg
        # the profile's DRAM traffic is within a few per cent of the algorithmic
        # bytes (the chains' draft also reads a few rows ahead of their tests)
        assert 1.0 <= int(rec["dram_bytes_per_launch"]) / alg < 1.05


def test_kernels_per_round():
    # tensor-core path: one persistent launch drafts, computes the confidences
    # and runs the schedule; verification is the accept tests (verify_chain,
    # or verify_decide after the draft's statistics, or after prep and row
    # statistics), bonus race and residual (their last CTAs write the
    # tokens).  CUDA-core path: a step and a finalize per position, the
    # confidence and schedule kernels, and a residual finalize as well
    b = wl.WORKLOADS["batch128"]
    assert bench.kernels_per_round(b) == 4
    assert bench.kernels_per_round(b, "early") == 4
    assert bench.kernels_per_round(b, "lazy") == 4
    assert bench.kernels_per_round(b, "all") == 6
    t = wl.WORKLOADS["tiny"]
    assert bench.kernels_per_round(t) == 2 * t.gamma + 6
    assert bench.kernels_per_round(t, "all") == 2 * t.gamma + 8
