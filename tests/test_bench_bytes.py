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

# round totals with ell = gamma and no residual, in MB, as tabulated by hand
# from U + T rows + W2 + h (+ the small terms)
ROUND_MB = {"qwen3_4b": 722.5, "batch128": 2656.4, "large_vocab": 1279.3, "serving512": 3000.9}


@pytest.mark.parametrize("name", sorted(ROUND_MB))
def test_round_bytes_match_the_tabulated_totals(name):
    w = wl.WORKLOADS[name]
    assert bench.round_bytes(w, w.B * w.gamma, 0) / 1e6 == pytest.approx(ROUND_MB[name], abs=0.1)


def test_round_bytes_terms():
    w = wl.WORKLOADS["batch128"]
    base = bench.round_bytes(w, 1000, 0)
    assert bench.round_bytes(w, 1001, 0) - base == 4 * w.V        # one more verified T row
    assert bench.round_bytes(w, 1000, 1) - base == 8 * w.V        # a rejection re-reads a U and a T row
    # every request reads at least its first T row (bonus or first verified)
    assert bench.round_bytes(w, 0, 0) >= 4 * w.B * w.gamma * w.V + 4 * w.V * w.B


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
    with open(bench.DRAFT_PROFILE) as f:
        rec = json.load(f)
    assert rec["workload"] == "batch128"
    alg = bench.stage_bytes_per_launch(w, rec["early_target_stats"])
    assert int(rec["algorithmic_bytes_per_launch"]) == alg
    # the profile's DRAM traffic is within a few per cent of the algorithmic bytes
    assert 1.0 <= int(rec["dram_bytes_per_launch"]) / alg < 1.05


def test_kernels_per_round():
    # tensor-core path: one persistent launch drafts, computes the confidences
    # and runs the schedule; verification is decide, bonus race and residual
    # (their last CTAs write the tokens), after prep and row statistics
    # unless the draft took the target-row statistics along.  CUDA-core
    # path: a step and a finalize per position, the confidence and schedule
    # kernels, and a residual finalize as well
    assert bench.kernels_per_round(wl.WORKLOADS["batch128"]) == 6
    assert bench.kernels_per_round(wl.WORKLOADS["batch128"], early=True) == 4
    t = wl.WORKLOADS["tiny"]
    assert bench.kernels_per_round(t) == 2 * t.gamma + 8
