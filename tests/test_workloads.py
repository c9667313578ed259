"""The synthetic input recipe (on the CPU): shapes, dtypes and the stated
distributions of the seeded workloads, at reduced sizes with each workload's
own parameters, and the determinism of the seeds."""
import dataclasses

import numpy as np
import pytest
import torch

from speculative_decoding_02_gb300 import workloads as wl


def _small(name, V=4096, gamma=None):
    w = wl.WORKLOADS[name]
    return dataclasses.replace(w, B=min(w.B, 16), V=V, gamma=gamma or min(w.gamma, 4), H=min(w.H, 256),
                               sps_len=None if w.sps_len is None else 16 * ((gamma or min(w.gamma, 4)) + 1) + 1)


@pytest.mark.parametrize("name", ["qwen3_4b", "batch128", "large_vocab", "serving512"])
def test_shapes_dtypes_and_layout(name):
    w = _small(name)
    d = wl.make_inputs(w, 0, "cpu")
    B, G, V = w.B, w.gamma, w.V
    assert d["U"].shape == (B, G, V) and d["U"].dtype == torch.float32
    assert d["T"].shape == (B, G + 1, V) and d["T"].dtype == torch.float32
    assert d["W1"].shape == (V, w.r) and d["W2"].shape == (V, w.r) and d["W1"].dtype == w.wdtype
    assert d["h"].shape == (B, G, w.H) and d["h"].dtype == w.wdtype
    assert d["w"].shape == (w.H + w.r,) and d["anchor"].dtype == torch.int32
    assert int(d["anchor"].min()) >= 0 and int(d["anchor"].max()) < V


def test_stated_distributions():
    # batch128's recipe: U ~ N(0, 3^2) with +8 on one token per row; T = U +
    # N(0, sigma_r^2), sigma_r from {0.3, 1, 2}; weights N(0, 0.02^2); h N(0, 1);
    # w N(0, 0.1^2)
    w = dataclasses.replace(_small("batch128", V=32768), B=32)
    d = wl.make_inputs(w, 0, "cpu")
    U = d["U"].double()
    top = U.max(dim=2).values
    assert float(top.min()) > 8.0            # the +8 token dominates every row
    body = U.clone()
    body[U > 8.0 + 6.0] = float("nan")       # leave the planted tokens out
    assert float(torch.nanmean(body)) == pytest.approx(0.0, abs=0.01)
    assert float(np.nanstd(body.numpy())) == pytest.approx(w.u_sigma, rel=0.01)
    noise = d["T"][:, : w.gamma].double() - U
    sig = d["target_sigma"].double()
    assert set(np.round(sig.numpy(), 6)) <= {0.3, 1.0, 2.0}
    per_req = noise.std(dim=(1, 2))
    assert torch.allclose(per_req, sig, rtol=0.02)
    assert float(d["W1"].float().std()) == pytest.approx(w.weight_sigma, rel=0.02)
    assert float(d["h"].float().std()) == pytest.approx(1.0, rel=0.02)
    assert float(d["w"].std()) == pytest.approx(w.w_sigma, rel=0.1)


def test_uniform_target_sigma_and_sps_tables():
    w = _small("serving512")
    d = wl.make_inputs(w, 0, "cpu")
    sig = d["target_sigma"].numpy()
    assert np.all((sig >= 0.3) & (sig <= 2.0))
    b = np.arange(w.sps_len, dtype=np.float64)
    assert np.allclose(d["sps"].numpy(), b / (1.0 + b / w.sps_b0), rtol=1e-6)
    steps = dataclasses.replace(w, sps_kind="steps")
    assert np.allclose(wl.sps_table(steps).numpy(), 1.0 / (1.0 + b / w.sps_b0), rtol=1e-6)
    assert wl.sps_table(dataclasses.replace(w, sps_b0=None)) is None


def test_seeds_are_deterministic_and_rounds_differ():
    w = _small("qwen3_4b")
    a = wl.make_round_inputs(w, 3, "cpu")
    b = wl.make_round_inputs(w, 3, "cpu")
    c = wl.make_round_inputs(w, 4, "cpu")
    assert torch.equal(a["U"], b["U"]) and torch.equal(a["T"], b["T"])
    assert not torch.equal(a["U"], c["U"])
    assert torch.equal(wl.make_weights(w, "cpu")["W2"], wl.make_weights(w, "cpu")["W2"])
