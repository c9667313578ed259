"""Shared helpers of the GPU parity tests: run the CUDA path, run the oracle on
the same seeded inputs (teacher-forced on the GPU's discrete upstream decisions)
and compare under the parity rules:

* token ids, accepted counts and corrected / bonus tokens bit-exact wherever
  the deciding margin exceeds 1e-4 (the top-two Gumbel-perturbed logit gap of
  an argmax, |u - p_t/p_d| of an accept test);
* probabilities and confidences within 1e-5 relative with fp32 weights; with
  bf16 weights the fused logits within 2e-2 absolute: lse_k and the drafted
  token's own logit l_k(x_k) = log p_k(x_k) + lse_k;
* verify lengths bit-exact unless two survival products near the cut lie
  within 1e-5 relative or Theta at the stop is within 1e-6 relative of the
  best; then the achieved Theta within 1e-5 relative.
"""
import numpy as np
import torch

import oracle
import speculative_decoding_02_gb300 as ds
from speculative_decoding_02_gb300 import workloads as wl

MARGIN = 1e-4


def host(inp):
    return {k: wl.to_numpy(v) for k, v in inp.items() if isinstance(v, torch.Tensor)}


def is_bf16(inp):
    return inp["W1"].dtype == torch.bfloat16


def ranges(reqs, B):
    """Contiguous [b0, b1) runs covering the requests (all when None), so that
    the oracle handles each run in one call (in parallel over its requests)."""
    reqs = sorted(set(range(B) if reqs is None else reqs))
    out = []
    for b in reqs:
        if out and out[-1][1] == b:
            out[-1][1] = b + 1
        else:
            out.append([b, b + 1])
    return [tuple(r) for r in out]


def check_draft(h, out_x, out_p, out_lse, seed, rnd, bf16, reqs=None):
    """Teacher-forced oracle draft on the requests `reqs` (all when None)."""
    B = h["U"].shape[0]
    stats = dict(checked=0, low_margin=0)
    for b0, b1 in ranges(reqs, B):
        d = oracle.draft(h["U"], h["W1"], h["W2"], h["anchor"], seed, rnd, x_force=out_x, b0=b0, b1=b1)
        for b in range(b0, b1):
            sure = d["margin"][b] > MARGIN
            stats["checked"] += int(sure.sum())
            stats["low_margin"] += int((~sure).sum())
            assert np.array_equal(d["x"][b][sure], out_x[b][sure]), \
                f"request {b}: draft tokens {out_x[b].tolist()} vs oracle {d['x'][b].tolist()}"
            if bf16:
                # lse_k and the drafted token's fused logit l_k(x_k) = log p + lse
                np.testing.assert_allclose(out_lse[b], d["lse"][b], rtol=0, atol=2e-2)
                np.testing.assert_allclose(np.log(out_p[b]) + out_lse[b], np.log(d["p"][b]) + d["lse"][b], rtol=0,
                                           atol=2e-2)
            else:
                np.testing.assert_allclose(out_lse[b], d["lse"][b], rtol=1e-5)
                np.testing.assert_allclose(out_p[b], d["p"][b], rtol=1e-5)
    return stats


def check_confidence(h, x, c_gpu, sts_T=None):
    c = oracle.confidence(h["h"], h["W1"], h["w"], h["anchor"], x, sts_T=sts_T)
    np.testing.assert_allclose(c_gpu, c, rtol=1e-5, atol=1e-6)
    return c


def check_schedule(c_gpu, sps, mode, ell_gpu, nstar_gpu, theta_gpu, K=-1):
    """Oracle scheduler on the GPU's own confidences (teacher forcing)."""
    o = oracle.schedule(c_gpu.astype(np.float64), sps, mode, K=K)
    if np.array_equal(o["ell"], ell_gpu):
        if mode != oracle.MODE_FIXED:
            assert abs(theta_gpu - o["theta"]) <= 1e-9 * abs(o["theta"]) + 1e-12
        assert nstar_gpu == o["nstar"]
        return o
    # allowed only at near-ties: check the achieved Theta instead
    a = np.sort(np.cumprod(c_gpu.astype(np.float64), axis=1).ravel())[::-1]
    n = o["nstar"]
    near = np.any(np.abs(np.diff(a[max(n - 2, 0):n + 2])) <= 1e-5 * np.abs(a[max(n - 2, 0):n + 1]))
    assert near, f"schedule differs without a near-tie: {ell_gpu.tolist()} vs {o['ell'].tolist()}"
    assert abs(theta_gpu - o["theta"]) <= 1e-5 * abs(o["theta"])
    return o


def check_verify(h, x, ell, n_gpu, tok_gpu, seed, rnd, reqs=None):
    """Teacher-forced oracle verification (GPU draft tokens and lengths)."""
    B = h["U"].shape[0]
    stats = dict(checked=0, low_margin=0, residual=0, bonus=0)
    for b0, b1 in ranges(reqs, B):
        v = oracle.verify(h["T"], h["U"], h["W1"], h["W2"], h["anchor"], x, ell, seed, rnd, b0=b0, b1=b1)
        for b in range(b0, b1):
            um = v["umargin"][b]
            evaluated = um[~np.isnan(um)]
            if evaluated.size and evaluated.min() <= MARGIN:
                stats["low_margin"] += 1
                continue
            assert n_gpu[b] == v["n"][b], f"request {b}: accepted {n_gpu[b]} vs oracle {v['n'][b]}"
            stats["checked"] += 1
            stats["residual" if v["flags"][b] & 2 else "bonus"] += 1
            if v["ymargin"][b] > MARGIN:
                assert tok_gpu[b] == v["y"][b], f"request {b}: token {tok_gpu[b]} vs oracle {v['y'][b]}"
    return stats


def run_round(inp, w, rnd=0, mode=None, khist=None, early_stats=False, all_row_stats=False, chain_stats=False,
              T=None, ws=None):
    mode = w.mode if mode is None else mode
    if mode == wl.MODE_TOPK and khist is None:
        khist = torch.zeros(2, dtype=torch.int32, device=inp["U"].device)
    out = ds.round(inp["U"], inp["T"] if T is None else T, inp["W1"], inp["W2"], inp["h"], inp["w"], inp["anchor"],
                   seed=w.seed, rnd=rnd, sps=inp["sps"], mode=mode, khist=khist, early_stats=early_stats,
                   all_row_stats=all_row_stats, chain_stats=chain_stats, ws=ws)
    torch.cuda.synchronize()
    return out


def check_status(w, dev):
    st = ds.read_status(ds.workspace(w.B, w.gamma, w.V, dev))
    assert st == ds.OK, f"device status {st}: {ds._strerror(st)}"
