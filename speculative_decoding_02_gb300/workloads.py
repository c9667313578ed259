"""Seeded synthetic workloads for the DSpark per-round hot path.

This module only draws random inputs; it holds none of the method's arithmetic.
It is the one module that the CUDA path's tests/bench and the oracle's checks
share.  No dataset, prompt or trained weight is used: the backbone logits U,
the target logits T, the Markov weights W1/W2, the hidden states h and the
confidence weight w are Gaussian draws shaped like the workloads the DSpark pages
describe (a Qwen3-4B-sized vocabulary and hidden size, a batch-128 engine point,
a large-vocabulary case and a high-concurrency serving round).

Layouts (row-major):
  U      [B, gamma, V]      float32   backbone logits, row k-1 scores position k
  T      [B, gamma+1, V]    float32   target logits, row k-1 scores position k,
                                      row gamma is the bonus row of a full accept
  W1     [V, r]             bf16/f32  Markov embedding of the previous token
  W2     [V, r]             bf16/f32  weight of the bias-free linear r -> V
  h      [B, gamma, H]      bf16/f32  backbone hidden states
  w      [H + r]            float32   confidence-head weight
  anchor [B]                int32     anchor tokens x_0
  sps    [n_sps]            float32   steps-per-second table indexed by batch size
"""
from dataclasses import dataclass, field
from typing import Optional

import torch

MODE_FIXED, MODE_GREEDY, MODE_TOPK = 0, 1, 2


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    gamma: int
    V: int
    r: int
    H: int
    wdtype: torch.dtype          # W1 / W2 / h storage type
    u_sigma: float               # U ~ N(0, u_sigma^2)
    peak: float                  # + peak on one uniformly chosen token per row
    t_sigma: tuple               # target noise: fixed value, set of values, or ("uniform", lo, hi)
    mode: int                    # schedule mode
    sps_b0: Optional[float]      # SPS(B) = B / (1 + B / sps_b0)
    sps_len: Optional[int]       # table length (covers B = 0 .. sps_len-1)
    seed: int
    rounds: int = 1
    w_sigma: float = 0.1
    weight_sigma: float = 0.02
    sps_kind: str = "saturating"  # "saturating": B/(1+B/b0); "steps": 1/(1+B/b0)
    extra: dict = field(default_factory=dict)


def _sps_len(B, gamma, minimum=0):
    return max(B * (gamma + 1) + 1, minimum)


# The five workloads.  Where the shape description leaves a detail open the
# reading is fixed here: the peaked token is uniform per row; per-request target
# sigma is drawn uniformly from its set; w ~ N(0, 0.1^2) everywhere; the fresh
# bonus row of T is drawn like a U row.
WORKLOADS = {
    "tiny": Workload("tiny", B=2, gamma=4, V=1024, r=16, H=64, wdtype=torch.float32,
                     u_sigma=2.0, peak=0.0, t_sigma=(0.5,), mode=MODE_GREEDY,
                     sps_b0=64.0, sps_len=_sps_len(2, 4), seed=0),
    "qwen3_4b": Workload("qwen3_4b", B=32, gamma=16, V=151936, r=256, H=2560,
                         wdtype=torch.bfloat16, u_sigma=3.0, peak=8.0, t_sigma=(1.0,),
                         mode=MODE_FIXED, sps_b0=None, sps_len=None, seed=1),
    "batch128": Workload("batch128", B=128, gamma=16, V=151936, r=256, H=2560,
                         wdtype=torch.bfloat16, u_sigma=3.0, peak=8.0, t_sigma=(0.3, 1.0, 2.0),
                         mode=MODE_GREEDY, sps_b0=256.0, sps_len=_sps_len(128, 16), seed=2),
    "large_vocab": Workload("large_vocab", B=64, gamma=8, V=262144, r=256, H=3840,
                            wdtype=torch.bfloat16, u_sigma=3.0, peak=0.0, t_sigma=(1.5,),
                            mode=MODE_GREEDY, sps_b0=512.0, sps_len=2049, seed=3),
    "serving512": Workload("serving512", B=512, gamma=5, V=129280, r=256, H=4096,
                           wdtype=torch.bfloat16, u_sigma=3.0, peak=0.0,
                           t_sigma=("uniform", 0.3, 2.0), mode=MODE_TOPK, sps_b0=384.0,
                           sps_len=_sps_len(512, 5, 3073), seed=4, rounds=100),
}


def custom(name="custom", **kw):
    """A workload of any shape (tests use this for small and ragged cases)."""
    base = dict(B=2, gamma=4, V=1024, r=16, H=64, wdtype=torch.float32, u_sigma=2.0, peak=0.0,
                t_sigma=(0.5,), mode=MODE_GREEDY, sps_b0=64.0, sps_len=None, seed=0)
    base.update(kw)
    if base["sps_len"] is None:
        base["sps_len"] = _sps_len(base["B"], base["gamma"])
    return Workload(name, **base)


def sps_table(wl: Workload) -> Optional[torch.Tensor]:
    """The SPS table at B = 0 .. sps_len-1 (float32): B / (1 + B / b0) as the
    workloads state it, or 1 / (1 + B / b0), a steps-per-second curve that falls
    with the batch size (used by tests to make the scheduler truncate)."""
    if wl.sps_b0 is None:
        return None
    b = torch.arange(wl.sps_len, dtype=torch.float64)
    if wl.sps_kind == "steps":
        return (1.0 / (1.0 + b / wl.sps_b0)).to(torch.float32)
    return (b / (1.0 + b / wl.sps_b0)).to(torch.float32)


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, sigma, g, device, dtype=torch.float32):
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.normal_(0.0, sigma, generator=g)
    return t.to(dtype)


def _target_sigmas(wl: Workload, g, device):
    ts = wl.t_sigma
    if len(ts) == 3 and ts[0] == "uniform":
        lo, hi = ts[1], ts[2]
        return lo + (hi - lo) * torch.rand(wl.B, generator=g, device=device)
    vals = torch.tensor([float(v) for v in ts], device=device)
    idx = torch.randint(0, len(ts), (wl.B,), generator=g, device=device)
    return vals[idx]


def make_weights(wl: Workload, device="cpu"):
    """W1, W2 [V, r], w [H + r], anchor [B] for a workload (seeded)."""
    g = _gen(device, 1000003 * wl.seed + 17)
    W1 = _normal((wl.V, wl.r), wl.weight_sigma, g, device, wl.wdtype)
    W2 = _normal((wl.V, wl.r), wl.weight_sigma, g, device, wl.wdtype)
    w = _normal((wl.H + wl.r,), wl.w_sigma, g, device)
    anchor = torch.randint(0, wl.V, (wl.B,), generator=g, device=device, dtype=torch.int32)
    return dict(W1=W1, W2=W2, w=w, anchor=anchor)


def make_gates(wl: Workload, device="cpu"):
    """The gated recurrent head's gates g, c [r] float32 (seeded; both N(0, 1),
    so that the gates sigmoid(g * e + c) spread over (0, 1))."""
    g = _gen(device, 1000003 * wl.seed + 29)
    return dict(gate_g=_normal((wl.r,), 1.0, g, device), gate_c=_normal((wl.r,), 1.0, g, device))


def make_round_inputs(wl: Workload, rnd: int = 0, device="cpu"):
    """U [B,gamma,V], T [B,gamma+1,V], h [B,gamma,H] for round `rnd` (seeded)."""
    g = _gen(device, 1000003 * wl.seed + 7919 * (rnd + 1))
    B, G, V = wl.B, wl.gamma, wl.V
    # G + 1 backbone-like rows; the first G are U, the last seeds the bonus row of T
    U_ext = _normal((B, G + 1, V), wl.u_sigma, g, device)
    if wl.peak:
        idx = torch.randint(0, V, (B, G + 1, 1), generator=g, device=device)
        U_ext.scatter_add_(2, idx, torch.full((B, G + 1, 1), float(wl.peak), device=device))
    sig = _target_sigmas(wl, g, device)
    T = U_ext + _normal((B, G + 1, V), 1.0, g, device) * sig.view(B, 1, 1)
    U = U_ext[:, :G].contiguous()
    del U_ext
    h = _normal((B, G, wl.H), 1.0, g, device, wl.wdtype)
    return dict(U=U, T=T, h=h, target_sigma=sig)


def make_inputs(wl: Workload, rnd: int = 0, device="cpu"):
    d = make_weights(wl, device)
    d.update(make_round_inputs(wl, rnd, device))
    sps = sps_table(wl)
    d["sps"] = None if sps is None else sps.to(device)
    return d


def to_numpy(t: torch.Tensor):
    """Host numpy view of a tensor; bf16 becomes its raw uint16 bit pattern."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16")
    return t.numpy()
