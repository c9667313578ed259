"""Python binding of libdspark, the GB300 (sm_103a) DSpark per-round hot path.

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  Tensors must be contiguous CUDA tensors on one device; outputs are
allocated with torch on that device and every call is enqueued on the current
torch stream.  If the compiled library is missing, every call raises
``DSparkError`` -- there is no CPU fallback.

Entry points (same names as the C ABI in include/dspark.h; the optional
arguments of markov_draft, schedule, verify and round map to the C ABI's _ex
forms):
  markov_draft, confidence, schedule, verify, round, read_status,
  acceptance_label, sts_fit
"""
import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libdspark.so")

OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_WORKSPACE, ERR_NONFINITE = range(7)
F32, BF16 = 0, 1
SCHED_FIXED, SCHED_GREEDY, SCHED_TOPK = 0, 1, 2
EARLY_TARGET_STATS, ADVANCE_ROUND, TARGET_STATS_FROM_VERIFY, SCRATCH_FROM_DRAFT, GATED_STATES = 1, 2, 4, 8, 16
ALL_ROW_STATS = 32
CHAIN_TARGET_STATS = 64


class DSparkError(RuntimeError):
    def __init__(self, code, where=""):
        self.code = code
        msg = _strerror(code) if _lib is not None else f"status {code}"
        super().__init__(f"{where}: {msg} (status {code})" if where else msg)


_lib = None


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise DSparkError(ERR_CUDA, f"libdspark is not built ({LIB_PATH} missing); run "
                                    f"`python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, u64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_size_t
    L.dspark_workspace_size.argtypes = [i32, i32, i32]
    L.dspark_workspace_size.restype = sz
    L.dspark_markov_draft.argtypes = [vp, vp, vp, i32, vp, i32, i32, i32, i32, u64, u64, vp, vp, vp, vp, sz, vp]
    L.dspark_markov_draft.restype = i32
    L.dspark_markov_draft_ex.argtypes = [vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, u64, u64, vp, vp, vp, vp, vp,
                                         sz, vp]
    L.dspark_markov_draft_ex.restype = i32
    L.dspark_gated_markov_draft.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp, i32, i32, i32, i32, u64, u64, vp, vp,
                                            vp, vp, vp, sz, vp]
    L.dspark_gated_markov_draft.restype = i32
    L.dspark_confidence.argtypes = [vp, i32, vp, i32, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp]
    L.dspark_confidence.restype = i32
    L.dspark_schedule.argtypes = [vp, i32, i32, vp, i32, i32, u64, vp, vp, vp, vp, vp, sz, vp]
    L.dspark_schedule.restype = i32
    L.dspark_schedule_ex.argtypes = [vp, i32, i32, vp, i32, i32, u64, vp, vp, vp, vp, vp, vp, sz, vp]
    L.dspark_schedule_ex.restype = i32
    L.dspark_verify.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp, vp, vp, i32, i32, i32, i32, u64, u64, vp, vp,
                                vp, sz, vp]
    L.dspark_verify.restype = i32
    L.dspark_verify_ex.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp, vp, vp, i32, i32, i32, i32, u64, u64, vp,
                                   ctypes.c_uint, vp, vp, vp, sz, vp]
    L.dspark_verify_ex.restype = i32
    L.dspark_acceptance_label.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp, vp, i32, i32, i32, i32, vp, vp,
                                          ctypes.c_size_t, vp]
    L.dspark_acceptance_label.restype = i32
    L.dspark_acceptance_label_ex.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp, vp, i32, i32, i32, i32, ctypes.c_uint,
                                             vp, vp, ctypes.c_size_t, vp]
    L.dspark_acceptance_label_ex.restype = i32
    L.dspark_sts_workspace_size.argtypes = [i32, i32, i32]
    L.dspark_sts_workspace_size.restype = sz
    L.dspark_sts_fit.argtypes = [vp, vp, vp, i32, i32, vp, i32, vp, vp, vp, sz, vp]
    L.dspark_sts_fit.restype = i32
    L.dspark_round.argtypes = [vp, vp, vp, vp, i32, vp, i32, vp, vp, vp, i32, i32, i32, i32, i32, vp, i32, i32,
                               vp, u64, u64, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.dspark_round.restype = i32
    L.dspark_round_ex.argtypes = [vp, vp, vp, vp, i32, vp, i32, vp, vp, vp, i32, i32, i32, i32, i32, vp, i32, i32,
                                  vp, u64, u64, vp, ctypes.c_uint, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.dspark_round_ex.restype = i32
    L.dspark_draft_schedule.argtypes = [vp, vp, vp, vp, i32, vp, i32, vp, vp, vp, i32, i32, i32, i32, i32, vp, i32,
                                        i32, vp, u64, u64, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.dspark_draft_schedule.restype = i32
    L.dspark_draft_schedule_ex.argtypes = [vp, vp, vp, vp, i32, vp, i32, vp, vp, vp, i32, i32, i32, i32, i32, vp,
                                           i32, i32, vp, u64, u64, vp, ctypes.c_uint, vp, vp, vp, vp, vp, vp, vp,
                                           vp, sz, vp]
    L.dspark_draft_schedule_ex.restype = i32
    L.dspark_read_status.argtypes = [vp, ctypes.POINTER(i32), vp]
    L.dspark_read_status.restype = i32
    L.dspark_selftest_wait_timeout.argtypes = [i32, vp, sz, vp]
    L.dspark_selftest_wait_timeout.restype = i32
    L.dspark_strerror.argtypes = [i32]
    L.dspark_strerror.restype = ctypes.c_char_p
    _lib = L
    return L


def _strerror(code):
    return _lib.dspark_strerror(int(code)).decode()


def library():
    """The loaded ctypes library (raises DSparkError if it is not built)."""
    return _load()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check(code, where):
    if code != OK:
        raise DSparkError(code, where)


def _dt(t, what):
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"{what} must be float32 or bfloat16, got {t.dtype}")


def _need(t, what, dtype=None, device=None):
    if t is None:
        raise ValueError(f"{what} is required")
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{what} must be {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{what} is on {t.device}, expected {device}")
    return t


def _sized(t, what, shape):
    """Raise unless t has this shape.  The kernels index every tensor from the
    sizes alone, so a tensor smaller than its sizes say would be read or
    written past its end on the device."""
    if t is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{what} must be {list(shape)}, got {list(t.shape)}")
    return t


_ws_cache = {}


def workspace_size(B, gamma, V):
    return int(_load().dspark_workspace_size(B, gamma, V))


def workspace(B, gamma, V, device):
    """A cached, 256-byte aligned device workspace for these sizes."""
    n = workspace_size(B, gamma, V)
    key = (torch.device(device), n)
    ws = _ws_cache.get(key)
    if ws is None:
        ws = torch.zeros(n + 256, dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    off = (-ws.data_ptr()) % 256
    return ws[off:off + n]


def _round_dev(round_dev, dev):
    if round_dev is not None:
        _need(round_dev, "round_dev", torch.int64, dev)
        _sized(round_dev, "round_dev", (1,))
    return _ptr(round_dev)


def markov_draft(U, W1, W2, anchor, seed, rnd=0, ws=None, T_early=None, round_dev=None):
    """x [B,G] i32, p [B,G] f32, lse [B,G] f32 = the Markov draft of one round.
    T_early [B,G+1,V] f32: target logits whose rows j < G get their softmax
    statistics into ws while the draft runs (for verify(early_stats=True)).
    round_dev: int64 [1] device tensor holding the round index (rnd ignored)."""
    L = _load()
    _need(U, "U", torch.float32)
    dev = U.device
    B, G, V = U.shape
    _need(W1, "W1", device=dev); _need(W2, "W2", W1.dtype, dev); _need(anchor, "anchor", torch.int32, dev)
    r = W1.shape[-1]
    _sized(W1, "W1", (V, r)); _sized(W2, "W2", (V, r)); _sized(anchor, "anchor", (B,))
    if T_early is not None:
        _need(T_early, "T_early", torch.float32, dev)
        _sized(T_early, "T_early", (B, G + 1, V))
    rd = _round_dev(round_dev, dev)
    x = torch.empty((B, G), dtype=torch.int32, device=dev)
    p = torch.empty((B, G), dtype=torch.float32, device=dev)
    lse = torch.empty((B, G), dtype=torch.float32, device=dev)
    ws = workspace(B, G, V, dev) if ws is None else ws
    _check(L.dspark_markov_draft_ex(_ptr(U), _ptr(T_early), _ptr(W1), _ptr(W2), _dt(W1, "W1"), _ptr(anchor), B, G,
                                    V, r, seed, rnd, rd, _ptr(x), _ptr(p), _ptr(lse), _ptr(ws), ws.numel(),
                                    _stream(dev)), "markov_draft")
    return x, p, lse


def gated_markov_draft(U, W1, W2, gate_g, gate_c, anchor, seed, rnd=0, ws=None, T_early=None, round_dev=None):
    """x, p, lse of the draft with the gated recurrent head (s_k = e_k + a_k *
    s_{k-1}, a_k = sigmoid(gate_g * e_k + gate_c), e_k = W1[x_{k-1}]; bias
    s_k . W2).  gate_g, gate_c: float32 [r].  The states stay in ws for
    verify(gated=True).  Tensor-core path only (bf16, r = 256)."""
    L = _load()
    _need(U, "U", torch.float32)
    dev = U.device
    B, G, V = U.shape
    _need(W1, "W1", device=dev); _need(W2, "W2", W1.dtype, dev); _need(anchor, "anchor", torch.int32, dev)
    r = W1.shape[-1]
    _sized(W1, "W1", (V, r)); _sized(W2, "W2", (V, r)); _sized(anchor, "anchor", (B,))
    _need(gate_g, "gate_g", torch.float32, dev); _need(gate_c, "gate_c", torch.float32, dev)
    _sized(gate_g, "gate_g", (r,)); _sized(gate_c, "gate_c", (r,))
    if T_early is not None:
        _need(T_early, "T_early", torch.float32, dev)
        _sized(T_early, "T_early", (B, G + 1, V))
    rd = _round_dev(round_dev, dev)
    x = torch.empty((B, G), dtype=torch.int32, device=dev)
    p = torch.empty((B, G), dtype=torch.float32, device=dev)
    lse = torch.empty((B, G), dtype=torch.float32, device=dev)
    ws = workspace(B, G, V, dev) if ws is None else ws
    _check(L.dspark_gated_markov_draft(_ptr(U), _ptr(T_early), _ptr(W1), _ptr(W2), _dt(W1, "W1"), _ptr(gate_g),
                                       _ptr(gate_c), _ptr(anchor), B, G, V, r, seed, rnd, rd, _ptr(x), _ptr(p),
                                       _ptr(lse), _ptr(ws), ws.numel(), _stream(dev)), "gated_markov_draft")
    return x, p, lse


def confidence(h, W1, w, anchor, x, sts_T=None):
    """c [B,G] f32 = sigmoid(w . [h_k ; W1[x_{k-1}]] / T_k)."""
    L = _load()
    _need(h, "h")
    dev = h.device
    B, G, H = h.shape
    _need(W1, "W1", device=dev); _need(w, "w", torch.float32, dev)
    _need(anchor, "anchor", torch.int32, dev); _need(x, "x", torch.int32, dev)
    if sts_T is not None:
        _need(sts_T, "sts_T", torch.float32, dev)
    if W1.dim() != 2:
        raise ValueError(f"W1 must be [V, r], got {list(W1.shape)}")
    V, r = W1.shape
    _sized(w, "w", (H + r,)); _sized(anchor, "anchor", (B,)); _sized(x, "x", (B, G)); _sized(sts_T, "sts_T", (G,))
    c = torch.empty((B, G), dtype=torch.float32, device=dev)
    _check(L.dspark_confidence(_ptr(h), _dt(h, "h"), _ptr(W1), _dt(W1, "W1"), _ptr(w), _ptr(sts_T), _ptr(anchor),
                               _ptr(x), B, G, H, r, V, _ptr(c), _stream(dev)), "confidence")
    return c


def schedule(c, sps=None, mode=SCHED_GREEDY, rnd=0, khist=None, ws=None, round_dev=None):
    """ell [B] i32, nstar [1] i32, theta [1] f64 from confidences c [B,G]."""
    L = _load()
    _need(c, "c", torch.float32)
    dev = c.device
    B, G = c.shape
    if sps is not None:
        _need(sps, "sps", torch.float32, dev)
    if khist is not None:
        _need(khist, "khist", torch.int32, dev)
    _sized(khist, "khist", (2,))
    ell = torch.empty(B, dtype=torch.int32, device=dev)
    nstar = torch.empty(1, dtype=torch.int32, device=dev)
    theta = torch.empty(1, dtype=torch.float64, device=dev)
    ws = workspace(B, G, 8, dev) if ws is None else ws
    n_sps = 0 if sps is None else sps.numel()
    rd = _round_dev(round_dev, dev)
    _check(L.dspark_schedule_ex(_ptr(c), B, G, _ptr(sps), n_sps, mode, rnd, rd, _ptr(khist), _ptr(ell),
                                _ptr(nstar), _ptr(theta), _ptr(ws), ws.numel(), _stream(dev)), "schedule")
    return ell, nstar, theta


def verify(T, U, W1, W2, anchor, x, p_d, lse_d, ell, seed, rnd=0, ws=None, early_stats=False, round_dev=None,
           advance_round=False, scratch_from_draft=False, gated=False, all_row_stats=False):
    """n [B] i32 accepted counts, tok [B] i32 corrected / bonus tokens.
    early_stats: ws already holds the target-row statistics from
    markov_draft(T_early=T).  round_dev / advance_round: the round index as a
    device int64 [1], advanced by the call's last kernel.
    scratch_from_draft: a draft_schedule on ws cleared the call's scratch.
    gated: the draft was gated_markov_draft on ws (its states are the
    residual's bias operand).  all_row_stats: take the statistics of every
    row j < ell (for acceptance_label(stats="verify")) instead of only the
    rows the accept tests reach."""
    L = _load()
    _need(T, "T", torch.float32)
    dev = T.device
    _need(U, "U", torch.float32, dev)
    B, G, V = U.shape
    if tuple(T.shape) != (B, G + 1, V):
        raise ValueError(f"T must be [B, gamma+1, V] = {(B, G + 1, V)}, got {tuple(T.shape)}")
    _need(W1, "W1", device=dev); _need(W2, "W2", W1.dtype, dev)
    for t, n in [(anchor, "anchor"), (x, "x"), (ell, "ell")]:
        _need(t, n, torch.int32, dev)
    _need(p_d, "p_d", torch.float32, dev); _need(lse_d, "lse_d", torch.float32, dev)
    r = W1.shape[-1]
    _sized(W1, "W1", (V, r)); _sized(W2, "W2", (V, r)); _sized(anchor, "anchor", (B,)); _sized(ell, "ell", (B,))
    for t, n in [(x, "x"), (p_d, "p_d"), (lse_d, "lse_d")]:
        _sized(t, n, (B, G))
    n = torch.empty(B, dtype=torch.int32, device=dev)
    tok = torch.empty(B, dtype=torch.int32, device=dev)
    ws = workspace(B, G, V, dev) if ws is None else ws
    rd = _round_dev(round_dev, dev)
    flags = ((EARLY_TARGET_STATS if early_stats else 0) | (ADVANCE_ROUND if advance_round else 0) |
             (SCRATCH_FROM_DRAFT if scratch_from_draft else 0) | (GATED_STATES if gated else 0) |
             (ALL_ROW_STATS if all_row_stats else 0))
    _check(L.dspark_verify_ex(_ptr(T), _ptr(U), _ptr(W1), _ptr(W2), _dt(W1, "W1"), _ptr(anchor), _ptr(x),
                              _ptr(p_d), _ptr(lse_d), _ptr(ell), B, G, V, r, seed, rnd, rd, flags, _ptr(n), _ptr(tok),
                              _ptr(ws), ws.numel(), _stream(dev)), "verify")
    return n, tok


def acceptance_label(T, U, W1, W2, anchor, x, lse_d, ell, ws=None, stats=None):
    """label [B, gamma] f32: sum_v min(p_d, p_t) for every verified position
    k <= ell[b] (0 elsewhere).  Tensor-core path only (bf16, r = 256).
    stats: None (the call streams the target rows' statistics first),
    "early" (ws holds them from markov_draft(T_early=T)) or "verify" (ws
    holds them from a verify or round with all_row_stats=True)."""
    L = _load()
    _need(T, "T", torch.float32)
    dev = T.device
    _need(U, "U", torch.float32, dev)
    B, G, V = U.shape
    if tuple(T.shape) != (B, G + 1, V):
        raise ValueError(f"T must be [B, gamma+1, V] = {(B, G + 1, V)}, got {tuple(T.shape)}")
    _need(W1, "W1", device=dev); _need(W2, "W2", W1.dtype, dev)
    for t, n in [(anchor, "anchor"), (x, "x"), (ell, "ell")]:
        _need(t, n, torch.int32, dev)
    _need(lse_d, "lse_d", torch.float32, dev)
    r = W1.shape[-1]
    _sized(W1, "W1", (V, r)); _sized(W2, "W2", (V, r)); _sized(anchor, "anchor", (B,)); _sized(ell, "ell", (B,))
    _sized(x, "x", (B, G)); _sized(lse_d, "lse_d", (B, G))
    label = torch.empty(B, G, dtype=torch.float32, device=dev)
    ws = workspace(B, G, V, dev) if ws is None else ws
    flags = {None: 0, "early": EARLY_TARGET_STATS, "verify": TARGET_STATS_FROM_VERIFY}[stats]
    _check(L.dspark_acceptance_label_ex(_ptr(T), _ptr(U), _ptr(W1), _ptr(W2), _dt(W1, "W1"), _ptr(anchor), _ptr(x),
                                        _ptr(lse_d), _ptr(ell), B, G, V, r, flags, _ptr(label), _ptr(ws), ws.numel(),
                                        _stream(dev)), "acceptance_label")
    return label


def sts_fit(z, ell, acc, grid):
    """Sequential temperature scaling: (T [gamma] f32, ece [gamma] f32) fitted on
    the samples (z [N, gamma] f32 logits, ell and acc [N] i32) over the grid of
    temperatures (f32), all on one device."""
    L = _load()
    _need(z, "z", torch.float32)
    dev = z.device
    N, G = z.shape
    _need(ell, "ell", torch.int32, dev); _need(acc, "acc", torch.int32, dev); _need(grid, "grid", torch.float32, dev)
    _sized(ell, "ell", (N,)); _sized(acc, "acc", (N,)); _sized(grid, "grid", (grid.numel(),))
    T = torch.empty(G, dtype=torch.float32, device=dev)
    e = torch.empty(G, dtype=torch.float32, device=dev)
    nbytes = L.dspark_sts_workspace_size(N, G, grid.numel())
    ws = torch.empty(max(256, nbytes), dtype=torch.uint8, device=dev)
    _check(L.dspark_sts_fit(_ptr(z), _ptr(ell), _ptr(acc), N, G, _ptr(grid), grid.numel(), _ptr(T), _ptr(e), _ptr(ws),
                            ws.numel(), _stream(dev)), "sts_fit")
    return T, e


class RoundOutputs:
    """Device output buffers of one round (reused across rounds)."""

    def __init__(self, B, G, device):
        i32, f32 = torch.int32, torch.float32
        self.x = torch.empty((B, G), dtype=i32, device=device)
        self.p = torch.empty((B, G), dtype=f32, device=device)
        self.lse = torch.empty((B, G), dtype=f32, device=device)
        self.c = torch.empty((B, G), dtype=f32, device=device)
        self.ell = torch.empty(B, dtype=i32, device=device)
        self.nstar = torch.empty(1, dtype=i32, device=device)
        self.theta = torch.empty(1, dtype=torch.float64, device=device)
        self.n = torch.empty(B, dtype=i32, device=device)
        self.tok = torch.empty(B, dtype=i32, device=device)

    def as_dict(self):
        return dict(x=self.x, p=self.p, lse=self.lse, c=self.c, ell=self.ell, nstar=self.nstar,
                    theta=self.theta, n=self.n, tok=self.tok)

    def check(self, B, G, device):
        """Raise unless every buffer has the shape, dtype and device of a
        round of B requests and G positions."""
        i32, f32 = torch.int32, torch.float32
        want = dict(x=((B, G), i32), p=((B, G), f32), lse=((B, G), f32), c=((B, G), f32), ell=((B,), i32),
                    nstar=((1,), i32), theta=((1,), torch.float64), n=((B,), i32), tok=((B,), i32))
        for name, (shape, dtype) in want.items():
            t = getattr(self, name)
            _need(t, f"out.{name}", dtype, device)
            _sized(t, f"out.{name}", shape)


def _round_args(U, T, W1, W2, h, w, anchor, sps, khist, sts_T):
    # shared checks of round and draft_schedule (T may be None for the latter)
    _need(U, "U", torch.float32)
    dev = U.device
    B, G, V = U.shape
    if T is not None:
        _need(T, "T", torch.float32, dev)
        if tuple(T.shape) != (B, G + 1, V):
            raise ValueError(f"T must be [B, gamma+1, V] = {(B, G + 1, V)}, got {tuple(T.shape)}")
    _need(W1, "W1", device=dev); _need(W2, "W2", W1.dtype, dev); _need(h, "h", device=dev)
    _need(w, "w", torch.float32, dev); _need(anchor, "anchor", torch.int32, dev)
    if sps is not None:
        _need(sps, "sps", torch.float32, dev)
    if khist is not None:
        _need(khist, "khist", torch.int32, dev)
    if sts_T is not None:
        _need(sts_T, "sts_T", torch.float32, dev)
    if h.dim() != 3:
        raise ValueError(f"h must be [B, gamma, H], got {list(h.shape)}")
    r, H = W1.shape[-1], h.shape[2]
    _sized(W1, "W1", (V, r)); _sized(W2, "W2", (V, r)); _sized(h, "h", (B, G, H)); _sized(w, "w", (H + r,))
    _sized(anchor, "anchor", (B,)); _sized(khist, "khist", (2,)); _sized(sts_T, "sts_T", (G,))
    return dev, B, G, V, r, H


def draft_schedule(U, W1, W2, h, w, anchor, seed, rnd=0, sps=None, mode=SCHED_GREEDY, khist=None, sts_T=None,
                   out=None, ws=None, T_early=None, round_dev=None, chain_stats=False):
    """The first stage of a round (draft, confidence head, schedule; one
    persistent launch on the tensor-core path) into out.x, p, lse, c, ell,
    nstar, theta.  T_early: target logits whose statistics the draft takes
    along (chain_stats: only of the rows the accept tests can reach; verify
    with early_stats=True either way).  Returns the RoundOutputs."""
    L = _load()
    if chain_stats and T_early is None:
        raise ValueError("chain_stats needs T_early")
    dev, B, G, V, r, H = _round_args(U, T_early, W1, W2, h, w, anchor, sps, khist, sts_T)
    out = RoundOutputs(B, G, dev) if out is None else out
    out.check(B, G, dev)
    ws = workspace(B, G, V, dev) if ws is None else ws
    n_sps = 0 if sps is None else sps.numel()
    rd = _round_dev(round_dev, dev)
    _check(L.dspark_draft_schedule_ex(_ptr(U), _ptr(T_early), _ptr(W1), _ptr(W2), _dt(W1, "W1"), _ptr(h),
                                      _dt(h, "h"), _ptr(w), _ptr(sts_T), _ptr(anchor), B, G, V, r, H, _ptr(sps),
                                      n_sps, mode, _ptr(khist), seed, rnd, rd,
                                      CHAIN_TARGET_STATS if chain_stats else 0, _ptr(out.x), _ptr(out.p),
                                      _ptr(out.lse), _ptr(out.c), _ptr(out.ell), _ptr(out.nstar), _ptr(out.theta),
                                      _ptr(ws), ws.numel(), _stream(dev)), "draft_schedule")
    return out


def round(U, T, W1, W2, h, w, anchor, seed, rnd=0, sps=None, mode=SCHED_GREEDY, khist=None, sts_T=None,
          out=None, ws=None, early_stats=False, round_dev=None, advance_round=False, all_row_stats=False,
          chain_stats=False):
    """One whole round (draft, confidence, schedule, verify) on U's device.
    early_stats: the draft takes the target rows' statistics while it runs.
    chain_stats: the draft takes those of the rows the accept tests reach.
    all_row_stats: verification takes the statistics of every row j < ell
    (otherwise only the rows the accept tests reach).
    round_dev / advance_round: the round index as a device int64 [1] (rnd
    ignored), advanced by the round's last kernel.
    Returns a RoundOutputs (device tensors)."""
    L = _load()
    _need(T, "T", torch.float32)
    dev, B, G, V, r, H = _round_args(U, T, W1, W2, h, w, anchor, sps, khist, sts_T)
    out = RoundOutputs(B, G, dev) if out is None else out
    out.check(B, G, dev)
    ws = workspace(B, G, V, dev) if ws is None else ws
    n_sps = 0 if sps is None else sps.numel()
    rd = _round_dev(round_dev, dev)
    flags = ((EARLY_TARGET_STATS if early_stats else 0) | (ADVANCE_ROUND if advance_round else 0) |
             (ALL_ROW_STATS if all_row_stats else 0) | (CHAIN_TARGET_STATS if chain_stats else 0))
    _check(L.dspark_round_ex(_ptr(U), _ptr(T), _ptr(W1), _ptr(W2), _dt(W1, "W1"), _ptr(h), _dt(h, "h"), _ptr(w),
                             _ptr(sts_T), _ptr(anchor), B, G, V, r, H, _ptr(sps), n_sps, mode, _ptr(khist), seed,
                             rnd, rd, flags, _ptr(out.x), _ptr(out.p), _ptr(out.lse), _ptr(out.c), _ptr(out.ell),
                             _ptr(out.nstar), _ptr(out.theta), _ptr(out.n), _ptr(out.tok), _ptr(ws), ws.numel(),
                             _stream(dev)), "round")
    return out


def selftest_wait_timeout(mode, ws):
    """Enqueue the bounded-wait self-test (mode 0: mbarrier, 1: grid barrier);
    its status word then reads ERR_TIMEOUT (see read_status)."""
    L = _load()
    _check(L.dspark_selftest_wait_timeout(int(mode), _ptr(ws), ws.numel(), _stream(ws.device)),
           "selftest_wait_timeout")


def read_status(ws, device=None):
    """Synchronise the current stream and return (and clear) the status word."""
    L = _load()
    st = ctypes.c_int(0)
    dev = ws.device if device is None else device
    _check(L.dspark_read_status(_ptr(ws), ctypes.byref(st), _stream(dev)), "read_status")
    return int(st.value)
