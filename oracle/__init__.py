"""ctypes shim over the plain-C double-precision oracle (``dspark_oracle.c``).

TEST INFRASTRUCTURE ONLY.  The oracle is the independent, slow, obviously
correct CPU statement of the DSpark per-round hot path against which the CUDA
library is checked.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it; the
library itself never does.  It shares no code with the CUDA path.

All array arguments are numpy arrays on the host.  bf16 tensors are passed as
their raw ``uint16`` bit patterns.
"""
import ctypes
import numpy as np

from . import build as _build

_lib = None

F32, BF16 = 0, 1

_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")


def lib():
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        c_int, c_u32, c_u64, c_dbl = ctypes.c_int, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_double
        vp = ctypes.c_void_p
        L.oracle_philox4x32_10.argtypes = [ctypes.POINTER(c_u32), ctypes.POINTER(c_u32), ctypes.POINTER(c_u32)]
        L.oracle_philox4x32_10.restype = None
        L.oracle_rng_word.argtypes = [c_u64, c_u64, c_u32, c_u32, c_u32, c_u32]
        L.oracle_rng_word.restype = c_u32
        L.oracle_u01.argtypes = [c_u32]
        L.oracle_u01.restype = c_dbl
        L.oracle_philox_word.argtypes = [c_u64, c_u64, c_u32, c_u32, c_u32, c_u32, c_u32]
        L.oracle_philox_word.restype = c_u32
        L.oracle_u01_bits.argtypes = [c_u32]
        L.oracle_u01_bits.restype = c_dbl
        L.oracle_gumbel_from_bits.argtypes = [c_u32]
        L.oracle_gumbel_from_bits.restype = c_dbl
        L.oracle_draft_logits.argtypes = [c_int, c_int, vp, vp, vp, c_int, c_int, vp]
        L.oracle_draft_logits.restype = None
        L.oracle_draft_probs.argtypes = [c_int, c_int, vp, vp, vp, c_int, c_int, vp]
        L.oracle_draft_probs.restype = None
        L.oracle_logsumexp.argtypes = [c_int, vp]
        L.oracle_logsumexp.restype = c_dbl
        L.oracle_softmax.argtypes = [c_int, vp, vp]
        L.oracle_softmax.restype = None
        L.oracle_block_sample.argtypes = [c_int, vp, c_u64, c_u64, c_u32, c_u32, ctypes.POINTER(c_dbl)]
        L.oracle_block_sample.restype = c_int
        L.oracle_block_draw.argtypes = [c_int, vp, c_dbl, c_u64, c_u64, c_u32, c_u32, c_u32, ctypes.POINTER(c_dbl)]
        L.oracle_block_draw.restype = c_int
        L.oracle_softmax_draw.argtypes = [c_int, vp, c_u64, c_u64, c_u32, c_u32, c_u32, ctypes.POINTER(c_dbl)]
        L.oracle_softmax_draw.restype = c_int
        L.oracle_residual.argtypes = [c_int, vp, vp, vp]
        L.oracle_residual.restype = None
        L.oracle_acceptance_label.argtypes = [c_int, vp, vp]
        L.oracle_acceptance_label.restype = c_dbl
        L.oracle_draft.argtypes = [c_int, c_int, c_int, c_int, vp, vp, vp, c_int, vp, vp,
                                   c_u64, c_u64, c_int, c_int, vp, vp, vp, vp]
        L.oracle_draft.restype = c_int
        L.oracle_confidence.argtypes = [c_int, c_int, c_int, c_int, vp, c_int, vp, c_int, vp, vp,
                                        vp, vp, c_int, vp]
        L.oracle_confidence.restype = c_int
        L.oracle_schedule.argtypes = [c_int, c_int, vp, vp, c_int, c_int, c_int, vp, vp, vp, vp]
        L.oracle_schedule.restype = c_int
        L.oracle_verify.argtypes = [c_int, c_int, c_int, c_int, vp, vp, vp, vp, c_int, vp, vp, vp,
                                    c_u64, c_u64, c_int, c_int, vp, vp, vp, vp, vp, vp]
        L.oracle_verify.restype = c_int
        L.oracle_gated_states.argtypes = [c_int, c_int, c_int, vp, c_int, vp, vp, c_int, vp, c_int, vp]
        L.oracle_gated_states.restype = c_int
        L.oracle_gated_draft.argtypes = [c_int, c_int, c_int, c_int, vp, vp, vp, c_int, vp, vp, c_int, vp, vp,
                                         c_u64, c_u64, c_int, c_int, vp, vp, vp, vp]
        L.oracle_gated_draft.restype = c_int
        L.oracle_gated_verify.argtypes = [c_int, c_int, c_int, c_int, vp, vp, vp, vp, c_int, vp, vp, c_int, vp, vp,
                                          vp, c_u64, c_u64, c_int, c_int, vp, vp, vp, vp, vp, vp]
        L.oracle_gated_verify.restype = c_int
        L.oracle_num_threads.argtypes = []
        L.oracle_num_threads.restype = c_int
        L.oracle_set_num_threads.argtypes = [c_int]
        L.oracle_set_num_threads.restype = None
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _wdt(a):
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"weights must be float32 or bf16 bits (uint16), got {a.dtype}")


def _c(a, dtype=None):
    if a is None:
        return None
    a = np.ascontiguousarray(a if dtype is None else a.astype(dtype, copy=False))
    return a


def _check(status, what):
    if status != 0:
        raise RuntimeError(f"oracle {what} failed with status {status}")


# --------------------------------------------------------------------------
# generator
# --------------------------------------------------------------------------

def philox4x32_10(ctr, key):
    c = (ctypes.c_uint32 * 4)(*[int(x) & 0xffffffff for x in ctr])
    k = (ctypes.c_uint32 * 2)(*[int(x) & 0xffffffff for x in key])
    o = (ctypes.c_uint32 * 4)()
    lib().oracle_philox4x32_10(c, k, o)
    return [int(o[i]) for i in range(4)]


def rng_word(seed, rnd, stream, req, k, v):
    return int(lib().oracle_rng_word(seed, rnd, stream, req, k, v))


def philox_word(seed, rnd, stream, req, k, c0, word):
    return int(lib().oracle_philox_word(seed, rnd, stream, req, k, c0, word))


def u01(word):
    """The accept uniform from a whole 32-bit word (its top 23 bits)."""
    return float(lib().oracle_u01(word))


def block_draw(w, seed, rnd, stream, req, k, logscale=0.0):
    """Two-level draw from non-negative weights w: (entry, margin)."""
    w = _c(w, np.float64)
    m = ctypes.c_double(0.0)
    x = lib().oracle_block_draw(w.size, _ptr(w), float(logscale), seed, rnd, stream, req, k, ctypes.byref(m))
    return int(x), float(m.value)


def softmax_draw(score, seed, rnd, stream, req, k):
    """Two-level draw from softmax(score): (entry, margin)."""
    score = _c(score, np.float64)
    m = ctypes.c_double(0.0)
    x = lib().oracle_softmax_draw(score.size, _ptr(score), seed, rnd, stream, req, k, ctypes.byref(m))
    return int(x), float(m.value)


def block_sample(l, seed, rnd, req, k):
    """The draft sampler's draw from softmax(l): (token, margin)."""
    l = _c(l, np.float64)
    m = ctypes.c_double(0.0)
    x = lib().oracle_block_sample(l.size, _ptr(l), seed, rnd, req, k, ctypes.byref(m))
    return int(x), float(m.value)


def u01_bits(m):
    return float(lib().oracle_u01_bits(m))


def gumbel_from_bits(m):
    return float(lib().oracle_gumbel_from_bits(m))


def draft_logits(U_row, W1, W2, prev):
    U_row = _c(U_row, np.float32)
    W1, W2 = _c(W1), _c(W2)
    V, r = W2.shape
    out = np.empty(V, np.float64)
    lib().oracle_draft_logits(V, r, _ptr(U_row), _ptr(W1), _ptr(W2), _wdt(W1), int(prev), _ptr(out))
    return out


def draft_probs(U_row, W1, W2, prev):
    U_row = _c(U_row, np.float32)
    W1, W2 = _c(W1), _c(W2)
    V, r = W2.shape
    out = np.empty(V, np.float64)
    lib().oracle_draft_probs(V, r, _ptr(U_row), _ptr(W1), _ptr(W2), _wdt(W1), int(prev), _ptr(out))
    return out


def logsumexp(l):
    l = _c(l, np.float64)
    return float(lib().oracle_logsumexp(l.size, _ptr(l)))


def softmax(l):
    l = _c(l, np.float64)
    out = np.empty_like(l)
    lib().oracle_softmax(l.size, _ptr(l), _ptr(out))
    return out


def residual(p_t, p_d):
    p_t, p_d = _c(p_t, np.float64), _c(p_d, np.float64)
    out = np.empty_like(p_t)
    lib().oracle_residual(p_t.size, _ptr(p_t), _ptr(p_d), _ptr(out))
    return out


def acceptance_label(p_d, p_t):
    p_d, p_t = _c(p_d, np.float64), _c(p_t, np.float64)
    return float(lib().oracle_acceptance_label(p_d.size, _ptr(p_d), _ptr(p_t)))


# --------------------------------------------------------------------------
# the four steps
# --------------------------------------------------------------------------

def draft(U, W1, W2, anchor, seed, rnd, x_force=None, b0=0, b1=None):
    """Markov draft.  Returns dict(x [B,G] i32, p, lse, margin [B,G] f64).
    Rows outside [b0, b1) are left as -1 / NaN."""
    U = _c(U, np.float32)
    B, G, V = U.shape
    W1, W2 = _c(W1), _c(W2)
    r = W1.shape[1]
    anchor = _c(anchor, np.int32)
    xf = _c(x_force, np.int32)
    b1 = B if b1 is None else b1
    x = np.full((B, G), -1, np.int32)
    p = np.full((B, G), np.nan)
    lse = np.full((B, G), np.nan)
    mg = np.full((B, G), np.nan)
    st = lib().oracle_draft(B, G, V, r, _ptr(U), _ptr(W1), _ptr(W2), _wdt(W1), _ptr(anchor), _ptr(xf),
                            seed, rnd, b0, b1, _ptr(x), _ptr(p), _ptr(lse), _ptr(mg))
    _check(st, "draft")
    return dict(x=x, p=p, lse=lse, margin=mg)


def confidence(h, W1, w, anchor, x, sts_T=None):
    """Confidence head c [B,G] (f64).  h is float32 or bf16 bits."""
    h = _c(h)
    B, G, H = h.shape
    W1 = _c(W1)
    V, r = W1.shape
    w = _c(w, np.float32)
    anchor, x = _c(anchor, np.int32), _c(x, np.int32)
    sts = _c(sts_T, np.float32)
    c = np.empty((B, G), np.float64)
    st = lib().oracle_confidence(B, G, H, r, _ptr(h), _wdt(h), _ptr(W1), _wdt(W1), _ptr(w), _ptr(sts),
                                 _ptr(anchor), _ptr(x), V, _ptr(c))
    _check(st, "confidence")
    return c


MODE_FIXED, MODE_GREEDY, MODE_TOPK = 0, 1, 2


def schedule(c, sps=None, mode=MODE_GREEDY, K=-1):
    """Prefix scheduler.  Returns dict(ell [R] i32, nstar, theta, order [R*G])."""
    c = _c(c, np.float64)
    R, G = c.shape
    sps = _c(sps, np.float32)
    n_sps = 0 if sps is None else sps.size
    ell = np.empty(R, np.int32)
    nstar = np.zeros(1, np.int32)
    theta = np.zeros(1, np.float64)
    order = np.empty(R * G, np.int32)
    st = lib().oracle_schedule(R, G, _ptr(c), _ptr(sps), n_sps, mode, int(K), _ptr(ell), _ptr(nstar),
                               _ptr(theta), _ptr(order))
    _check(st, "schedule")
    return dict(ell=ell, nstar=int(nstar[0]), theta=float(theta[0]), order=order)


def verify(T, U, W1, W2, anchor, x, ell, seed, rnd, b0=0, b1=None):
    """Rejection-sampling verification.  Returns dict(n, y, flags [B] i32,
    ratio, umargin [B,G] f64, ymargin [B] f64).  Rows outside [b0, b1) are -1."""
    T, U = _c(T, np.float32), _c(U, np.float32)
    B, G, V = U.shape
    assert T.shape == (B, G + 1, V)
    W1, W2 = _c(W1), _c(W2)
    r = W1.shape[1]
    anchor, x, ell = _c(anchor, np.int32), _c(x, np.int32), _c(ell, np.int32)
    b1 = B if b1 is None else b1
    n = np.full(B, -1, np.int32)
    y = np.full(B, -1, np.int32)
    fl = np.zeros(B, np.int32)
    ratio = np.full((B, G), np.nan)
    um = np.full((B, G), np.nan)
    ym = np.full(B, np.nan)
    st = lib().oracle_verify(B, G, V, r, _ptr(T), _ptr(U), _ptr(W1), _ptr(W2), _wdt(W1), _ptr(anchor),
                             _ptr(x), _ptr(ell), seed, rnd, b0, b1, _ptr(n), _ptr(y), _ptr(fl),
                             _ptr(ratio), _ptr(um), _ptr(ym))
    _check(st, "verify")
    return dict(n=n, y=y, flags=fl, ratio=ratio, umargin=um, ymargin=ym)


# --------------------------------------------------------------------------
# the gated recurrent head (e_k = W1[x_{k-1}], a_k = sigmoid(g * e_k + c),
# s_k = e_k + a_k * s_{k-1}, bias s_k . W2[v]; g, c float32 [r])
# --------------------------------------------------------------------------

def gated_states(W1, g, c, anchor, x_prefix, G, bf16_state=False):
    """The states s_1..s_G [G, r] (f64) of one request: anchor, then x_prefix[0..G-2].
    bf16_state: each state rounded to bf16 as it is formed (the precision a
    tensor-core operand holds it in); False: the exact definition."""
    W1 = _c(W1)
    V, r = W1.shape
    g, c = _c(g, np.float32), _c(c, np.float32)
    xp = _c(np.asarray(x_prefix, np.int32).reshape(-1)[:max(G - 1, 0)], np.int32) if G > 1 else None
    out = np.empty((G, r), np.float64)
    st = lib().oracle_gated_states(G, V, r, _ptr(W1), _wdt(W1), _ptr(g), _ptr(c), int(anchor), _ptr(xp),
                                   int(bool(bf16_state)), _ptr(out))
    _check(st, "gated_states")
    return out


def gated_draft(U, W1, W2, g, c, anchor, seed, rnd, x_force=None, b0=0, b1=None, bf16_state=False):
    """The draft with the gated recurrent head; as draft() (bf16_state as for
    gated_states)."""
    U = _c(U, np.float32)
    B, G, V = U.shape
    W1, W2 = _c(W1), _c(W2)
    r = W1.shape[1]
    g, c = _c(g, np.float32), _c(c, np.float32)
    anchor = _c(anchor, np.int32)
    xf = _c(x_force, np.int32)
    b1 = B if b1 is None else b1
    x = np.full((B, G), -1, np.int32)
    p = np.full((B, G), np.nan)
    lse = np.full((B, G), np.nan)
    mg = np.full((B, G), np.nan)
    st = lib().oracle_gated_draft(B, G, V, r, _ptr(U), _ptr(W1), _ptr(W2), _wdt(W1), _ptr(g), _ptr(c),
                                  int(bool(bf16_state)), _ptr(anchor), _ptr(xf), seed, rnd, b0, b1, _ptr(x), _ptr(p), _ptr(lse), _ptr(mg))
    _check(st, "gated_draft")
    return dict(x=x, p=p, lse=lse, margin=mg)


def gated_verify(T, U, W1, W2, g, c, anchor, x, ell, seed, rnd, b0=0, b1=None, bf16_state=False):
    """Verification of a gated-head draft; as verify() (bf16_state as for
    gated_states)."""
    T, U = _c(T, np.float32), _c(U, np.float32)
    B, G, V = U.shape
    assert T.shape == (B, G + 1, V)
    W1, W2 = _c(W1), _c(W2)
    r = W1.shape[1]
    g, c = _c(g, np.float32), _c(c, np.float32)
    anchor, x, ell = _c(anchor, np.int32), _c(x, np.int32), _c(ell, np.int32)
    b1 = B if b1 is None else b1
    n = np.full(B, -1, np.int32)
    y = np.full(B, -1, np.int32)
    fl = np.zeros(B, np.int32)
    ratio = np.full((B, G), np.nan)
    um = np.full((B, G), np.nan)
    ym = np.full(B, np.nan)
    st = lib().oracle_gated_verify(B, G, V, r, _ptr(T), _ptr(U), _ptr(W1), _ptr(W2), _wdt(W1), _ptr(g), _ptr(c),
                                   int(bool(bf16_state)), _ptr(anchor), _ptr(x), _ptr(ell), seed, rnd, b0, b1, _ptr(n), _ptr(y), _ptr(fl),
                                   _ptr(ratio), _ptr(um), _ptr(ym))
    _check(st, "gated_verify")
    return dict(n=n, y=y, flags=fl, ratio=ratio, umargin=um, ymargin=ym)


def num_threads():
    return int(lib().oracle_num_threads())


def set_num_threads(n):
    """Threads of the parallel request loops from now on (n >= 1)."""
    lib().oracle_set_num_threads(int(n))
