"""CPU oracle (float64) for the state-passing mixer forward and decode update.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by
``__graft_entry__.smoke()`` and by the benchmark's CPU-baseline leg, never by
the product package.  It shares no code with the CUDA path; the only common
module is ``synth`` (seeded input draws, no method arithmetic).

The arithmetic lives in ``oracle.c`` (plain C, float64, literal loops; see the
header there for what each function follows).  This module compiles it with
gcc on first use and marshals numpy arrays.

Functions
---------
conv_state_fwd(x, w, bias, S, apply_silu=True) -> (u, F)
    Causal depthwise conv with an explicit (K-1)-sample state in the
    extended-sequence form ("Chapter 7: state, chunking and incremental
    inference", section on defining the state through the extended sequence).
ssm_scan(u, dt, A, B, C, h0) -> (y, hT)
    Scalar-decay recurrence h_t = exp(dt_t A_h) h_{t-1} + x_t B_t^T,
    y_t = h_t C_t ("Understanding and Improving Length Generalization in
    Recurrent Models", Eq. (1), from a non-zero h_{-1} as in Eq. (4)).
conv_state_bwd(x, w, bias, S, dy, dF, apply_silu=True) -> (dx, dS, dw, dbias)
    Its gradient with state (same chapter, section on the backward pass
    with state).
mixer_update(...) -> (y, conv_pool', ssm_pool', n_skipped)
    Single/multi-token update over a circular conv-state pool (same chapter,
    sections on the single-token update, circular mode and continuous
    batching), followed by the recurrence on the pool's SSM state.
mixer_fwd(...) -> (y, F, hT)
    conv_state_fwd then ssm_scan (a segment of the streaming forward).
mamba2_mixer_fwd(...) -> (y, F, hT)
    The full Mamba-2 mixer wiring: the conv over all xBC channels, dt bias
    and softplus, the dt-scaled input, the D skip and the SiLU(z) gate.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int32)
_L = ctypes.c_long


def build(force: bool = False) -> str:
    """Compile oracle.c -> _build/liboracle.so (gcc, -O2, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off",
                               "-std=c11", "-fPIC", "-shared", "-pthread", _SRC,
                               "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            l = ctypes.CDLL(build())
            l.orc_conv_state_fwd.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _L, _L, _L,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_int]
            l.orc_conv_state_bwd.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp,
                                             _L, _L, _L, ctypes.c_int, ctypes.c_int, ctypes.c_int]
            l.orc_ssm_scan.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _L, _L, _L,
                                       _L, _L, _L, ctypes.c_int]
            l.orc_ssm_scan_bwd.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp,
                                           _dp, _dp, _dp, _dp, _L, _L, _L, _L, _L, _L,
                                           ctypes.c_int]
            l.orc_mixer_update.argtypes = [_dp, _dp, _dp, _dp, _L, _L, _ip, _ip, _dp, _dp,
                                           _dp, _dp, _dp, _dp, _L, _L, _L, _L, _L, _L,
                                           ctypes.c_int, ctypes.c_int]
            l.orc_mamba2_scan.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _L, _L,
                                          _L, _L, _L, _L, ctypes.c_int]
            l.orc_num_threads.argtypes = [ctypes.c_int]
            for f in (l.orc_conv_state_fwd, l.orc_conv_state_bwd, l.orc_ssm_scan, l.orc_ssm_scan_bwd,
                      l.orc_mixer_update, l.orc_mamba2_scan, l.orc_num_threads):
                f.restype = ctypes.c_int
            _lib = l
    return _lib


def num_threads(nthreads: int = 0) -> int:
    return int(lib().orc_num_threads(nthreads))


def _f64(a) -> np.ndarray:
    if a is None:
        return None
    if hasattr(a, "f64"):
        a = a.f64()
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    if a is None:
        return ctypes.cast(None, _dp)
    return a.ctypes.data_as(_dp)


def conv_state_fwd(x, w, bias=None, S=None, apply_silu: bool = True, nthreads: int = 0):
    """x [Bz, L, D], w [D, K], bias [D] | None, S [Bz, D, K-1] | None.

    Returns u [Bz, L, D] and the final state F [Bz, D, K-1] (float64)."""
    x, w, bias, S = _f64(x), _f64(w), _f64(bias), _f64(S)
    Bz, L, D = x.shape
    K = w.shape[1]
    u = np.empty((Bz, L, D))
    F = np.empty((Bz, D, K - 1))
    rc = lib().orc_conv_state_fwd(_ptr(x), _ptr(w), _ptr(bias), _ptr(S), _ptr(u), _ptr(F),
                                  Bz, L, D, K, int(bool(apply_silu)), nthreads)
    if rc != 0:
        raise ValueError("orc_conv_state_fwd: bad sizes")
    return u, F


def conv_state_bwd(x, w, bias, S, dy, dF=None, apply_silu: bool = True, nthreads: int = 0):
    """Gradient of conv_state_fwd: x [Bz, L, D], w [D, K], bias [D] | None,
    S [Bz, D, K-1] | None, dy = dL/du [Bz, L, D], dF = dL/dF [Bz, D, K-1] | None.

    Returns dx [Bz, L, D], dS [Bz, D, K-1], dw [D, K], dbias [D] (float64)."""
    x, w, bias, S, dy, dF = (_f64(a) for a in (x, w, bias, S, dy, dF))
    Bz, L, D = x.shape
    K = w.shape[1]
    dx = np.empty((Bz, L, D))
    dS = np.empty((Bz, D, K - 1))
    dw = np.empty((D, K))
    db = np.empty(D)
    rc = lib().orc_conv_state_bwd(_ptr(x), _ptr(w), _ptr(bias), _ptr(S), _ptr(dy), _ptr(dF),
                                  _ptr(dx), _ptr(dS), _ptr(dw), _ptr(db), Bz, L, D, K,
                                  int(bool(apply_silu)), nthreads)
    if rc != 0:
        raise ValueError("orc_conv_state_bwd: bad sizes")
    return dx, dS, dw, db


def ssm_scan(u, dt, A, B, C, h0=None, nthreads: int = 0):
    """u [Bz, L, H, P] (or [Bz, L, D]), dt [Bz, L, H], A [H], B/C [Bz, L, G, N],
    h0 [Bz, H, P, N] | None.  Returns y [Bz, L, H, P] and hT [Bz, H, P, N]."""
    dt, A, B, C, h0 = _f64(dt), _f64(A), _f64(B), _f64(C), _f64(h0)
    Bz, L, H = dt.shape
    G, N = B.shape[2], B.shape[3]
    u = _f64(u)
    P = u.shape[3] if u.ndim == 4 else u.shape[2] // H
    u = u.reshape(Bz, L, H, P)
    y = np.empty((Bz, L, H, P))
    hT = np.empty((Bz, H, P, N))
    rc = lib().orc_ssm_scan(_ptr(u), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(h0),
                            _ptr(y), _ptr(hT), Bz, L, H, P, N, G, nthreads)
    if rc != 0:
        raise ValueError("orc_ssm_scan: bad sizes")
    return y, hT


def ssm_scan_bwd(u, dt, A, B, C, h0, dy, dhT=None, nthreads: int = 0):
    """Gradient of ssm_scan: dy = dL/dy [Bz, L, H, P], dhT = dL/dhT [Bz, H, P, N] | None.

    Returns du [Bz, L, H, P], ddt [Bz, L, H], dA [H], dB [Bz, L, G, N],
    dC [Bz, L, G, N] and dh0 [Bz, H, P, N] (float64)."""
    dt, A, B, C, h0, dhT = _f64(dt), _f64(A), _f64(B), _f64(C), _f64(h0), _f64(dhT)
    Bz, L, H = dt.shape
    G, N = B.shape[2], B.shape[3]
    u = _f64(u)
    P = u.shape[3] if u.ndim == 4 else u.shape[2] // H
    u = u.reshape(Bz, L, H, P)
    dy = _f64(dy).reshape(Bz, L, H, P)
    du = np.empty((Bz, L, H, P))
    ddt = np.empty((Bz, L, H))
    dA = np.empty((H,))
    dB = np.empty((Bz, L, G, N))
    dC = np.empty((Bz, L, G, N))
    dh0 = np.empty((Bz, H, P, N))
    rc = lib().orc_ssm_scan_bwd(_ptr(u), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(h0),
                                _ptr(dy), _ptr(dhT), _ptr(du), _ptr(ddt), _ptr(dA), _ptr(dB),
                                _ptr(dC), _ptr(dh0), Bz, L, H, P, N, G, nthreads)
    if rc != 0:
        raise ValueError("orc_ssm_scan_bwd: bad sizes")
    return du, ddt, dA, dB, dC, dh0


def mixer_fwd(x, dt, A, B, C, w, bias, conv_state=None, h0=None, nthreads: int = 0):
    """One segment of the streaming forward: conv (with state) + SiLU, then
    the scan from h0.  Returns y [Bz, L, H, P], F [Bz, D, K-1], hT."""
    u, F = conv_state_fwd(x, w, bias, conv_state, True, nthreads)
    y, hT = ssm_scan(u, dt, A, B, C, h0, nthreads)
    return y, F, hT


def mamba2_mixer_fwd(xBC, z, dt_raw, dt_bias, A, D_skip, w, bias, conv_state, h0, H, G, N,
                     nthreads: int = 0):
    """The full Mamba-2 mixer wiring over one segment (the Mamba-2 layers of
    "Understanding and Improving Length Generalization in Recurrent Models";
    the xBC conv of "Chapter 7: state, chunking and incremental inference").

    xBC [Bz, L, D + 2 G N] (channels [0, D) are x, then B, then C), z [Bz, L,
    D] | None (no gate), dt_raw [Bz, L, H], dt_bias [H] | None, A [H],
    D_skip [H] | None, w [D + 2 G N, K], bias [D + 2 G N] | None,
    conv_state [Bz, D + 2 G N, K-1] | None, h0 [Bz, H, P, N] | None.
    The conv (+ SiLU) runs over every channel; then per token
    dt = softplus(dt_raw + dt_bias), a = exp(dt A_h), h = a h + dt x B^T,
    y = (h C + D_h x) SiLU(z).  Returns y [Bz, L, H, P], F [Bz, D + 2 G N,
    K-1] and hT [Bz, H, P, N] (float64)."""
    u, F = conv_state_fwd(xBC, w, bias, conv_state, True, nthreads)
    dt_raw, dt_bias, A, D_skip, h0 = _f64(dt_raw), _f64(dt_bias), _f64(A), _f64(D_skip), _f64(h0)
    z = _f64(z)
    Bz, L, Dt = u.shape
    P = (Dt - 2 * G * N) // H
    if H * P + 2 * G * N != Dt or dt_raw.shape != (Bz, L, H):
        raise ValueError("mamba2_mixer_fwd: channel count is not H P + 2 G N")
    y = np.empty((Bz, L, H, P))
    hT = np.empty((Bz, H, P, N))
    rc = lib().orc_mamba2_scan(_ptr(u), _ptr(z), _ptr(dt_raw), _ptr(dt_bias), _ptr(A),
                               _ptr(D_skip), _ptr(h0), _ptr(y), _ptr(hT), Bz, L, H, P, N, G,
                               nthreads)
    if rc != 0:
        raise ValueError("orc_mamba2_scan: bad sizes")
    return y, F, hT


def mixer_update(x, w, bias, conv_pool, cache_seqlens, conv_state_indices, dt, A, B, C,
                 ssm_pool, nthreads: int = 0):
    """x [Bz, L_new, D]; conv_pool [pool, D, S_len]; cache_seqlens [Bz] int, or
    None for the non-circular mode (each row holds its newest S_len inputs,
    oldest first, and is shifted by L_new);
    conv_state_indices [Bz] int | None (identity); dt [Bz, L_new, H]; A [H];
    B/C [Bz, L_new, G, N]; ssm_pool [pool, H, P, N].

    Returns (y [Bz, L_new, H, P], new conv pool, new SSM pool, n_skipped).
    The input pools are not modified."""
    x, w, bias = _f64(x), _f64(w), _f64(bias)
    dt, A, B, C = _f64(dt), _f64(A), _f64(B), _f64(C)
    cp = _f64(conv_pool).copy()
    sp = _f64(ssm_pool).copy()
    Bz, Lnew, D = x.shape
    H = dt.shape[2]
    pool, _, S_len = cp.shape
    P = D // H
    G, N = B.shape[2], B.shape[3]
    K = w.shape[1]
    sl = None
    if cache_seqlens is not None:
        sl = np.ascontiguousarray(getattr(cache_seqlens, "data", cache_seqlens), dtype=np.int32)
    ix = None
    if conv_state_indices is not None:
        ix = np.ascontiguousarray(getattr(conv_state_indices, "data", conv_state_indices),
                                  dtype=np.int32)
    y = np.empty((Bz, Lnew, H, P))
    rc = lib().orc_mixer_update(_ptr(x), _ptr(w), _ptr(bias), _ptr(cp), pool, S_len,
                                sl.ctypes.data_as(_ip) if sl is not None else ctypes.cast(None, _ip),
                                ix.ctypes.data_as(_ip) if ix is not None else ctypes.cast(None, _ip),
                                _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(sp), _ptr(y),
                                Bz, Lnew, H, P, N, G, K, nthreads)
    if rc < 0:
        raise ValueError("orc_mixer_update: bad sizes")
    return y, cp, sp, rc


# ---------------------------------------------------------------------------
# state-passing training utilities ("Understanding and Improving Length
# Generalization in Recurrent Models", sections 4.2-4.4 and 3.5)
# ---------------------------------------------------------------------------

def state_reset(u, p_reset, h, conv_state=None):
    """State passing with occasional resets (section 4.4): batch row b starts
    from zero when its uniform draw u[b] < p_reset (the pages use p = 0.1),
    else from the passed state.  h [Bz, ...] and conv_state [Bz, ...] (or
    None); returns new copies."""
    u = _f64(u)
    keep = (u >= p_reset).astype(np.float64)
    h = _f64(h)
    h2 = h * keep.reshape((-1,) + (1,) * (h.ndim - 1))
    c2 = None
    if conv_state is not None:
        c = _f64(conv_state)
        c2 = c * keep.reshape((-1,) + (1,) * (c.ndim - 1))
    return h2, c2


def fitted_noise_update(hT, mu=None, var=None, beta: float = 0.1):
    """Fitted noise, Eqs. (5)-(6) (section 4.2): per head, the mean and the
    variance of the final states over the batch, the channels P and the state
    size N, mixed into the running values with weight 1 - beta on the new
    statistic and beta on the history (beta = 0.1: the new statistic weighs
    0.9).  Without a history (mu, var None) the batch statistics are taken
    as they are.  hT [Bz, H, P, N]; returns (mu [H], var [H])."""
    hT = _f64(hT)
    H = hT.shape[1]
    flat = np.moveaxis(hT, 1, 0).reshape(H, -1)
    m = flat.mean(axis=1)
    v = ((flat - m[:, None]) ** 2).mean(axis=1)          # population variance
    if mu is None:
        return m, v
    return (1.0 - beta) * m + beta * _f64(mu), (1.0 - beta) * v + beta * _f64(var)


def fitted_noise_sample(mu, var, eps):
    """Initial states drawn independently per element from the fitted
    per-head Gaussian: h0 = mu_h + sqrt(var_h) eps with eps ~ N(0, 1) given,
    eps [Bz, H, P, N]."""
    mu, var, eps = _f64(mu), _f64(var), _f64(eps)
    return mu[None, :, None, None] + np.sqrt(var)[None, :, None, None] * eps


def state_std_trace(u, dt, A, B, C, h0, stride: int):
    """The state-scale diagnostic of section 3.5 (Figs. 4 and 9): the standard
    deviation, over a head's P x N state elements, of h_t after tokens
    t = stride - 1, 2 stride - 1, ... and after the last token, for every
    batch row and head.  Runs the recurrence token by token (small sizes).
    Returns [Bz, ceil(L / stride), H]."""
    dt, A, B, C = _f64(dt), _f64(A), _f64(B), _f64(C)
    Bz, L, H = dt.shape
    G, N = B.shape[2], B.shape[3]
    u = _f64(u)
    P = u.shape[3] if u.ndim == 4 else u.shape[2] // H
    u = u.reshape(Bz, L, H, P)
    g_of_h = np.arange(H) // (H // G)
    h = np.zeros((Bz, H, P, N)) if h0 is None else _f64(h0).copy()
    out = np.zeros((Bz, -(-L // stride), H))
    for t in range(L):
        a = np.exp(dt[:, t, :] * A[None, :])                       # [Bz, H]
        Bt = B[:, t, g_of_h, :]                                     # [Bz, H, N]
        h = a[:, :, None, None] * h + u[:, t, :, :, None] * Bt[:, :, None, :]
        if (t + 1) % stride == 0 or t == L - 1:
            out[:, t // stride, :] = h.reshape(Bz, H, -1).std(axis=2)
    return out


def prefill_to_pool(x, state_in, K, hT, conv_pool, ssm_pool, cache_seqlens, conv_state_indices):
    """The state a prompt leaves, written into pool rows (the causal-conv
    chapter's "continuous batching" and "circular mode" sections): for
    request b, pool row r = conv_state_indices[b] (b when None) receives the
    newest S_len entries of the extended sequence u = [state_in, x] (zeros
    where u has none), laid out as the decode update reads them - circular
    mode (cache_seqlens given, p = cache_seqlens[b] the length after the
    prompt, the prompt at logical positions p - L .. p - 1): position q in
    slot q mod S_len; non-circular (cache_seqlens None): oldest first - and
    ssm_pool[r] = hT[b].  Rows with r outside [0, pool) or p < 0 are skipped.
    x [Bz, L, D], state_in [Bz, D, K-1] | None, hT [Bz, H, P, N] | None.
    Returns new copies of the two pools and the number of skipped rows."""
    x = _f64(x)
    Bz, L, D = x.shape
    cp = _f64(conv_pool).copy()
    sp = _f64(ssm_pool).copy() if ssm_pool is not None else None
    pool, _, S_len = cp.shape
    S = np.zeros((Bz, D, K - 1)) if state_in is None else _f64(state_in)
    sl = None if cache_seqlens is None else np.asarray(getattr(cache_seqlens, "data", cache_seqlens))
    ix = None if conv_state_indices is None else np.asarray(
        getattr(conv_state_indices, "data", conv_state_indices))
    bad = 0
    for b in range(Bz):
        r = int(ix[b]) if ix is not None else b
        p = int(sl[b]) if sl is not None else L
        if r < 0 or r >= pool or p < 0:
            bad += 1
            continue
        u = np.concatenate([S[b], x[b].T], axis=1)           # [D, K-1+L], u[:, i] at position p-L-(K-1)+i
        first = p - L - (K - 1)
        for j in range(S_len):
            q = p - S_len + j                                 # the j-th oldest of the newest S_len positions
            i = q - first
            v = u[:, i] if 0 <= i < u.shape[1] else np.zeros(D)
            slot = (q % S_len) if sl is not None else j
            cp[r, :, slot] = v
        if sp is not None and hT is not None:
            sp[r] = _f64(hT)[b]
    return cp, sp, bad


def conv_state_fwd_packed(x, w, bias, S, seq_idx, apply_silu: bool = True):
    """The conv with state over rows that pack several samples ("Chapter 7:
    state, chunking and incremental inference", section "packed sequence
    boundaries"): tap k of token t reads extended-sequence entry u_{t+k} only
    when that entry's sequence id equals token t's (identity equality, as
    the page states: a reused id is not recognised as a reset).  The state
    entries (positions < 0) carry token 0's id: a call continues the sample
    its first token belongs to.  F = u[L : L+K-1] as without ids.
    x [Bz, L, D], w [D, K], bias [D] | None, S [Bz, D, K-1] | None,
    seq_idx [Bz, L] int.  Returns (out [Bz, L, D], F [Bz, D, K-1])."""
    x, w = _f64(x), _f64(w)
    Bz, L, D = x.shape
    K = w.shape[1]
    bias = np.zeros(D) if bias is None else _f64(bias)
    S = np.zeros((Bz, D, K - 1)) if S is None else _f64(S)
    ids = np.asarray(getattr(seq_idx, "data", seq_idx)).astype(np.int64)
    out = np.empty((Bz, L, D))
    F = np.empty((Bz, D, K - 1))
    for b in range(Bz):
        u = np.concatenate([S[b], x[b].T], axis=1)              # [D, K-1+L]
        uid = np.concatenate([np.full(K - 1, ids[b, 0] if L else 0), ids[b]])
        for t in range(L):
            z = bias.copy()
            for k in range(K):
                if uid[t + k] == ids[b, t]:
                    z += w[:, k] * u[:, t + k]
            out[b, t] = z / (1.0 + np.exp(-z)) if apply_silu else z
        F[b] = u[:, L:L + K - 1]
    return out, F


def ssm_scan_packed(u, dt, A, B, C, h0, seq_idx):
    """The scan over rows packing several samples: at a token whose sequence
    id differs from the previous token's the state restarts from zero (no
    history crosses a sample boundary, the state counterpart of the conv's
    packed-boundary rule); the first token continues from h0.  Token by token.
    Returns (y [Bz, L, H, P], hT)."""
    dt, A, B, C = _f64(dt), _f64(A), _f64(B), _f64(C)
    Bz, L, H = dt.shape
    G, N = B.shape[2], B.shape[3]
    u = _f64(u)
    P = u.shape[3] if u.ndim == 4 else u.shape[2] // H
    u = u.reshape(Bz, L, H, P)
    ids = np.asarray(getattr(seq_idx, "data", seq_idx)).astype(np.int64)
    g_of_h = np.arange(H) // (H // G)
    h = np.zeros((Bz, H, P, N)) if h0 is None else _f64(h0).copy()
    y = np.zeros((Bz, L, H, P))
    for t in range(L):
        a = np.exp(dt[:, t, :] * A[None, :])
        if t > 0:
            a = np.where((ids[:, t] != ids[:, t - 1])[:, None], 0.0, a)
        Bt = B[:, t, g_of_h, :]
        Ct = C[:, t, g_of_h, :]
        h = a[:, :, None, None] * h + u[:, t, :, :, None] * Bt[:, :, None, :]
        y[:, t] = np.einsum("bhpn,bhn->bhp", h, Ct)
    return y, h


def mixer_fwd_packed(x, dt, A, B, C, w, bias, conv_state, h0, seq_idx):
    """One segment of the forward over packed rows: the packed conv, then the
    packed scan."""
    u, F = conv_state_fwd_packed(x, w, bias, conv_state, seq_idx, True)
    y, hT = ssm_scan_packed(u, dt, A, B, C, h0, seq_idx)
    return y, F, hT
