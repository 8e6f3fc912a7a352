"""The C-ABI library loads and exports every entry point its header declares;
host-side argument checks answer without touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sss.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    path = __graft_entry__._build_module().build()
    return ctypes.CDLL(path)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sss_[a-z_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("sss_conv_state_fwd", "sss_ssm_scan_fwd", "sss_mixer_update",
                     "sss_device_status"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"not exported: {missing}"


def test_version_and_status_strings(lib):
    lib.sss_version.restype = ctypes.c_int
    assert lib.sss_version() >= 100
    lib.sss_status_string.restype = ctypes.c_char_p
    assert lib.sss_status_string(0) == b"ok"
    assert b"index" in lib.sss_status_string(4)


def test_invalid_arguments_rejected_before_launch(lib):
    i64 = ctypes.c_int64
    f = lib.sss_conv_state_fwd
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, i64, i64, i64,
                  ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    assert f(None, 0, None, None, None, None, None, 0, 1, 4, 8, 0, 1, None) == 1   # K < 1
    assert f(None, 0, None, None, None, None, None, 0, 1, 4, 8, 4, 1, None) == 1   # null w/x/u
    assert f(None, 7, None, None, None, None, None, 0, 1, 4, 8, 4, 1, None) == 1   # bad dtype
    assert f(None, 0, None, None, None, None, None, 0, 1, 4, 8, 9, 1, None) == 2   # K > 8
    assert f(None, 0, None, None, None, None, None, 0, 0, 4, 8, 4, 1, None) == 0   # empty batch
    g = lib.sss_ssm_scan_fwd
    g.restype = ctypes.c_int
    g.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, i64, i64, ctypes.c_int,
                  ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
                  ctypes.c_void_p]
    assert g(None, 0, None, None, None, None, 0, None, None, None, 0, 1, 8, 3, 4, 8, 2, None, 0,
             None) == 1  # H % G != 0
    assert g(None, 0, None, None, None, None, 0, None, None, None, 0, 1, 8, 2, 4, 8, 1, None, 0,
             None) == 1  # null A
    h = lib.sss_mixer_update
    h.restype = ctypes.c_int
    h.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_void_p, i64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p, i64, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    # S_len < K-1
    assert h(None, 1, None, None, None, 4, 2, None, None, None, None, None, None, None, None, 2,
             1, 2, 4, 8, 1, 4, None) == 1
    # L_new above the supported maximum
    assert h(None, 1, None, None, None, 4, 4, None, None, None, None, None, None, None, None, 2,
             65, 2, 4, 8, 1, 4, None) == 2


def test_scan_path_selection(lib):
    lib.sss_ssm_scan_path.restype = ctypes.c_int
    lib.sss_ssm_scan_path.argtypes = [ctypes.c_int64, ctypes.c_int64] + [ctypes.c_int] * 7
    assert lib.sss_ssm_scan_path(1, 64, 2, 4, 8, 1, 0, 0, 0) == 0      # fp32 -> CUDA cores
    assert lib.sss_ssm_scan_path(1, 64, 2, 4, 1000, 1, 0, 0, 0) == -1  # N too large


def test_conv_backward_host_checks(lib):
    """Workspace size and argument checks of the conv backward (each case
    returns before any launch)."""
    i64 = ctypes.c_int64
    ws = lib.sss_conv_state_bwd_workspace_size
    ws.restype = ctypes.c_size_t
    ws.argtypes = [i64, i64, i64, ctypes.c_int]
    # one row of D * (K+1) fp32 partial sums per sequence and token group:
    # 256 tokens for K = 4 (the channel-pair walk's CTA rows), 512 otherwise
    assert ws(8, 1024, 2048, 4) == 8 * 4 * 2048 * 5 * 4
    assert ws(2, 257, 64, 4) == 2 * 2 * 64 * 5 * 4
    assert ws(2, 513, 10, 3) == 2 * 2 * 10 * 4 * 4
    assert ws(2, 0, 10, 3) == 0
    f = lib.sss_conv_state_bwd
    f.restype = ctypes.c_int
    P = ctypes.c_void_p
    f.argtypes = [P, ctypes.c_int, P, P, P, P, ctypes.c_int, P, P, ctypes.c_int, P, P, P,
                  i64, i64, i64, ctypes.c_int, ctypes.c_int, P, ctypes.c_size_t, P]
    a = lambda k: ctypes.c_void_p(0x10000000 * k)  # aligned stand-ins, never dereferenced
    args = lambda **kw: dict(dict(x=a(1), xt=1, w=a(2), b=a(3), s=a(4), dy=a(5), dyt=0, q=a(6),
                                  dx=a(7), dxt=1, ds=a(8), dw=a(9), db=a(10), Bz=2, L=100, D=64,
                                  K=4, silu=1, ws=a(11), wsb=ws(2, 100, 64, 4), st=None), **kw)
    call = lambda d: f(*d.values())
    assert call(args(K=9)) == 2                      # K > 8
    assert call(args(K=0)) == 1                      # K < 1
    assert call(args(dyt=5)) == 1                    # unknown dtype
    assert call(args(wsb=16)) == 1                   # workspace too small
    assert call(args(ws=None)) == 1                  # no workspace
    assert call(args(ds=a(6))) == 1                  # dS would overwrite dF
    assert call(args(dw=None)) == 1                  # no weight gradient buffer
    assert call(args(Bz=0)) == 0                     # empty batch: nothing to do


def test_scan_backward_host_checks(lib):
    """Workspace size and argument checks of the scan backward (each case
    returns before any launch)."""
    i64, ci = ctypes.c_int64, ctypes.c_int
    ws = lib.sss_ssm_scan_bwd_workspace_size
    ws.restype = ctypes.c_size_t
    ws.argtypes = [i64, i64, ci, ci, ci, ci]
    al = lambda v: (v + 255) // 256 * 256
    # chunk-entry states (one more than the 64-token chunks), chunk-end state
    # gradients, per-head dB and dC shares and per-chunk dA shares, fp32
    Bz, L, H, P, N = 2, 130, 4, 64, 128
    nC = 3
    expect = (al(4 * Bz * H * (nC + 1) * P * N) + al(4 * Bz * H * nC * P * N)
              + 2 * al(4 * Bz * L * H * N) + al(4 * Bz * H * nC))
    assert ws(Bz, L, H, P, N, 1) == expect
    f = lib.sss_ssm_scan_bwd
    f.restype = ci
    Pp = ctypes.c_void_p
    f.argtypes = [Pp, ci, Pp, Pp, Pp, Pp, ci, Pp, Pp, Pp, Pp, Pp, Pp, Pp, Pp, Pp,
                  i64, i64, ci, ci, ci, ci, Pp, ctypes.c_size_t, Pp]
    a = lambda k: ctypes.c_void_p(0x10000000 * k)  # aligned stand-ins, never dereferenced
    args = lambda **kw: dict(dict(x=a(1), xt=1, dt=a(2), A=a(3), B=a(4), C=a(5), at=1, h0=a(6),
                                  dy=a(7), dhT=a(8), dx=a(9), ddt=a(10), dA=a(11), dB=a(12),
                                  dC=a(13), dh0=a(14), Bz=Bz, L=L, H=H, P=P, N=N, G=1,
                                  ws=a(15), wsb=expect, st=None), **kw)
    call = lambda d: f(*d.values())
    assert call(args(P=65)) == 2                     # P > 64
    assert call(args(N=129)) == 2                    # N > 128
    assert call(args(G=3)) == 1                      # H not a multiple of G
    assert call(args(xt=7)) == 1                     # unknown dtype
    assert call(args(wsb=expect - 1)) == 1           # workspace too small
    assert call(args(ws=None)) == 1                  # no workspace
    assert call(args(dB=None)) == 1                  # no dB buffer
    assert call(args(dh0=ctypes.c_void_p(0x80000000 + 64))) == 1  # dh0 half over dhT
    assert call(args(dy=ctypes.c_void_p(0x70000002))) == 1        # misaligned dy


def test_span_forward_host_checks(lib):
    """Workspace size and the argument checks of the span-parallel forward that
    return before any launch or device query."""
    i64, ci = ctypes.c_int64, ctypes.c_int
    ws = lib.sss_fwd_spans_workspace_size
    ws.restype = ctypes.c_size_t
    ws.argtypes = [i64, i64, ci, ci, ci, ci, ci]
    al = lambda v: (v + 255) // 256 * 256
    # partial decay sums per 64-token piece of each span, the spans'
    # zero-start final states and initial states (fp32), their conv states
    # (bf16, K - 1 per channel)
    Bz, L, H, P, N, K, ns = 2, 1024, 48, 64, 128, 4, 4
    Ls = L // ns
    expect = (al(4 * Bz * ns * (Ls // 64) * H) + 2 * al(4 * Bz * ns * H * P * N)
              + al(2 * Bz * ns * H * P * (K - 1)))
    assert ws(Bz, L, H, P, N, K, ns) == expect
    assert ws(Bz, L, H, P, N, 1, ns) == expect - al(2 * Bz * ns * H * P * (K - 1))  # scan alone
    assert ws(Bz, 1000, H, P, N, K, 5) == (al(4 * Bz * 5 * 4 * H) + 2 * al(4 * Bz * 5 * H * P * N)
                                           + al(2 * Bz * 5 * H * P * (K - 1)))  # 200-token spans: 4 pieces
    assert ws(Bz, L, H, P, N, K, 1) == 0 and ws(Bz, L, H, P, N, K, 33) == 0
    f = lib.sss_mixer_fwd_spans
    f.restype = ci
    Pp = ctypes.c_void_p
    f.argtypes = [Pp, ci, Pp, Pp, Pp, Pp, Pp, Pp, Pp, Pp, Pp, Pp, Pp, ci, i64, i64, ci, ci, ci,
                  ci, ci, ci, Pp, ctypes.c_size_t, Pp]
    a = lambda k: ctypes.c_void_p(0x10000000 * k)  # aligned stand-ins, never dereferenced
    args = lambda **kw: dict(dict(x=a(1), xt=1, w=a(2), bias=a(3), s_in=a(4), s_out=a(4), dt=a(5),
                                  A=a(6), B=a(7), C=a(8), h0=a(9), hT=a(9), y=a(10), yt=1, Bz=Bz,
                                  L=L, H=H, P=P, N=N, G=1, K=K, ns=ns, ws=a(11), wsb=expect,
                                  st=None), **kw)
    call = lambda d: f(*d.values())
    assert call(args(ns=0)) == 1                     # no spans
    assert call(args(ns=33)) == 1                    # more spans than warp lanes
    assert call(args(L=1023)) == 1                   # L not a multiple of ns
    assert call(args(L=8, ns=4)) == 1                # 2-token spans < K - 1
    assert call(args(xt=7)) == 1                     # unknown dtype
    assert call(args(G=5)) == 1                      # H not a multiple of G


def test_mamba2_forward_host_checks(lib):
    """Workspace size and the argument checks of the full Mamba-2 forward that
    return before any launch."""
    i64, ci, Pp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
    ws = lib.sss_mamba2_mixer_fwd_workspace_size
    ws.restype = ctypes.c_size_t
    ws.argtypes = [i64, i64, ci, ci, ci, ci]
    Bz, L, H, P, N, G, K = 2, 100, 4, 16, 32, 2, 4
    # the fp32 conv output of every xBC channel
    assert ws(Bz, L, H, P, N, G) == 4 * Bz * L * (H * P + 2 * G * N)
    assert ws(Bz, 0, H, P, N, G) == 0
    f = lib.sss_mamba2_mixer_fwd
    f.restype = ci
    f.argtypes = [Pp, Pp, ci, Pp, Pp, Pp, Pp, Pp, Pp, Pp, Pp, Pp, Pp, Pp, ci, i64, i64, ci, ci,
                  ci, ci, ci, Pp, ctypes.c_size_t, Pp]
    a = lambda k: ctypes.c_void_p(0x10000000 * k)  # aligned stand-ins, never dereferenced
    need = ws(Bz, L, H, P, N, G)
    base = dict(xBC=a(1), z=a(2), at=1, dtr=a(3), dtb=a(4), A=a(5), Dsk=a(6), w=a(7), b=a(8),
                s_in=a(9), s_out=a(9), h0=a(10), hT=a(10), y=a(11), yt=1, Bz=Bz, L=L, H=H, P=P,
                N=N, G=G, K=K, ws=a(12), wsb=need, st=None)
    call = lambda **kw: f(*dict(base, **kw).values())
    INVALID, UNSUPPORTED = 1, 2
    assert call(xBC=None) == INVALID                 # tokens but no input
    assert call(A=None) == INVALID
    assert call(ws=None) == INVALID                  # no workspace
    assert call(wsb=need - 4) == INVALID             # workspace too small
    assert call(at=7) == INVALID                     # unknown dtype
    assert call(H=3) == INVALID                      # H not a multiple of G
    assert call(K=9) == UNSUPPORTED                  # conv wider than 8
    assert call(P=200) == UNSUPPORTED                # head dim beyond the scan's
    assert call(Bz=0) == 0                           # nothing to do
