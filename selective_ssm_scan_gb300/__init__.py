"""Python binding of libsss (ctypes): the state-passing mixer forward and the
decode update on GB300.

Argument marshalling only: every step runs in the CUDA kernels of libsss.
Tensors are torch CUDA tensors (torch supplies device memory and streams);
calls are enqueued on torch's current stream.  Importing this module loads
``_build/libsss.so`` and raises if it is missing (build it with
``python selective_ssm_scan_gb300/build.py``); there is no fallback.

Functions (same names as the C ABI in include/sss.h, minus the prefix):
    conv_state_fwd, conv_state_bwd, conv_state_bwd_workspace_size,
    conv_state_bwd_noalloc, ssm_scan_fwd,
    ssm_scan_path, ssm_scan_workspace_size, mixer_update_path,
    mixer_update, device_status, version, status_string
plus ``mixer_fwd`` (conv_state_fwd then ssm_scan_fwd: one segment of the
streaming forward with both states passed) and ``library_path``.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "_build", "libsss.so")

SSS_OK = 0
SSS_ERR_INVALID_ARG = 1
SSS_ERR_UNSUPPORTED = 2
SSS_ERR_INDEX = 4
SSS_ERR_TIMEOUT = 8
SSS_ERR_CUDA = 16
SSS_F32 = 0
SSS_BF16 = 1

if not os.path.exists(library_path):
    raise ImportError(
        f"libsss.so not found at {library_path}; build it with "
        "`python selective_ssm_scan_gb300/build.py` (needs nvcc)")

_lib = ctypes.CDLL(library_path)
_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_i = ctypes.c_int

_lib.sss_version.restype = _i
_lib.sss_status_string.restype = ctypes.c_char_p
_lib.sss_status_string.argtypes = [_i]
_lib.sss_last_cuda_error.restype = ctypes.c_char_p
_lib.sss_conv_state_fwd.restype = _i
_lib.sss_conv_state_fwd.argtypes = [_p, _i, _p, _p, _p, _p, _p, _i, _i64, _i64, _i64, _i, _i, _p]
_lib.sss_conv_state_bwd_workspace_size.restype = ctypes.c_size_t
_lib.sss_conv_state_bwd_workspace_size.argtypes = [_i64, _i64, _i64, _i]
_lib.sss_conv_state_bwd.restype = _i
_lib.sss_conv_state_bwd.argtypes = [_p, _i, _p, _p, _p, _p, _i, _p, _p, _i, _p, _p, _p,
                                    _i64, _i64, _i64, _i, _i, _p, ctypes.c_size_t, _p]
_lib.sss_conv_state_bwd_noalloc.restype = _i
_lib.sss_conv_state_bwd_noalloc.argtypes = [_p, _i, _p, _p, _p, _p, _i, _p, _p, _i, _p, _p, _p,
                                            _i64, _i64, _i64, _i, _i, _p]
_lib.sss_ssm_scan_workspace_size.restype = ctypes.c_size_t
_lib.sss_ssm_scan_workspace_size.argtypes = [_i64, _i64, _i, _i, _i, _i, _i, _i]
_lib.sss_mixer_update_path.restype = _i
_lib.sss_mixer_update_path.argtypes = [_i, _i, _i, _i, _i, _i]
_lib.sss_ssm_scan_path.restype = _i
_lib.sss_ssm_scan_path.argtypes = [_i64, _i64, _i, _i, _i, _i, _i, _i, _i]
_lib.sss_ssm_scan_fwd.restype = _i
_lib.sss_ssm_scan_fwd.argtypes = [_p, _i, _p, _p, _p, _p, _i, _p, _p, _p, _i, _i64, _i64, _i, _i,
                                  _i, _i, _p, ctypes.c_size_t, _p]
_lib.sss_ssm_scan_bwd_workspace_size.restype = ctypes.c_size_t
_lib.sss_ssm_scan_bwd_workspace_size.argtypes = [_i64, _i64, _i, _i, _i, _i]
_lib.sss_ssm_scan_bwd.restype = _i
_lib.sss_ssm_scan_bwd.argtypes = [_p, _i, _p, _p, _p, _p, _i, _p, _p, _p, _p, _p, _p, _p, _p, _p,
                                  _i64, _i64, _i, _i, _i, _i, _p, ctypes.c_size_t, _p]
_lib.sss_ssm_scan_fwd_packed.restype = _i
_lib.sss_ssm_scan_fwd_packed.argtypes = [_p, _i, _p, _p, _p, _p, _i, _p, _p, _p, _p, _i, _i64, _i64,
                                         _i, _i, _i, _i, _p]
_lib.sss_mixer_fwd_packed.restype = _i
_lib.sss_mixer_fwd_packed.argtypes = [_p, _i, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _i,
                                      _i64, _i64, _i, _i, _i, _i, _i, _p]
_lib.sss_conv_state_fwd_packed.restype = _i
_lib.sss_conv_state_fwd_packed.argtypes = [_p, _i, _p, _p, _p, _p, _p, _p, _i, _i64, _i64, _i64,
                                           _i, _i, _p]
_lib.sss_prefill_to_pool.restype = _i
_lib.sss_prefill_to_pool.argtypes = [_p, _i, _p, _i, _p, _p, _i64, _i, _p, _p, _p, _i64, _i64,
                                     _i64, _i, _i, _i, _p]
_lib.sss_state_reset.restype = _i
_lib.sss_state_reset.argtypes = [_p, ctypes.c_float, _p, _i64, _i64, _p, _i, _i64, _p]
_lib.sss_fitted_noise_update.restype = _i
_lib.sss_fitted_noise_update.argtypes = [_p, _i64, _i, _i, _i, ctypes.c_float, _i, _p, _p, _p]
_lib.sss_fitted_noise_sample.restype = _i
_lib.sss_fitted_noise_sample.argtypes = [_p, _p, _p, _p, _i64, _i, _i, _i, _p]
_lib.sss_state_std_trace.restype = _i
_lib.sss_state_std_trace.argtypes = [_p, _i, _p, _p, _p, _i, _p, _p, _i64, _i64, _i, _i, _i, _i,
                                     _i, _p]
_lib.sss_mixer_update.restype = _i
_lib.sss_mixer_update.argtypes = [_p, _i, _p, _p, _p, _i64, _i, _p, _p, _p, _p, _p, _p, _p, _p,
                                  _i64, _i, _i, _i, _i, _i, _i, _p]
_lib.sss_mixer_fwd_supported.restype = _i
_lib.sss_mixer_fwd_supported.argtypes = [_i64, _i64, _i, _i, _i, _i, _i, _i, _i]
_lib.sss_mamba2_mixer_fwd_workspace_size.restype = ctypes.c_size_t
_lib.sss_mamba2_mixer_fwd_workspace_size.argtypes = [_i64, _i64, _i, _i, _i, _i]
_lib.sss_mamba2_mixer_fwd.restype = _i
_lib.sss_mamba2_mixer_fwd.argtypes = [_p, _p, _i, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _i,
                                      _i64, _i64, _i, _i, _i, _i, _i, _p, ctypes.c_size_t, _p]
_lib.sss_mixer_fwd.restype = _i
_lib.sss_mixer_fwd.argtypes = [_p, _i, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _i, _i64, _i64,
                               _i, _i, _i, _i, _i, _p]
_lib.sss_mixer_fwd_span_count.restype = _i
_lib.sss_mixer_fwd_span_count.argtypes = [_i64, _i64, _i, _i, _i, _i, _i, _i, _i]
_lib.sss_ssm_scan_fwd_span_count.restype = _i
_lib.sss_ssm_scan_fwd_span_count.argtypes = [_i64, _i64, _i, _i, _i, _i, _i, _i, _i]
_lib.sss_fwd_spans_workspace_size.restype = ctypes.c_size_t
_lib.sss_fwd_spans_workspace_size.argtypes = [_i64, _i64, _i, _i, _i, _i, _i]
_lib.sss_mixer_fwd_spans.restype = _i
_lib.sss_mixer_fwd_spans.argtypes = [_p, _i, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _i, _i64,
                                     _i64, _i, _i, _i, _i, _i, _i, _p, ctypes.c_size_t, _p]
_lib.sss_ssm_scan_fwd_spans.restype = _i
_lib.sss_ssm_scan_fwd_spans.argtypes = [_p, _i, _p, _p, _p, _p, _i, _p, _p, _p, _i, _i64, _i64,
                                        _i, _i, _i, _i, _i, _p, ctypes.c_size_t, _p]
_lib.sss_device_status.restype = _i
_lib.sss_device_status.argtypes = [ctypes.POINTER(_i), _i, _p]


class SSSError(RuntimeError):
    def __init__(self, fn: str, status: int):
        msg = f"{fn}: {status_string(status)} (status {status})"
        if status & SSS_ERR_CUDA:
            msg += f": {_lib.sss_last_cuda_error().decode()}"
        super().__init__(msg)
        self.status = status


def version() -> int:
    return int(_lib.sss_version())


def status_string(s: int) -> str:
    return _lib.sss_status_string(int(s)).decode()


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SSS_F32
    if t.dtype == torch.bfloat16:
        return SSS_BF16
    raise TypeError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")


def _dtype_code(d) -> int:
    return _dt(torch.empty(0, dtype=d)) if isinstance(d, torch.dtype) else int(d)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr() if t.numel() else None


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream if hasattr(s, "cuda_stream") else int(s)


def _check(fn: str, rc: int):
    if rc != SSS_OK:
        raise SSSError(fn, rc)


def conv_state_fwd(x: torch.Tensor, w: torch.Tensor, bias: Optional[torch.Tensor] = None,
                   state_in: Optional[torch.Tensor] = None,
                   state_out: Optional[torch.Tensor] = None, u: Optional[torch.Tensor] = None,
                   u_dtype=torch.float32, apply_silu: bool = True, stream=None) -> torch.Tensor:
    """x [Bz, L, D]; w [D, K] fp32; bias [D] fp32; state_in/state_out [Bz, D, K-1]
    (x's dtype, may be the same tensor).  Returns u [Bz, L, D]."""
    Bz, L, D = x.shape
    K = w.shape[1]
    if u is None:
        u = torch.empty((Bz, L, D), dtype=u_dtype, device=x.device)
    rc = _lib.sss_conv_state_fwd(_ptr(x), _dt(x), _ptr(w), _ptr(bias), _ptr(state_in),
                                 _ptr(state_out), _ptr(u), _dt(u), Bz, L, D, K,
                                 int(bool(apply_silu)), _stream(stream))
    _check("sss_conv_state_fwd", rc)
    return u


def conv_state_bwd_workspace_size(Bz, L, D, K) -> int:
    return int(_lib.sss_conv_state_bwd_workspace_size(Bz, L, D, K))


def conv_state_bwd(x: torch.Tensor, w: torch.Tensor, bias: Optional[torch.Tensor],
                   state_in: Optional[torch.Tensor], dy: torch.Tensor,
                   dstate_out: Optional[torch.Tensor] = None, dx: Optional[torch.Tensor] = None,
                   dstate_in: Optional[torch.Tensor] = None, dw: Optional[torch.Tensor] = None,
                   dbias: Optional[torch.Tensor] = None, dx_dtype=None, apply_silu: bool = True,
                   workspace: Optional[torch.Tensor] = None, stream=None):
    """Gradient of conv_state_fwd.  dy = dL/du [Bz, L, D]; dstate_out = dL/dF
    [Bz, D, K-1] (dy's dtype) or None.  Returns (dx [Bz, L, D], dstate_in
    [Bz, D, K-1] (dx's dtype), dw [D, K] fp32, dbias [D] fp32)."""
    Bz, L, D = x.shape
    K = w.shape[1]
    dev = x.device
    dx_dtype = dx_dtype or x.dtype
    if dx is None:
        dx = torch.empty((Bz, L, D), dtype=dx_dtype, device=dev)
    if dstate_in is None:
        dstate_in = torch.empty((Bz, D, K - 1), dtype=dx.dtype, device=dev)
    if dw is None:
        dw = torch.empty((D, K), dtype=torch.float32, device=dev)
    if dbias is None:
        dbias = torch.empty((D,), dtype=torch.float32, device=dev)
    need = conv_state_bwd_workspace_size(Bz, L, D, K)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = _lib.sss_conv_state_bwd(_ptr(x), _dt(x), _ptr(w), _ptr(bias), _ptr(state_in), _ptr(dy),
                                 _dt(dy), _ptr(dstate_out), _ptr(dx), _dt(dx), _ptr(dstate_in),
                                 _ptr(dw), _ptr(dbias), Bz, L, D, K, int(bool(apply_silu)),
                                 _ptr(workspace), ws_bytes, _stream(stream))
    _check("sss_conv_state_bwd", rc)
    return dx, dstate_in, dw, dbias


# Size of the library's static scratch behind conv_state_bwd_noalloc (the
# SSS_CONV_BWD_NOALLOC_SCRATCH_BYTES of the C header), read from the library.
_lib.sss_conv_state_bwd_noalloc_scratch_bytes.restype = ctypes.c_size_t
_lib.sss_conv_state_bwd_noalloc_scratch_bytes.argtypes = []
CONV_BWD_NOALLOC_SCRATCH_BYTES = int(_lib.sss_conv_state_bwd_noalloc_scratch_bytes())


def conv_state_bwd_noalloc(x: torch.Tensor, w: torch.Tensor, bias: Optional[torch.Tensor],
                           state_in: Optional[torch.Tensor], dy: torch.Tensor,
                           dstate_out: Optional[torch.Tensor], dx: torch.Tensor,
                           dstate_in: torch.Tensor, dw: torch.Tensor,
                           dbias: Optional[torch.Tensor] = None, apply_silu: bool = True,
                           stream=None):
    """conv_state_bwd for callers that cannot allocate device memory: every
    output is passed in, and the partial sums go to the library's static
    scratch of CONV_BWD_NOALLOC_SCRATCH_BYTES bytes (calls needing more raise
    with SSS_ERR_UNSUPPORTED).  Calls that may run at the same time on the
    GPU share that scratch and race; issue them on one stream.  Returns
    (dx, dstate_in, dw, dbias)."""
    Bz, L, D = x.shape
    K = w.shape[1]
    rc = _lib.sss_conv_state_bwd_noalloc(_ptr(x), _dt(x), _ptr(w), _ptr(bias), _ptr(state_in),
                                         _ptr(dy), _dt(dy), _ptr(dstate_out), _ptr(dx), _dt(dx),
                                         _ptr(dstate_in), _ptr(dw), _ptr(dbias), Bz, L, D, K,
                                         int(bool(apply_silu)), _stream(stream))
    _check("sss_conv_state_bwd_noalloc", rc)
    return dx, dstate_in, dw, dbias


def ssm_scan_workspace_size(Bz, L, H, P, N, G, x_dtype, act_dtype) -> int:
    return int(_lib.sss_ssm_scan_workspace_size(Bz, L, H, P, N, G, _dtype_code(x_dtype),
                                                _dtype_code(act_dtype)))


def _nbytes(t: Optional[torch.Tensor]) -> int:
    return t.numel() * t.element_size() if t is not None else 0


def fwd_spans_workspace_size(Bz, L, H, P, N, K, spans) -> int:
    return int(_lib.sss_fwd_spans_workspace_size(Bz, L, H, P, N, K, spans))


def _span_workspace(Bz, L, H, P, N, K, spans, workspace, dev):
    """The caller's workspace as given (the library checks its size and
    alignment), else a fresh one of the size the library asks for."""
    if workspace is None:
        need = fwd_spans_workspace_size(Bz, L, H, P, N, K, spans)
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    return workspace


def mixer_fwd_span_count(Bz, L, H, P, N, G, K, x_dtype, y_dtype) -> int:
    return int(_lib.sss_mixer_fwd_span_count(Bz, L, H, P, N, G, K, _dtype_code(x_dtype),
                                             _dtype_code(y_dtype)))


def ssm_scan_fwd_span_count(Bz, L, H, P, N, G, x_dtype, act_dtype, y_dtype) -> int:
    return int(_lib.sss_ssm_scan_fwd_span_count(Bz, L, H, P, N, G, _dtype_code(x_dtype),
                                                _dtype_code(act_dtype), _dtype_code(y_dtype)))


def ssm_scan_path(Bz, L, H, P, N, G, x_dtype, act_dtype, y_dtype) -> int:
    """1 = tcgen05 chunked scan, 0 = fp32 CUDA-core scan, -1 = unsupported."""
    return int(_lib.sss_ssm_scan_path(Bz, L, H, P, N, G, _dtype_code(x_dtype),
                                      _dtype_code(act_dtype), _dtype_code(y_dtype)))


def ssm_scan_fwd(x: torch.Tensor, dt: torch.Tensor, A: torch.Tensor, B: torch.Tensor,
                 C: torch.Tensor, h0: Optional[torch.Tensor] = None,
                 hT: Optional[torch.Tensor] = None, y: Optional[torch.Tensor] = None,
                 y_dtype=None, workspace: Optional[torch.Tensor] = None, stream=None,
                 spans: Optional[int] = None):
    """x [Bz, L, H, P] (or [Bz, L, D] with H taken from dt); dt [Bz, L, H];
    A [H] fp32; B, C [Bz, L, G, N]; h0/hT [Bz, H, P, N] fp32 (may be the same
    tensor).  Returns (y, hT).

    spans: the number of equal spans the sequence is cut into and run in
    parallel (sss_ssm_scan_fwd_spans); None = the library's choice for these
    sizes on this device, 1 = one pass."""
    Bz, L, H = dt.shape
    G, N = B.shape[2], B.shape[3]
    P = x.shape[-1] if x.dim() == 4 else x.shape[-1] // H
    dev = x.device
    if y is None:
        y = torch.empty((Bz, L, H, P), dtype=y_dtype or dt.dtype, device=dev)
    if hT is None:
        hT = torch.empty((Bz, H, P, N), dtype=torch.float32, device=dev)
    if spans is None:
        spans = int(_lib.sss_ssm_scan_fwd_span_count(Bz, L, H, P, N, G, _dt(x), _dt(dt), _dt(y)))
    if spans > 1:
        workspace = _span_workspace(Bz, L, H, P, N, 1, spans, workspace, dev)
        rc = _lib.sss_ssm_scan_fwd_spans(_ptr(x), _dt(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C),
                                         _dt(dt), _ptr(h0), _ptr(hT), _ptr(y), _dt(y), Bz, L, H,
                                         P, N, G, spans, _ptr(workspace), _nbytes(workspace),
                                         _stream(stream))
        _check("sss_ssm_scan_fwd_spans", rc)
        return y, hT
    ws = ssm_scan_workspace_size(Bz, L, H, P, N, G, x.dtype, dt.dtype)
    if ws and (workspace is None or workspace.numel() * workspace.element_size() < ws):
        workspace = torch.empty(ws, dtype=torch.uint8, device=dev)
    wsb = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = _lib.sss_ssm_scan_fwd(_ptr(x), _dt(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _dt(dt),
                               _ptr(h0), _ptr(hT), _ptr(y), _dt(y), Bz, L, H, P, N, G,
                               _ptr(workspace), wsb, _stream(stream))
    _check("sss_ssm_scan_fwd", rc)
    return y, hT


def ssm_scan_bwd_workspace_size(Bz, L, H, P, N, G) -> int:
    return int(_lib.sss_ssm_scan_bwd_workspace_size(Bz, L, H, P, N, G))


def ssm_scan_bwd(x: torch.Tensor, dt: torch.Tensor, A: torch.Tensor, B: torch.Tensor,
                 C: torch.Tensor, h0: Optional[torch.Tensor], dy: torch.Tensor,
                 dhT: Optional[torch.Tensor] = None, dh0: Optional[torch.Tensor] = None,
                 want_dh0: bool = True, workspace: Optional[torch.Tensor] = None, stream=None):
    """Gradient of ssm_scan_fwd.  dy [Bz, L, H, P] fp32, dhT [Bz, H, P, N] fp32
    or None.  Returns (dx [Bz, L, H, P], ddt [Bz, L, H], dA [H], dB and dC
    [Bz, L, G, N], dh0 [Bz, H, P, N] or None), all fp32."""
    Bz, L, H = dt.shape
    G, N = B.shape[2], B.shape[3]
    P = x.shape[-1] if x.dim() == 4 else x.shape[-1] // H
    dev = x.device
    f32 = torch.float32
    dx = torch.empty((Bz, L, H, P), dtype=f32, device=dev)
    ddt = torch.empty((Bz, L, H), dtype=f32, device=dev)
    dA = torch.empty((H,), dtype=f32, device=dev)
    dB = torch.empty((Bz, L, G, N), dtype=f32, device=dev)
    dC = torch.empty((Bz, L, G, N), dtype=f32, device=dev)
    if dh0 is None and want_dh0:
        dh0 = torch.empty((Bz, H, P, N), dtype=f32, device=dev)
    need = ssm_scan_bwd_workspace_size(Bz, L, H, P, N, G)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    wsb = workspace.numel() * workspace.element_size()
    rc = _lib.sss_ssm_scan_bwd(_ptr(x), _dt(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _dt(dt),
                               _ptr(h0), _ptr(dy), _ptr(dhT), _ptr(dx), _ptr(ddt), _ptr(dA),
                               _ptr(dB), _ptr(dC), _ptr(dh0), Bz, L, H, P, N, G,
                               _ptr(workspace), wsb, _stream(stream))
    _check("sss_ssm_scan_bwd", rc)
    return dx, ddt, dA, dB, dC, dh0


def ssm_scan_fwd_packed(x: torch.Tensor, dt: torch.Tensor, A: torch.Tensor, B: torch.Tensor,
                        C: torch.Tensor, h0: Optional[torch.Tensor], seq_idx: torch.Tensor,
                        hT: Optional[torch.Tensor] = None, y_dtype=None, stream=None):
    """ssm_scan_fwd over rows packing several samples: the state restarts at
    every change of seq_idx [Bz, L] int32.  Returns (y, hT)."""
    Bz, L, H = dt.shape
    G, N = B.shape[2], B.shape[3]
    P = x.shape[-1] if x.dim() == 4 else x.shape[-1] // H
    y = torch.empty((Bz, L, H, P), dtype=y_dtype or dt.dtype, device=x.device)
    if hT is None:
        hT = torch.empty((Bz, H, P, N), dtype=torch.float32, device=x.device)
    _check("sss_ssm_scan_fwd_packed", _lib.sss_ssm_scan_fwd_packed(
        _ptr(x), _dt(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _dt(dt), _ptr(h0), _ptr(hT),
        _ptr(seq_idx), _ptr(y), _dt(y), Bz, L, H, P, N, G, _stream(stream)))
    return y, hT


def mixer_fwd_packed(x: torch.Tensor, dt: torch.Tensor, A: torch.Tensor, B: torch.Tensor,
                     C: torch.Tensor, w: torch.Tensor, bias: Optional[torch.Tensor],
                     conv_state: Optional[torch.Tensor], h0: Optional[torch.Tensor],
                     seq_idx: torch.Tensor, y_dtype=None, stream=None):
    """mixer_fwd over rows packing several samples (seq_idx [Bz, L] int32):
    the conv's taps and the scan's state stop at sample boundaries.  Returns
    (y, F, hT)."""
    Bz, L, D = x.shape
    H = dt.shape[2]
    P = D // H
    G, N = B.shape[2], B.shape[3]
    K = w.shape[1]
    y = torch.empty((Bz, L, H, P), dtype=y_dtype or x.dtype, device=x.device)
    F = torch.empty((Bz, D, K - 1), dtype=x.dtype, device=x.device)
    hT = torch.empty((Bz, H, P, N), dtype=torch.float32, device=x.device)
    _check("sss_mixer_fwd_packed", _lib.sss_mixer_fwd_packed(
        _ptr(x), _dt(x), _ptr(w), _ptr(bias), _ptr(conv_state), _ptr(F), _ptr(dt), _ptr(A),
        _ptr(B), _ptr(C), _ptr(h0), _ptr(hT), _ptr(seq_idx), _ptr(y), _dt(y), Bz, L, H, P, N, G,
        K, _stream(stream)))
    return y, F, hT


def conv_state_fwd_packed(x: torch.Tensor, w: torch.Tensor, bias: Optional[torch.Tensor],
                          state_in: Optional[torch.Tensor], seq_idx: torch.Tensor,
                          state_out: Optional[torch.Tensor] = None, u: Optional[torch.Tensor] = None,
                          u_dtype=torch.float32, apply_silu: bool = True, stream=None):
    """conv_state_fwd over rows packing several samples: tap k of token t reads
    u_{t+k} only when seq_idx agrees (seq_idx [Bz, L] int32).  Returns (u, F)."""
    Bz, L, D = x.shape
    K = w.shape[1]
    if seq_idx.dtype != torch.int32:
        raise TypeError("seq_idx must be int32")
    if u is None:
        u = torch.empty((Bz, L, D), dtype=u_dtype, device=x.device)
    if state_out is None:
        state_out = torch.empty((Bz, D, K - 1), dtype=x.dtype, device=x.device)
    _check("sss_conv_state_fwd_packed", _lib.sss_conv_state_fwd_packed(
        _ptr(x), _dt(x), _ptr(w), _ptr(bias), _ptr(state_in), _ptr(state_out), _ptr(seq_idx),
        _ptr(u), _dt(u), Bz, L, D, K, int(bool(apply_silu)), _stream(stream)))
    return u, state_out


def prefill_to_pool(x: torch.Tensor, conv_state_in: Optional[torch.Tensor], K: int,
                    hT: Optional[torch.Tensor], conv_pool: torch.Tensor,
                    ssm_pool: Optional[torch.Tensor], cache_seqlens: Optional[torch.Tensor],
                    conv_state_indices: Optional[torch.Tensor], H: int, stream=None):
    """Write a prompt's conv history (the newest S_len inputs of [conv_state_in,
    x]) and its final SSM state hT into the pool rows conv_state_indices, in
    place: circular layout when cache_seqlens (the lengths after the prompt)
    is given, oldest first otherwise."""
    Bz, L, D = x.shape
    pool, _, S_len = conv_pool.shape
    P = D // H
    N = hT.shape[-1] if hT is not None else (ssm_pool.shape[-1] if ssm_pool is not None else 1)
    _check("sss_prefill_to_pool", _lib.sss_prefill_to_pool(
        _ptr(x), _dt(x), _ptr(conv_state_in), int(K), _ptr(hT), _ptr(conv_pool), pool, S_len,
        _ptr(ssm_pool), _ptr(cache_seqlens), _ptr(conv_state_indices), Bz, L, D, H, P, N,
        _stream(stream)))
    return conv_pool, ssm_pool


def state_reset(u: torch.Tensor, p_reset: float, h: Optional[torch.Tensor],
                conv_state: Optional[torch.Tensor] = None, stream=None):
    """Zero, in place, row b of h and of conv_state where u[b] < p_reset (u [Bz]
    fp32 uniforms); other rows are not touched."""
    Bz = u.shape[0]
    hr = h[0].numel() if h is not None and Bz else 0
    cr = conv_state[0].numel() if conv_state is not None and Bz else 0
    cdt = _dt(conv_state) if conv_state is not None else 0
    _check("sss_state_reset", _lib.sss_state_reset(_ptr(u), float(p_reset), _ptr(h), Bz, hr,
                                                   _ptr(conv_state), cdt, cr, _stream(stream)))
    return h, conv_state


def fitted_noise_update(hT: torch.Tensor, mu: torch.Tensor, var: torch.Tensor, beta: float = 0.1,
                        has_history: bool = True, stream=None):
    """Per-head mean and variance of hT [Bz, H, P, N] mixed into mu, var [H]
    (in place) with weight 1 - beta on the new statistic."""
    Bz, H, P, N = hT.shape
    _check("sss_fitted_noise_update",
           _lib.sss_fitted_noise_update(_ptr(hT), Bz, H, P, N, float(beta), int(bool(has_history)),
                                        _ptr(mu), _ptr(var), _stream(stream)))
    return mu, var


def fitted_noise_sample(mu: torch.Tensor, var: torch.Tensor, eps: torch.Tensor,
                        h0: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """h0 = mu_h + sqrt(var_h) eps, eps [Bz, H, P, N] standard normal draws."""
    Bz, H, P, N = eps.shape
    if h0 is None:
        h0 = torch.empty_like(eps)
    _check("sss_fitted_noise_sample", _lib.sss_fitted_noise_sample(
        _ptr(mu), _ptr(var), _ptr(eps), _ptr(h0), Bz, H, P, N, _stream(stream)))
    return h0


def state_std_trace(x: torch.Tensor, dt: torch.Tensor, A: torch.Tensor, B: torch.Tensor,
                    h0: Optional[torch.Tensor], stride: int = 64, stream=None) -> torch.Tensor:
    """Per-head standard deviation of the scan state every `stride` tokens (and
    after the last one): [Bz, ceil(L / stride), H] fp32."""
    Bz, L, H = dt.shape
    G, N = B.shape[2], B.shape[3]
    P = x.shape[-1] if x.dim() == 4 else x.shape[-1] // H
    out = torch.empty((Bz, -(-L // stride), H), dtype=torch.float32, device=x.device)
    _check("sss_state_std_trace", _lib.sss_state_std_trace(
        _ptr(x), _dt(x), _ptr(dt), _ptr(A), _ptr(B), _dt(dt), _ptr(h0), _ptr(out), Bz, L, H, P, N,
        G, int(stride), _stream(stream)))
    return out


def mixer_fwd_supported(Bz, L, H, P, N, G, K, x_dtype, y_dtype) -> bool:
    return bool(_lib.sss_mixer_fwd_supported(Bz, L, H, P, N, G, K, _dtype_code(x_dtype),
                                             _dtype_code(y_dtype)))


def mixer_fwd(x, dt, A, B, C, w, bias, conv_state=None, h0=None, conv_state_out=None,
              hT=None, y=None, u_dtype=torch.float32, y_dtype=None, fused=None, stream=None,
              spans=None, workspace=None):
    """One segment of the streaming forward: conv (with state) + SiLU, then the
    scan from h0.  Returns (y, conv_state_out, hT).

    fused=None picks the single-kernel sss_mixer_fwd when the library supports
    the shapes, else the two calls conv_state_fwd + ssm_scan_fwd (u kept in
    u_dtype between them); fused=True / False forces one or the other.
    spans: for the fused call, the number of equal spans the sequence is cut
    into and run in parallel (sss_mixer_fwd_spans); None = the library's
    choice for these sizes on this device, 1 = one pass."""
    Bz, L, D = x.shape
    H = dt.shape[2]
    P = D // H
    G, N = B.shape[2], B.shape[3]
    K = w.shape[1]
    y_dtype = y_dtype or x.dtype
    if conv_state_out is None:
        conv_state_out = torch.empty((Bz, D, K - 1), dtype=x.dtype, device=x.device)
    if hT is None:
        hT = torch.empty((Bz, H, P, N), dtype=torch.float32, device=x.device)
    if y is None:
        y = torch.empty((Bz, L, H, P), dtype=y_dtype, device=x.device)
    if fused is None:
        fused = mixer_fwd_supported(Bz, L, H, P, N, G, K, x.dtype, y.dtype)
    if fused and spans is None:
        spans = mixer_fwd_span_count(Bz, L, H, P, N, G, K, x.dtype, y.dtype)
    if fused and spans > 1:
        workspace = _span_workspace(Bz, L, H, P, N, K, spans, workspace, x.device)
        rc = _lib.sss_mixer_fwd_spans(_ptr(x), _dt(x), _ptr(w), _ptr(bias), _ptr(conv_state),
                                      _ptr(conv_state_out), _ptr(dt), _ptr(A), _ptr(B), _ptr(C),
                                      _ptr(h0), _ptr(hT), _ptr(y), _dt(y), Bz, L, H, P, N, G, K,
                                      spans, _ptr(workspace), _nbytes(workspace), _stream(stream))
        _check("sss_mixer_fwd_spans", rc)
        return y, conv_state_out, hT
    if fused:
        rc = _lib.sss_mixer_fwd(_ptr(x), _dt(x), _ptr(w), _ptr(bias), _ptr(conv_state),
                                _ptr(conv_state_out), _ptr(dt), _ptr(A), _ptr(B), _ptr(C),
                                _ptr(h0), _ptr(hT), _ptr(y), _dt(y), Bz, L, H, P, N, G, K,
                                _stream(stream))
        _check("sss_mixer_fwd", rc)
        return y, conv_state_out, hT
    u = conv_state_fwd(x, w, bias, conv_state, conv_state_out, u_dtype=u_dtype, stream=stream)
    ssm_scan_fwd(u, dt, A, B, C, h0, hT, y=y, stream=stream)
    return y, conv_state_out, hT


def mixer_update(x_new: torch.Tensor, w: torch.Tensor, bias: Optional[torch.Tensor],
                 conv_pool: torch.Tensor, cache_seqlens: Optional[torch.Tensor],
                 conv_state_indices: Optional[torch.Tensor], dt: torch.Tensor, A: torch.Tensor,
                 B: torch.Tensor, C: torch.Tensor, ssm_pool: torch.Tensor,
                 y: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """x_new [Bz, L_new, D]; conv_pool [pool, D, S_len] (updated in place);
    cache_seqlens, conv_state_indices [Bz] int32; dt [Bz, L_new, H]; A [H];
    B, C [Bz, L_new, G, N]; ssm_pool [pool, H, P, N] fp32 (updated in place).
    Returns y [Bz, L_new, H, P].  cache_seqlens is not advanced; None selects
    the non-circular mode (each row keeps its newest S_len inputs, oldest
    first, and is shifted by L_new)."""
    Bz, L_new, D = x_new.shape
    H = dt.shape[2]
    P = D // H
    pool, _, S_len = conv_pool.shape
    G, N = B.shape[2], B.shape[3]
    K = w.shape[1]
    if (cache_seqlens is not None and cache_seqlens.dtype != torch.int32) or (
            conv_state_indices is not None and conv_state_indices.dtype != torch.int32):
        raise TypeError("cache_seqlens and conv_state_indices must be int32")
    if y is None:
        y = torch.empty((Bz, L_new, H, P), dtype=x_new.dtype, device=x_new.device)
    rc = _lib.sss_mixer_update(_ptr(x_new), _dt(x_new), _ptr(w), _ptr(bias), _ptr(conv_pool),
                               pool, S_len, _ptr(cache_seqlens), _ptr(conv_state_indices),
                               _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(ssm_pool), _ptr(y), Bz,
                               L_new, H, P, N, G, K, _stream(stream))
    _check("sss_mixer_update", rc)
    return y


def mixer_update_path(L_new, P, N, K, S_len, act_dtype) -> int:
    """1 = bulk-copy pipelined update kernel, 0 = one CTA per (request, head),
    -1 = unsupported (for 16-byte aligned tensors with a bias)."""
    return int(_lib.sss_mixer_update_path(L_new, P, N, K, S_len, _dtype_code(act_dtype)))


def device_status(clear: bool = True, stream=None) -> int:
    """OR of device-raised status bits since the last clear (synchronises)."""
    v = ctypes.c_int(0)
    _check("sss_device_status", _lib.sss_device_status(ctypes.byref(v), int(bool(clear)),
                                                       _stream(stream)))
    return int(v.value)

def mamba2_mixer_fwd_workspace_size(Bz, L, H, P, N, G) -> int:
    return int(_lib.sss_mamba2_mixer_fwd_workspace_size(Bz, L, H, P, N, G))


def mamba2_mixer_fwd(xBC, z, dt_raw, dt_bias, A, D_skip, w, bias, H: int, G: int, N: int,
                     conv_state=None, h0=None, conv_state_out=None, hT=None, y=None,
                     y_dtype=None, workspace=None, stream=None):
    """One segment of the full Mamba-2 mixer wiring (sss_mamba2_mixer_fwd):
    the conv with state over every channel of xBC [Bz, L, H*P + 2 G N]
    (x, then B, then C), then per token dt = softplus(dt_raw + dt_bias),
    h = exp(dt A) h + dt x B^T, y = (h C + D_skip x) SiLU(z).  z, dt_bias,
    D_skip, bias, conv_state and h0 may be None.  Returns (y, conv_state_out,
    hT)."""
    Bz, L, Dt = xBC.shape
    P = (Dt - 2 * G * N) // H
    if P < 1 or H * P + 2 * G * N != Dt or w.shape[0] != Dt or dt_raw.shape != (Bz, L, H):
        raise ValueError("mamba2_mixer_fwd: xBC channels must be H*P + 2*G*N and match w, dt_raw")
    K = w.shape[1]
    y_dtype = y_dtype or xBC.dtype
    if conv_state_out is None:
        conv_state_out = torch.empty((Bz, Dt, K - 1), dtype=xBC.dtype, device=xBC.device)
    if hT is None:
        hT = torch.empty((Bz, H, P, N), dtype=torch.float32, device=xBC.device)
    if y is None:
        y = torch.empty((Bz, L, H, P), dtype=y_dtype, device=xBC.device)
    need = mamba2_mixer_fwd_workspace_size(Bz, L, H, P, N, G)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=xBC.device)
    _check("sss_mamba2_mixer_fwd", _lib.sss_mamba2_mixer_fwd(
        _ptr(xBC), _ptr(z), _dt(xBC), _ptr(dt_raw), _ptr(dt_bias), _ptr(A), _ptr(D_skip),
        _ptr(w), _ptr(bias), _ptr(conv_state), _ptr(conv_state_out), _ptr(h0), _ptr(hT),
        _ptr(y), _dt(y), Bz, L, H, P, N, G, K, _ptr(workspace), _nbytes(workspace),
        _stream(stream)))
    return y, conv_state_out, hT
