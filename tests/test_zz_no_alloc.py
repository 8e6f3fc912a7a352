"""The conv backward entry point that allocates nothing, against the regular one.

sss_conv_state_bwd_noalloc serves callers that cannot allocate device memory
when they run the backward (an engine plugin whose execute step may not
allocate, code with a fixed memory budget it has no allocator for): its
partial sums live in a static device array of the library instead of a
workspace.  These tests call it through the C ABI twice in a row, on
different shapes and dtypes so that the second call runs over the first
call's leftover partial sums, and compare each result with
sss_conv_state_bwd given a workspace of its own.  The file is named so that
pytest collects it last.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import synth  # noqa: E402
from helpers import F32_REL, assert_rel, assert_y_close, f64, to_torch  # noqa: E402

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import selective_ssm_scan_gb300 as sss  # noqa: E402

DEV = torch.device("cuda:0")


def _inputs(seed, Bz, L, D, K, xdt, dydt):
    g = np.random.default_rng(seed)
    T = lambda a: to_torch(a, DEV)
    x = T(synth.store(g.standard_normal((Bz, L, D)), xdt))
    w = T(synth.f32(g.normal(0, np.sqrt(0.5), (D, K))))
    bias = T(synth.f32(np.full(D, 0.1)))
    S = T(synth.store(g.standard_normal((Bz, D, K - 1)), xdt))
    dy = T(synth.store(g.standard_normal((Bz, L, D)), dydt))
    q = T(synth.store(g.standard_normal((Bz, D, K - 1)), dydt))
    return x, w, bias, S, dy, q


def _noalloc(x, w, bias, S, dy, q, dx_dtype):
    Bz, L, D = x.shape
    K = w.shape[1]
    dx = torch.empty((Bz, L, D), dtype=dx_dtype, device=DEV)
    dS = torch.empty((Bz, D, K - 1), dtype=dx_dtype, device=DEV)
    dw = torch.empty((D, K), dtype=torch.float32, device=DEV)
    db = torch.empty((D,), dtype=torch.float32, device=DEV)
    torch.cuda.synchronize()
    before = torch.cuda.memory_allocated(DEV)
    out = sss.conv_state_bwd_noalloc(x, w, bias, S, dy, q, dx, dS, dw, db)
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated(DEV) == before
    return out


def _compare(got, ref, bf16_out):
    dx, dS, dw, db = (f64(t) for t in got)
    rdx, rdS, rdw, rdb = (f64(t) for t in ref)
    if bf16_out:
        assert_y_close(dx, rdx, "dx")
        assert_y_close(dS, rdS, "dS")
    else:
        assert_rel(dx, rdx, F32_REL, "dx")
        assert_rel(dS, rdS, F32_REL, "dS")
    assert_rel(dw, rdw, F32_REL, "dw")
    assert_rel(db, rdb, F32_REL, "dbias")


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    # first call: a full 1024-token segment of the Mamba-2 370M-like layer
    # (1.3 MiB of partial sums); second call: a smaller ragged fp32 case that
    # reads only part of what the first call left in the scratch
    cases = [((1, 8, 1024, 2048, 4), "bf16", "f32", torch.bfloat16),
             ((2, 3, 301, 96, 4), "f32", "f32", torch.float32)]
    for (seed, Bz, L, D, K), xdt, dydt, odt in cases:
        x, w, bias, S, dy, q = _inputs(seed, Bz, L, D, K, xdt, dydt)
        assert sss.conv_state_bwd_workspace_size(Bz, L, D, K) <= sss.CONV_BWD_NOALLOC_SCRATCH_BYTES
        got = _noalloc(x, w, bias, S, dy, q, odt)
        ref = sss.conv_state_bwd(x, w, bias, S, dy, q, dx_dtype=odt)
        torch.cuda.synchronize()
        _compare(got, ref, odt == torch.bfloat16)
    assert sss.device_status() == 0


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # 64 sequences of 4096 tokens at D = 2048 need 40 MiB of partial sums:
    # the call returns SSS_ERR_UNSUPPORTED before looking at any pointer
    Bz, L, D, K = 64, 4096, 2048, 4
    assert sss.conv_state_bwd_workspace_size(Bz, L, D, K) > sss.CONV_BWD_NOALLOC_SCRATCH_BYTES
    rc = sss._lib.sss_conv_state_bwd_noalloc(
        None, sss.SSS_BF16, None, None, None, None, sss.SSS_F32, None, None, sss.SSS_BF16,
        None, None, None, Bz, L, D, K, 1, ctypes.c_void_p(0))
    assert rc == sss.SSS_ERR_UNSUPPORTED
