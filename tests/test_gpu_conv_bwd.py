"""Conv backward with state on the GPU against the float64 oracle.

Covers the gradient derived in "Chapter 7: state, chunking and incremental
inference" (section on the backward pass with state): dx, dS (the state's
gradient, including the direct path from the final state F), dw and dbias,
for fp32 and bf16 activations, short sequences (L < K-1, L = 0), no state,
chunked training (segment B's dS feeds segment A's dF), determinism of the
weight gradients, and the full-size segment on sampled channels.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import synth  # noqa: E402
from helpers import F32_REL, assert_rel, assert_y_close, f64, to_torch  # noqa: E402

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import selective_ssm_scan_gb300 as sss  # noqa: E402

DEV = torch.device("cuda:0")
TD = {"f32": torch.float32, "bf16": torch.bfloat16}


def T(a):
    return to_torch(a, DEV)


def _case(seed, Bz, L, D, K, xdt, dydt, state=True, dstate=True):
    g = np.random.default_rng(seed)
    x = synth.store(g.standard_normal((Bz, L, D)), xdt)
    w = synth.f32(g.normal(0, np.sqrt(0.5), (D, K)))
    bias = synth.f32(np.full(D, 0.1))
    S = synth.store(g.standard_normal((Bz, D, K - 1)), xdt) if state else None
    dy = synth.store(g.standard_normal((Bz, L, D)), dydt)
    q = synth.store(g.standard_normal((Bz, D, K - 1)), dydt) if dstate else None
    return x, w, bias, S, dy, q


def _run(x, w, bias, S, dy, q, dxdt, silu=True):
    out = sss.conv_state_bwd(T(x), T(w), T(bias), T(S) if S is not None else None, T(dy),
                             T(q) if q is not None else None, dx_dtype=TD[dxdt],
                             apply_silu=silu)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("Bz,L,D,K,silu", [
    (2, 37, 24, 4, True), (2, 37, 7, 4, False), (3, 1, 16, 4, True), (2, 2, 16, 4, True),
    (2, 70, 16, 3, True), (2, 65, 16, 2, True), (1, 130, 10, 5, True), (2, 9, 16, 8, True),
    (2, 5, 6, 1, True), (1, 64, 32, 4, True), (1, 129, 32, 4, True), (2, 600, 18, 3, True),
    (1, 520, 34, 8, False), (2, 769, 66, 4, True)])
def test_conv_bwd_fp32_parity(Bz, L, D, K, silu):
    x, w, bias, S, dy, q = _case(31 * L + D + K, Bz, L, D, K, "f32", "f32")
    dx_r, dS_r, dw_r, db_r = oracle.conv_state_bwd(x, w, bias, S, dy, q, apply_silu=silu)
    dx, dS, dw, db = _run(x, w, bias, S, dy, q, "f32", silu)
    assert_rel(f64(dx), dx_r, F32_REL, "dx")
    if K > 1:
        assert_rel(f64(dS), dS_r, F32_REL, "dS")
    assert_rel(f64(dw), dw_r, F32_REL, "dw")
    assert_rel(f64(db), db_r, F32_REL, "dbias")


@pytest.mark.parametrize("L", [3, 4, 63, 64, 66, 67, 68, 131, 512, 515, 577, 1091])
@pytest.mark.parametrize("D,silu,state,dstate", [
    (64, True, True, True), (128, False, True, True), (64, True, False, False),
    (192, True, True, False)])
def test_conv_bwd_k4_tiles_parity(L, D, silu, state, dstate):
    """K = 4 with D a multiple of 64 (the channel-pair walk): the first tile's
    state gradient, interior tiles, the look-ahead past a tile's end, the last
    tile's masks and the direct gradient of F, at lengths around the 64-token
    tile and the 512-token CTA row."""
    x, w, bias, S, dy, q = _case(101 * L + D, 2, L, D, 4, "f32", "f32", state=state,
                                 dstate=dstate)
    dx_r, dS_r, dw_r, db_r = oracle.conv_state_bwd(x, w, bias, S, dy, q, apply_silu=silu)
    dx, dS, dw, db = _run(x, w, bias, S, dy, q, "f32", silu)
    assert_rel(f64(dx), dx_r, F32_REL, "dx")
    assert_rel(f64(dS), dS_r, F32_REL, "dS")
    assert_rel(f64(dw), dw_r, F32_REL, "dw")
    assert_rel(f64(db), db_r, F32_REL, "dbias")


@pytest.mark.parametrize("dydt,dxdt", [("f32", "bf16"), ("bf16", "bf16"), ("f32", "f32")])
@pytest.mark.parametrize("L", [3, 300])
def test_conv_bwd_bf16_parity(dydt, dxdt, L):
    x, w, bias, S, dy, q = _case(7 + L, 2, L, 2048, 4, "bf16", dydt)
    dx_r, dS_r, dw_r, db_r = oracle.conv_state_bwd(x, w, bias, S, dy, q)
    dx, dS, dw, db = _run(x, w, bias, S, dy, q, dxdt)
    if dxdt == "bf16":
        assert_y_close(f64(dx), dx_r, "dx")
        assert_y_close(f64(dS), dS_r, "dS")
    else:
        assert_rel(f64(dx), dx_r, F32_REL, "dx")
        assert_rel(f64(dS), dS_r, F32_REL, "dS")
    assert_rel(f64(dw), dw_r, F32_REL, "dw")
    assert_rel(f64(db), db_r, F32_REL, "dbias")


def test_conv_bwd_without_state_and_state_gradient():
    x, w, bias, S, dy, q = _case(5, 2, 9, 32, 4, "f32", "f32", state=False, dstate=False)
    dx_r, dS_r, dw_r, db_r = oracle.conv_state_bwd(x, w, bias, None, dy, None)
    dx, dS, dw, db = _run(x, w, bias, None, dy, None, "f32")
    assert_rel(f64(dx), dx_r, F32_REL, "dx")
    assert_rel(f64(dS), dS_r, F32_REL, "dS")
    assert_rel(f64(dw), dw_r, F32_REL, "dw")


def test_conv_bwd_empty_sequence():
    """L = 0: dS = dF and zero weight gradients."""
    x, w, bias, S, dy, q = _case(6, 2, 0, 16, 4, "bf16", "f32")
    dx, dS, dw, db = _run(x, w, bias, S, dy, q, "f32")
    np.testing.assert_array_equal(f64(dS), q.f64())
    assert not dw.any() and not db.any()


def test_conv_bwd_chunked_equals_whole():
    """Backward of segment B from F_A, its dS fed as segment A's dF, gives the
    whole sequence's dx, dS, dw and dbias."""
    Bz, L, D, K, split = 2, 200, 64, 4, 77
    x, w, bias, S, dy, q = _case(9, Bz, L, D, K, "f32", "f32")
    xt, wt, bt, St, dyt, qt = T(x), T(w), T(bias), T(S), T(dy), T(q)
    dx, dS, dw, db = sss.conv_state_bwd(xt, wt, bt, St, dyt, qt)
    FA = torch.empty_like(St)
    sss.conv_state_fwd(xt[:, :split].contiguous(), wt, bt, St, FA)
    dxb, dSb, dwb, dbb = sss.conv_state_bwd(xt[:, split:].contiguous(), wt, bt, FA,
                                            dyt[:, split:].contiguous(), qt)
    dxa, dSa, dwa, dba = sss.conv_state_bwd(xt[:, :split].contiguous(), wt, bt, St,
                                            dyt[:, :split].contiguous(), dSb)
    torch.cuda.synchronize()
    assert_rel(f64(torch.cat([dxa, dxb], 1)), f64(dx), F32_REL, "dx")
    assert_rel(f64(dSa), f64(dS), F32_REL, "dS")
    assert_rel(f64(dwa + dwb), f64(dw), F32_REL, "dw")
    assert_rel(f64(dba + dbb), f64(db), F32_REL, "dbias")


def test_conv_bwd_weight_gradients_are_deterministic():
    x, w, bias, S, dy, q = _case(11, 4, 1000, 256, 4, "bf16", "f32")
    a = _run(x, w, bias, S, dy, q, "bf16")
    b = _run(x, w, bias, S, dy, q, "bf16")
    assert torch.equal(a[2], b[2]) and torch.equal(a[3], b[3])
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))


def test_conv_bwd_full_size_sampled():
    """The m370m_2k segment (Bz 8, 1024 tokens, D 2048), channels sampled for
    the oracle (the conv is depthwise: channels are independent)."""
    Bz, L, D, K = 8, 1024, 2048, 4
    x, w, bias, S, dy, q = _case(12, Bz, L, D, K, "bf16", "f32")
    dx, dS, dw, db = _run(x, w, bias, S, dy, q, "bf16")
    ch = np.r_[0:32, 1000:1008, 2040:2048]
    sub = lambda a, ax: synth.Arr(np.ascontiguousarray(np.take(a.data, ch, axis=ax)), a.dtype)
    dx_r, dS_r, dw_r, db_r = oracle.conv_state_bwd(
        sub(x, 2), synth.f32(w.f64()[ch]), synth.f32(bias.f64()[ch]), sub(S, 1), sub(dy, 2),
        sub(q, 1))
    assert_y_close(f64(dx[:, :, ch]), dx_r, "dx")
    assert_y_close(f64(dS[:, ch]), dS_r, "dS")
    assert_rel(f64(dw[ch]), dw_r, F32_REL, "dw")
    assert_rel(f64(db[ch]), db_r, F32_REL, "dbias")


# ---------------------------------------------------------------------------
# packed samples (seq_idx) in the conv forward
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("L,D,K,xdt,udt,bounds", [
    (40, 256, 4, "bf16", "f32", [5, 17, 18]),
    (33, 70, 3, "f32", "f32", [1]),
    (100, 64, 8, "bf16", "bf16", [50, 51, 52, 99]),
    (7, 32, 4, "f32", "bf16", []),
])
def test_packed_conv_matches_oracle(L, D, K, xdt, udt, bounds):
    g = np.random.default_rng(200 + L)
    Bz = 3
    x = synth.store(g.standard_normal((Bz, L, D)), xdt)
    w = synth.f32(g.normal(0, np.sqrt(0.5), (D, K)))
    bias = synth.f32(np.full(D, 0.1))
    S = synth.store(g.standard_normal((Bz, D, K - 1)), xdt)
    ids = np.zeros((Bz, L), np.int32)
    for i, s in enumerate(bounds):
        ids[:, s:] = i + 1
    ids[1] += 7                                         # other ids on another row
    u, F = sss.conv_state_fwd_packed(T(x), T(w), T(bias), T(S),
                                     torch.from_numpy(ids).to(DEV), u_dtype=TD[udt])
    torch.cuda.synchronize()
    ref, F_ref = oracle.conv_state_fwd_packed(x, w, bias, S, ids)
    if udt == "f32":
        assert_rel(f64(u), ref, F32_REL if xdt == "f32" else 1e-6, "u")
    else:
        assert_y_close(f64(u), ref, "u")
    np.testing.assert_array_equal(f64(F), F_ref)         # the state: copied inputs, bit-exact
