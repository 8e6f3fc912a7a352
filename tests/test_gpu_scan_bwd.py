"""Scan backward with state on the GPU against the float64 oracle.

Covers the gradient of the scalar-decay scan used for state-passing and
truncated-backpropagation training ("Understanding and Improving Length
Generalization in Recurrent Models" sections 4.4-4.5; the causal-conv
chapter's section on chunked training): dx, ddt, dA, dB, dC and the initial
state's gradient dh0, for fp32 and bf16 inputs, several chunks with a ragged
tail, grouped B/C, no initial state / no final-state gradient, L = 0 and
L = 1, segment B's dh0 fed to segment A as its dhT, determinism, and a
full-size segment on sampled heads.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import synth  # noqa: E402
from helpers import assert_rel, f64, to_torch  # noqa: E402

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import selective_ssm_scan_gb300 as sss  # noqa: E402

DEV = torch.device("cuda:0")
# every gradient is computed in fp32 from the exact input values; sums run
# over up to 128 terms and the decay gradient is a difference of such sums,
# so each tensor is held to max|gpu - ref| <= GRAD_REL * max|ref| (measured:
# below 1e-6 on every case here)
GRAD_REL = 1e-5


def T(a):
    return to_torch(a, DEV)


def _case(seed, Bz, L, H, P, N, G, xdt, adt, h0=True, dhT=True):
    g = np.random.default_rng(seed)
    x = synth.store(g.standard_normal((Bz, L, H, P)), xdt)
    dt = synth.store(np.log1p(np.exp(g.standard_normal((Bz, L, H)) - 2.0)), adt)
    A = synth.f32(-g.uniform(0.01, 1.0, H))
    B = synth.store(g.standard_normal((Bz, L, G, N)), adt)
    C = synth.store(g.standard_normal((Bz, L, G, N)), adt)
    s0 = synth.f32(g.normal(0.0, 0.1, (Bz, H, P, N))) if h0 else None
    dy = synth.f32(g.standard_normal((Bz, L, H, P)))
    gT = synth.f32(g.standard_normal((Bz, H, P, N))) if dhT else None
    return x, dt, A, B, C, s0, dy, gT


def _run(x, dt, A, B, C, s0, dy, gT):
    return sss.ssm_scan_bwd(T(x), T(dt), T(A), T(B), T(C), T(s0) if s0 is not None else None,
                            T(dy), T(gT) if gT is not None else None)


NAMES = ("dx", "ddt", "dA", "dB", "dC", "dh0")


@pytest.mark.parametrize("Bz,L,H,P,N,G,xdt,adt,h0,dhT", [
    (2, 150, 4, 64, 128, 1, "bf16", "bf16", True, True),    # 3 chunks, ragged tail
    (1, 64, 2, 16, 32, 1, "f32", "f32", True, True),        # exactly one chunk
    (2, 201, 6, 64, 128, 2, "f32", "bf16", False, True),    # groups, no h0
    (1, 129, 2, 40, 100, 1, "bf16", "f32", True, False),    # P, N not powers of two, no dhT
    (2, 1, 2, 8, 16, 1, "f32", "f32", True, True),          # one token
])
def test_scan_bwd_matches_oracle(Bz, L, H, P, N, G, xdt, adt, h0, dhT):
    args = _case(1000 + L + H, Bz, L, H, P, N, G, xdt, adt, h0, dhT)
    got = _run(*args)
    torch.cuda.synchronize()
    ref = oracle.ssm_scan_bwd(*args)
    for name, gv, rv in zip(NAMES, got, ref):
        assert_rel(f64(gv), rv, GRAD_REL, name)


def test_scan_bwd_empty_sequence():
    """L = 0: dh0 = dhT, dA = 0."""
    x, dt, A, B, C, s0, dy, gT = _case(7, 2, 0, 2, 8, 16, 1, "f32", "f32")
    dx, ddt, dA, dB, dC, dh0 = _run(x, dt, A, B, C, s0, dy, gT)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(f64(dh0), gT.f64())
    assert not f64(dA).any() and dx.shape[1] == 0


def test_scan_bwd_segments_chain_and_alias():
    """Segment B's dh0, written over the dhT buffer (allowed aliasing), is
    segment A's dhT: the two calls reproduce the whole sequence's gradients."""
    x, dt, A, B, C, s0, dy, gT = _case(8, 2, 300, 4, 64, 128, 1, "bf16", "bf16")
    whole = _run(x, dt, A, B, C, s0, dy, gT)
    split = 170
    sa, sb = slice(0, split), slice(split, None)
    cut = lambda a, sl: synth.Arr(np.ascontiguousarray(a.data[:, sl]), a.dtype)
    _, hA = oracle.ssm_scan(cut(x, sa), cut(dt, sa), A, cut(B, sa), cut(C, sa), s0)
    g = T(gT)
    gb = sss.ssm_scan_bwd(T(cut(x, sb)), T(cut(dt, sb)), T(A), T(cut(B, sb)), T(cut(C, sb)),
                          torch.from_numpy(hA.astype(np.float32)).to(DEV), T(cut(dy, sb)), g,
                          dh0=g)
    ga = sss.ssm_scan_bwd(T(cut(x, sa)), T(cut(dt, sa)), T(A), T(cut(B, sa)), T(cut(C, sa)),
                          T(s0), T(cut(dy, sa)), g)
    torch.cuda.synchronize()
    for k, name in ((0, "dx"), (1, "ddt"), (3, "dB"), (4, "dC")):
        assert_rel(np.concatenate([f64(ga[k]), f64(gb[k])], axis=1), f64(whole[k]), GRAD_REL, name)
    assert_rel(f64(ga[2]) + f64(gb[2]), f64(whole[2]), GRAD_REL, "dA")
    assert_rel(f64(ga[5]), f64(whole[5]), GRAD_REL, "dh0")


def test_scan_bwd_is_deterministic():
    args = _case(9, 2, 257, 4, 64, 128, 1, "bf16", "bf16")
    a = _run(*args)
    b = _run(*args)
    torch.cuda.synchronize()
    for name, u, v in zip(NAMES, a, b):
        assert torch.equal(u, v), name


def test_scan_bwd_full_segment_sampled():
    """The m370m_2k segment size (Bz 8, 1024 tokens, H 32, P 64, N 128, bf16):
    dx, ddt, dB, dC and dh0 of the first and last batch rows against the
    oracle run on just those rows (dA sums over every row and is covered by
    the smaller cases)."""
    s = synth.WORKLOADS["m370m_2k"]
    Bz, L, H, P, N = s.Bz, s.segments[0], s.H, s.P, s.N
    args = _case(10, Bz, L, H, P, N, 1, "bf16", "bf16")
    got = [f64(t) for t in _run(*args)]
    torch.cuda.synchronize()
    x, dt, A, B, C, s0, dy, gT = args
    for b in (0, Bz - 1):
        rows = slice(b, b + 1)
        sub = lambda a: synth.Arr(np.ascontiguousarray(a.data[rows]), a.dtype)
        ref = oracle.ssm_scan_bwd(sub(x), sub(dt), A, sub(B), sub(C), sub(s0), sub(dy), sub(gT))
        assert_rel(got[0][rows], ref[0], GRAD_REL, "dx")
        assert_rel(got[1][rows], ref[1], GRAD_REL, "ddt")
        assert_rel(got[3][rows], ref[3], GRAD_REL, "dB")
        assert_rel(got[4][rows], ref[4], GRAD_REL, "dC")
        assert_rel(got[5][rows], ref[5], GRAD_REL, "dh0")
