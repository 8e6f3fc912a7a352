"""State-passing training utilities on the GPU against the float64 oracle:
the zero reset of state passing (section 4.4 of "Understanding and Improving
Length Generalization in Recurrent Models"), the fitted-noise statistics and
initial states (section 4.2, Eqs. (5)-(6)) and the per-head state-scale trace
(section 3.5)."""
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


def T(a):
    return to_torch(a, DEV)


@pytest.mark.parametrize("conv_dtype", ["bf16", "f32"])
def test_state_reset(conv_dtype):
    g = np.random.default_rng(60)
    Bz = 1000
    u = synth.f32((np.arange(Bz) + 0.5) / Bz)
    g.shuffle(u.data)
    h = synth.f32(g.standard_normal((Bz, 2, 4, 8)))
    c = synth.store(g.standard_normal((Bz, 6, 3)), conv_dtype)
    th, tc = T(h), T(c)
    sss.state_reset(T(u), 0.1, th, tc)
    torch.cuda.synchronize()
    h_ref, c_ref = oracle.state_reset(u, 0.1, h, c)
    np.testing.assert_array_equal(f64(th), h_ref)
    np.testing.assert_array_equal(f64(tc), c_ref)
    assert int((f64(th).reshape(Bz, -1) == 0).all(axis=1).sum()) == 100


@pytest.mark.parametrize("has_history", [True, False])
def test_fitted_noise_update(has_history):
    s = synth.WORKLOADS["m370m_2k"]
    g = np.random.default_rng(61)
    hT = synth.f32(g.normal(0.3, 0.2, (s.Bz, s.H, s.P, s.N)))
    mu0 = synth.f32(g.standard_normal(s.H))
    var0 = synth.f32(g.uniform(0.1, 1.0, s.H))
    mu, var = T(mu0), T(var0)
    sss.fitted_noise_update(T(hT), mu, var, 0.1, has_history)
    torch.cuda.synchronize()
    m_ref, v_ref = (oracle.fitted_noise_update(hT, mu0, var0, 0.1) if has_history
                    else oracle.fitted_noise_update(hT))
    np.testing.assert_allclose(f64(mu), m_ref, rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(f64(var), v_ref, rtol=1e-6, atol=1e-9)


def test_fitted_noise_sample():
    g = np.random.default_rng(62)
    H = 6
    mu = synth.f32(g.standard_normal(H))
    var = synth.f32(g.uniform(0.01, 2.0, H))
    eps = synth.f32(g.standard_normal((3, H, 16, 32)))
    h0 = sss.fitted_noise_sample(T(mu), T(var), T(eps))
    torch.cuda.synchronize()
    assert_rel(f64(h0), oracle.fitted_noise_sample(mu, var, eps), 1e-6, "h0")


@pytest.mark.parametrize("L,stride,xdt", [(130, 64, "bf16"), (77, 7, "f32"), (40, 1, "bf16"),
                                          (64, 64, "f32")])
def test_state_std_trace(L, stride, xdt):
    g = np.random.default_rng(63 + L)
    Bz, H, P, N, G = 2, 4, 64, 128, 1
    x = synth.store(g.standard_normal((Bz, L, H, P)), xdt)
    dt = synth.store(np.log1p(np.exp(g.standard_normal((Bz, L, H)) - 2.0)), xdt)
    A = synth.f32(-g.uniform(0.01, 1.0, H))
    B = synth.store(g.standard_normal((Bz, L, G, N)), xdt)
    C = synth.store(g.standard_normal((Bz, L, G, N)), xdt)
    h0 = synth.f32(g.normal(0.0, 0.1, (Bz, H, P, N)))
    tr = sss.state_std_trace(T(x), T(dt), T(A), T(B), T(h0), stride)
    torch.cuda.synchronize()
    ref = oracle.state_std_trace(x, dt, A, B, C, h0, stride)
    assert tuple(tr.shape) == ref.shape
    assert_rel(f64(tr), ref, 1e-5, "state std")
