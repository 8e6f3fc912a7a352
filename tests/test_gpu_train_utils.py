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


@pytest.mark.parametrize("circular", [True, False])
@pytest.mark.parametrize("L,S_len,K", [(9, 4, 4), (2, 6, 4), (0, 3, 4), (130, 8, 3)])
def test_prefill_to_pool(circular, L, S_len, K):
    g = np.random.default_rng(64 + L + S_len)
    Bz, pool, H, P, N = 3, 6, 2, 64, 128
    D = H * P
    x = synth.bf16(g.standard_normal((Bz, L, D)))
    S0 = synth.bf16(g.standard_normal((Bz, D, K - 1)))
    hT = synth.f32(g.standard_normal((Bz, H, P, N)))
    cp0 = synth.bf16(g.standard_normal((pool, D, S_len)))
    sp0 = synth.f32(g.standard_normal((pool, H, P, N)))
    idx = synth.Arr(np.array([4, 0, 2], np.int32), "i32")
    lens = synth.Arr(np.array([L, L + 5, L + 13], np.int32), "i32") if circular else None
    cp, sp = T(cp0), T(sp0)
    sss.prefill_to_pool(T(x), T(S0), K, T(hT), cp, sp, T(lens) if circular else None, T(idx), H)
    torch.cuda.synchronize()
    cp_ref, sp_ref, bad = oracle.prefill_to_pool(x, S0, K, hT, cp0, sp0, lens, idx)
    assert bad == 0 and sss.device_status() == 0
    np.testing.assert_array_equal(f64(cp), cp_ref)
    np.testing.assert_array_equal(f64(sp), sp_ref)


@pytest.mark.parametrize("circular", [True, False])
def test_prefill_then_decode_continues_the_sequence(circular):
    """The fused forward on a prompt, its state written into the pool, then
    the decode update on the next tokens: y of those tokens matches the
    oracle's forward over the whole sequence."""
    g = np.random.default_rng(65)
    Bz, pool, H, P, N, K, S_len, L, Lnew = 2, 5, 4, 64, 128, 4, 4, 200, 3
    D = H * P
    T_all = L + Lnew
    x = synth.bf16(g.standard_normal((Bz, T_all, D)))
    dt = synth.bf16(np.log1p(np.exp(g.standard_normal((Bz, T_all, H)) - 2.0)))
    A = synth.f32(-g.uniform(0.01, 1.0, H))
    B = synth.bf16(g.standard_normal((Bz, T_all, 1, N)))
    C = synth.bf16(g.standard_normal((Bz, T_all, 1, N)))
    w = synth.f32(g.normal(0, np.sqrt(0.5), (D, K)))
    bias = synth.f32(np.full(D, 0.1))
    S0 = synth.bf16(g.standard_normal((Bz, D, K - 1)))
    h0 = synth.f32(g.normal(0.0, 0.1, (Bz, H, P, N)))
    cut = lambda a, sl: synth.Arr(np.ascontiguousarray(a.data[:, sl]), a.dtype)
    pre, post = slice(0, L), slice(L, None)
    _, F, hT = sss.mixer_fwd(T(cut(x, pre)), T(cut(dt, pre)), T(A), T(cut(B, pre)),
                             T(cut(C, pre)), T(w), T(bias), T(S0), T(h0))
    cp = torch.zeros((pool, D, S_len), dtype=torch.bfloat16, device=DEV)
    sp = torch.zeros((pool, H, P, N), dtype=torch.float32, device=DEV)
    idx = torch.tensor([3, 1], dtype=torch.int32, device=DEV)
    lens = torch.full((Bz,), L, dtype=torch.int32, device=DEV) if circular else None
    sss.prefill_to_pool(T(cut(x, pre)), T(S0), K, hT, cp, sp, lens, idx, H)
    y = sss.mixer_update(T(cut(x, post)), T(w), T(bias), cp, lens, idx, T(cut(dt, post)), T(A),
                         T(cut(B, post)), T(cut(C, post)), sp)
    torch.cuda.synchronize()
    assert sss.device_status() == 0
    y_ref, _, _ = oracle.mixer_fwd(x, dt, A, B, C, w, bias, S0, h0)
    from helpers import assert_y_close
    assert_y_close(f64(y), y_ref[:, post].reshape(Bz, Lnew, H * P).reshape(f64(y).shape))
