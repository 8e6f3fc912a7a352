"""GPU parity of the full Mamba-2 mixer wiring (sss_mamba2_mixer_fwd) against
the float64 oracle: the conv with state over every xBC channel, dt bias and
softplus, the dt-scaled input, the D skip and the SiLU(z) gate.

Tolerances as for the forward (tests/helpers.py): fp32 inputs 1e-5 of the
largest |y| and |hT|; bf16 inputs y elementwise 1e-2 + 2e-2 |ref| and the final
SSM state 1e-3 of its largest value; the final conv state bit-exact."""
import numpy as np
import pytest

import oracle
import synth
from helpers import F32_REL, STATE_REL, assert_rel, assert_y_close, f64, to_torch

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import selective_ssm_scan_gb300 as sss  # noqa: E402

DEV = torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _clean_status():
    sss.device_status(clear=True)
    yield
    assert sss.device_status() == 0


def T(a):
    return None if a is None else to_torch(a, DEV)


def _run_gpu(a, s, gate=True, skip=True, dt_bias=True, states=True, conv_out=None, hT=None):
    y, F, h = sss.mamba2_mixer_fwd(
        T(a["xBC"]), T(a["z"]) if gate else None, T(a["dt_raw"]), T(a["dt_bias"]) if dt_bias else None,
        T(a["A"]), T(a["D_skip"]) if skip else None, T(a["w"]), T(a["bias"]), s.H, s.G, s.N,
        conv_state=T(a["conv_state"]) if states else None, h0=T(a["h0"]) if states else None,
        conv_state_out=conv_out, hT=hT)
    torch.cuda.synchronize()
    return y, F, h


def _run_ref(a, s, gate=True, skip=True, dt_bias=True, states=True):
    return oracle.mamba2_mixer_fwd(
        a["xBC"], a["z"] if gate else None, a["dt_raw"], a["dt_bias"] if dt_bias else None,
        a["A"], a["D_skip"] if skip else None, a["w"], a["bias"],
        a["conv_state"] if states else None, a["h0"] if states else None, s.H, s.G, s.N)


def _check(gpu, ref, dtype):
    y, F, h = gpu
    y_ref, F_ref, h_ref = ref
    if dtype == "f32":
        assert_rel(f64(y), y_ref, F32_REL, "y")
        assert_rel(f64(h), h_ref, F32_REL, "hT")
    else:
        assert_y_close(f64(y), y_ref)
        assert_rel(f64(h), h_ref, STATE_REL, "hT")
    assert np.array_equal(f64(F), F_ref), "final conv state"


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("L", [1, 37, 130])
@pytest.mark.parametrize("H,P,N,G", [(4, 16, 32, 2), (2, 64, 128, 1), (2, 24, 48, 1)])
def test_mamba2_small_parity(dtype, L, H, P, N, G):
    s = synth.WORKLOADS["m370m_2k"].with_(dtype=dtype, Bz=2, segments=(L,), H=H, P=P, N=N, G=G,
                                           gaussian_init=True, seed=2101 + L)
    a = synth.mamba2_inputs(s)
    _check(_run_gpu(a, s), _run_ref(a, s), dtype)


@pytest.mark.parametrize("gate,skip,dt_bias,states", [
    (False, True, True, True), (True, False, True, True), (True, True, False, True),
    (True, True, True, False), (False, False, False, False)])
def test_mamba2_optional_terms(gate, skip, dt_bias, states):
    s = synth.WORKLOADS["m370m_2k"].with_(Bz=2, segments=(96,), H=4, P=32, N=64, G=2,
                                           gaussian_init=True, seed=2201)
    a = synth.mamba2_inputs(s)
    kw = dict(gate=gate, skip=skip, dt_bias=dt_bias, states=states)
    _check(_run_gpu(a, s, **kw), _run_ref(a, s, **kw), "bf16")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_mamba2_strong_decay_chunks(dtype):
    """Heads whose log decay over 32 tokens passes 60 (the kernel's direct
    form) beside ordinary heads (its scaled form), over a ragged tail."""
    s = synth.WORKLOADS["m370m_2k"].with_(dtype=dtype, Bz=2, segments=(203,), H=4, P=64, N=128,
                                           G=2, gaussian_init=True, seed=2151)
    a = synth.mamba2_inputs(s)
    a["A"] = synth.f32(np.array([-0.02, -14.0, -60.0, -1.0]))
    _check(_run_gpu(a, s), _run_ref(a, s), dtype)


def test_mamba2_segments_with_state_aliasing_equal_one_call():
    """Two calls that pass the conv state (every xBC channel) and the SSM
    state in place, against the oracle over the whole sequence."""
    s = synth.WORKLOADS["m370m_2k"].with_(Bz=2, segments=(70, 58), H=4, P=32, N=64, G=2,
                                           gaussian_init=True, seed=2301)
    a0, a1 = synth.mamba2_inputs(s, 0), synth.mamba2_inputs(s, 1)
    S = T(a0["conv_state"])
    h = T(a0["h0"])
    ys = []
    for a in (a0, a1):
        y, S, h = sss.mamba2_mixer_fwd(T(a["xBC"]), T(a["z"]), T(a["dt_raw"]), T(a["dt_bias"]),
                                       T(a["A"]), T(a["D_skip"]), T(a["w"]), T(a["bias"]),
                                       s.H, s.G, s.N, conv_state=S, h0=h, conv_state_out=S, hT=h)
        ys.append(f64(y))
    torch.cuda.synchronize()
    whole = dict(a0)
    for k in ("xBC", "z", "dt_raw"):
        whole[k] = synth.Arr(np.concatenate([a0[k].data, a1[k].data], axis=1), a0[k].dtype)
    y_ref, F_ref, h_ref = _run_ref(whole, s.with_(segments=(128,)))
    assert_y_close(np.concatenate(ys, axis=1), y_ref)
    assert np.array_equal(f64(S), F_ref)
    assert_rel(f64(h), h_ref, STATE_REL, "hT")


@pytest.mark.parametrize("name,rows", [("m370m_2k", slice(0, 2)), ("m1p3b_8k", slice(0, 1))])
def test_mamba2_workload_shapes(name, rows):
    """The 370M-like (one 1024-token segment) and 1.3B-like (8192 tokens,
    Gaussian initial states) layer shapes, on the first batch rows."""
    s = synth.WORKLOADS[name]
    n = rows.stop - rows.start
    s = s.with_(Bz=n) if name == "m1p3b_8k" else s.with_(Bz=n, segments=(s.segments[0],))
    a = synth.mamba2_inputs(s)
    _check(_run_gpu(a, s), _run_ref(a, s), "bf16")


def test_mamba2_rejects_bad_arguments():
    s = synth.WORKLOADS["m370m_2k"].with_(Bz=1, segments=(8,), H=2, P=16, N=32, G=1)
    a = synth.mamba2_inputs(s)
    with pytest.raises(ValueError):
        # the channel count is not H P + 2 G N
        sss.mamba2_mixer_fwd(T(a["xBC"])[:, :, :-1], None, T(a["dt_raw"]), None, T(a["A"]),
                             None, T(a["w"])[:-1], None, s.H, s.G, s.N)
