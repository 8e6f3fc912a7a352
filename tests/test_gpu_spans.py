"""Span-parallel forward on the GPU against the float64 oracle.

A sequence cut into ns equal spans run side by side, their states joined by
the associative composition of section 2.5 Eq. (4) of "Understanding and
Improving Length Generalization in Recurrent Models" (the state after a
stretch = its zero-start state + the inherited state times the stretch's
total decay).  The oracle runs the sequence as one piece, so any error in a
span's conv state, its decay or the carry shows up in y, F or hT.  Cases: 2
to 32 spans, spans shorter than a chunk and spans of several chunks, the
conv window reaching into the previous span, states passed in place,
grouped B/C, fp32 x and y on the scan alone, the library's choice of span
count, a full-size 780M-like segment pair on sampled heads, the whole
64-segment long-context stream at 4, 8 and 16 spans on sampled heads,
argument checks.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import synth  # noqa: E402
from helpers import STATE_REL, assert_rel, assert_y_close, f64, to_torch  # noqa: E402

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import selective_ssm_scan_gb300 as sss  # noqa: E402

DEV = torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _clean_status():
    sss.device_status(clear=True)
    yield
    assert sss.device_status(clear=True) == 0


def T(a):
    return to_torch(a, DEV)


def _mixer_case(seed, Bz, L, H, G=1, K=4, states=True):
    s = synth.WORKLOADS["m370m_2k"].with_(Bz=Bz, segments=(L,), H=H, G=G, K=K,
                                          gaussian_init=states, seed=seed)
    return s, synth.mixer_params(s), synth.mixer_segment(s, 0), synth.mixer_initial_states(s)


@pytest.mark.parametrize("ns,L,H,G", [
    (2, 512, 4, 1),     # two spans of four chunks
    (4, 512, 4, 1),
    (8, 1024, 2, 1),    # spans of one chunk
    (3, 390, 4, 2),     # spans of 130 tokens (a ragged chunk each), grouped B/C
    (32, 160, 2, 1),    # one lane per span in the carry; 5-token spans
    (16, 48, 2, 1),     # 3-token spans: the conv window is the whole previous span
])
def test_mixer_spans_match_oracle(ns, L, H, G):
    s, p, seg, st = _mixer_case(2000 + ns + L, 2, L, H, G)
    y_ref, F_ref, h_ref = oracle.mixer_fwd(seg["x"], seg["dt"], p["A"], seg["B"], seg["C"],
                                           p["w"], p["bias"], st["conv_state"], st["h0"])
    S, h = T(st["conv_state"]), T(st["h0"])
    y, F, hT = sss.mixer_fwd(T(seg["x"]), T(seg["dt"]), T(p["A"]), T(seg["B"]), T(seg["C"]),
                             T(p["w"]), T(p["bias"]), S, h, conv_state_out=S, hT=h, fused=True,
                             spans=ns)
    torch.cuda.synchronize()
    assert F.data_ptr() == S.data_ptr() and hT.data_ptr() == h.data_ptr()
    assert_y_close(f64(y).reshape(y_ref.shape), y_ref)
    np.testing.assert_array_equal(f64(F), F_ref)
    assert_rel(f64(hT), h_ref, STATE_REL, "hT")


def test_mixer_spans_without_states():
    s, p, seg, _ = _mixer_case(2100, 1, 600, 4, states=False)
    y_ref, F_ref, h_ref = oracle.mixer_fwd(seg["x"], seg["dt"], p["A"], seg["B"], seg["C"],
                                           p["w"], p["bias"], None, None)
    y, F, hT = sss.mixer_fwd(T(seg["x"]), T(seg["dt"]), T(p["A"]), T(seg["B"]), T(seg["C"]),
                             T(p["w"]), T(p["bias"]), None, None, fused=True, spans=6,
                             y_dtype=torch.float32)
    torch.cuda.synchronize()
    assert_y_close(f64(y).reshape(y_ref.shape), y_ref)
    np.testing.assert_array_equal(f64(F), F_ref)
    assert_rel(f64(hT), h_ref, STATE_REL, "hT")


@pytest.mark.parametrize("xdt,ydt", [("bf16", "bf16"), ("f32", "f32"), ("bf16", "f32")])
@pytest.mark.parametrize("ns", [2, 5])
def test_scan_spans_match_oracle(xdt, ydt, ns):
    g = np.random.default_rng(2200 + ns)
    Bz, L, H, P, N, G = 2, 700, 4, 64, 128, 1
    x = synth.store(g.standard_normal((Bz, L, H, P)), xdt)
    dt = synth.bf16(np.log1p(np.exp(g.standard_normal((Bz, L, H)) - 2.0)))
    A = synth.f32(-g.uniform(0.01, 1.0, H))
    B = synth.bf16(g.standard_normal((Bz, L, G, N)))
    C = synth.bf16(g.standard_normal((Bz, L, G, N)))
    h0 = synth.f32(g.normal(0.0, 0.1, (Bz, H, P, N)))
    y_ref, h_ref = oracle.ssm_scan(x, dt, A, B, C, h0)
    h = T(h0)
    y, hT = sss.ssm_scan_fwd(T(x), T(dt), T(A), T(B), T(C), h, h,
                             y_dtype=torch.float32 if ydt == "f32" else torch.bfloat16, spans=ns)
    torch.cuda.synchronize()
    assert_y_close(f64(y), y_ref)
    assert_rel(f64(hT), h_ref, STATE_REL, "hT")


def test_span_count_choice():
    """One 780M-like segment (batch 1, 48 heads: 24 head pairs) is split; the
    370M-like and 1.3B-like segments already fill the GPU and are not; the
    fp32 CUDA-core shapes never are."""
    bf = torch.bfloat16
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    ns = sss.mixer_fwd_span_count(1, 2048, 48, 64, 128, 1, 4, bf, bf)
    if sms >= 96:
        assert ns > 1 and 2048 % ns == 0
    assert sss.mixer_fwd_span_count(8, 1024, 32, 64, 128, 1, 4, bf, bf) == 1 or sms > 256
    assert sss.mixer_fwd_span_count(1, 2048, 2, 4, 8, 1, 4, torch.float32, torch.float32) == 1
    assert sss.ssm_scan_fwd_span_count(1, 64, 2, 4, 8, 1, torch.float32, torch.float32,
                                       torch.float32) == 1


def test_long_context_segments_with_spans_sampled():
    """Two full 780M-like segments (batch 1, 2048 tokens, H 48) through the
    library's own choice of spans, states passed in place; y and the states
    of heads 0, 23 and 47 against the oracle."""
    s = synth.WORKLOADS["m780m_128k"].with_(segments=(2048, 2048), gaussian_init=True)
    heads = [0, 23, 47]
    p = synth.mixer_params(s)
    st = synth.mixer_initial_states(s)
    A, w, bias = T(p["A"]), T(p["w"]), T(p["bias"])
    S, h = T(st["conv_state"]), T(st["h0"])
    chan = np.concatenate([np.arange(hh * s.P, (hh + 1) * s.P) for hh in heads])
    S_ref = st["conv_state"].f64()[:, chan]
    h_ref = st["h0"].f64()[:, heads]
    for i in range(len(s.segments)):
        seg = synth.mixer_segment(s, i)
        y, S, h = sss.mixer_fwd(T(seg["x"]), T(seg["dt"]), A, T(seg["B"]), T(seg["C"]), w, bias,
                                S, h, conv_state_out=S, hT=h)
        y_ref, S_ref, h_ref = oracle.mixer_fwd(seg["x"].f64()[:, :, chan],
                                               seg["dt"].f64()[:, :, heads], p["A"].f64()[heads],
                                               seg["B"].f64(), seg["C"].f64(), p["w"].f64()[chan],
                                               p["bias"].f64()[chan], S_ref, h_ref)
        assert_y_close(f64(y[:, :, heads]), y_ref, f"segment {i} y")
    torch.cuda.synchronize()
    np.testing.assert_array_equal(f64(S)[:, chan], S_ref)
    assert_rel(f64(h)[:, heads], h_ref, STATE_REL, "hT")


@pytest.mark.parametrize("ns", [4, 8, 16])
def test_long_context_stream_with_spans_sampled(ns):
    """The whole 780M-like long-context stream: 64 segments of 2048 tokens
    (batch 1, H 48, Gaussian initial states), every call cut into ns spans,
    conv and SSM states passed in place from call to call.  y of heads 0, 23
    and 47 in every segment, and the final states, against the oracle run
    segment by segment on those heads' channels (the conv is depthwise and
    the heads independent, so the sample is exact)."""
    s = synth.WORKLOADS["m780m_128k"].with_(gaussian_init=True)
    assert len(s.segments) == 64
    heads = [0, 23, 47]
    p = synth.mixer_params(s)
    st = synth.mixer_initial_states(s)
    A, w, bias = T(p["A"]), T(p["w"]), T(p["bias"])
    S, h = T(st["conv_state"]), T(st["h0"])
    chan = np.concatenate([np.arange(hh * s.P, (hh + 1) * s.P) for hh in heads])
    S_ref = st["conv_state"].f64()[:, chan]
    h_ref = st["h0"].f64()[:, heads]
    for i in range(len(s.segments)):
        seg = synth.mixer_segment(s, i)
        y, S, h = sss.mixer_fwd(T(seg["x"]), T(seg["dt"]), A, T(seg["B"]), T(seg["C"]), w, bias,
                                S, h, conv_state_out=S, hT=h, spans=ns)
        y_ref, S_ref, h_ref = oracle.mixer_fwd(seg["x"].f64()[:, :, chan],
                                               seg["dt"].f64()[:, :, heads], p["A"].f64()[heads],
                                               seg["B"].f64(), seg["C"].f64(), p["w"].f64()[chan],
                                               p["bias"].f64()[chan], S_ref, h_ref)
        assert_y_close(f64(y[:, :, heads]), y_ref, f"segment {i} y")
    torch.cuda.synchronize()
    np.testing.assert_array_equal(f64(S)[:, chan], S_ref)
    assert_rel(f64(h)[:, heads], h_ref, STATE_REL, "hT")


def test_span_argument_checks():
    s, p, seg, st = _mixer_case(2300, 1, 60, 2)
    args = (T(seg["x"]), T(seg["dt"]), T(p["A"]), T(seg["B"]), T(seg["C"]), T(p["w"]),
            T(p["bias"]), T(st["conv_state"]), T(st["h0"]))
    with pytest.raises(sss.SSSError) as e:          # 60 tokens do not split in 7
        sss.mixer_fwd(*args, fused=True, spans=7)
    assert e.value.status == sss.SSS_ERR_INVALID_ARG
    with pytest.raises(sss.SSSError) as e:          # 2-token spans < K - 1 = 3
        sss.mixer_fwd(*args, fused=True, spans=30)
    assert e.value.status == sss.SSS_ERR_INVALID_ARG
    with pytest.raises(sss.SSSError) as e:          # too small a workspace
        sss.mixer_fwd(*args, fused=True, spans=4,
                      workspace=torch.empty(64, dtype=torch.uint8, device=DEV))
    assert e.value.status == sss.SSS_ERR_INVALID_ARG
