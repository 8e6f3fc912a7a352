"""Pins of the CPU oracle to facts fixed by the pages and by mathematics.

Each test checks the oracle against something other than itself: a worked
example printed on a page (fixtures under tests/golden/, each with its
source), a closed form, a textbook routine (numpy convolve / cumsum), the
unrolled form of the recurrence (Eq. (4) of "Understanding and Improving
Length Generalization in Recurrent Models"), or an invariant the pages state
(segment equivalence under state passing, superposition of the initial
state).  No GPU is used.
"""
import json
import os

import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def silu(z):
    return z / (1.0 + np.exp(-z))


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# conv with state
# ---------------------------------------------------------------------------

def test_conv_worked_example_k4(golden_dir):
    """K=4, S=[a,b,c], x=[d]: the window is [a,b,c,d] and F=[b,c,d]."""
    ex = _load(golden_dir, "conv_state_examples.json")["examples"][0]
    K = ex["K"]
    S = np.array(ex["S"]).reshape(1, 1, K - 1)
    x = np.array(ex["x"]).reshape(1, 1, 1)
    w = np.array(ex["w"]).reshape(1, K)
    bias = np.array([ex["bias"]])
    u, F = oracle.conv_state_fwd(x, w, bias, S, apply_silu=False)
    np.testing.assert_array_equal(F.reshape(-1), ex["F"])
    assert not np.array_equal(F.reshape(-1), ex["wrong_F_zero_padded"])
    z = ex["bias"] + float(np.dot(ex["w"], ex["window"]))
    assert u.reshape(-1)[0] == z
    # with the activation: SiLU of the same pre-activation
    u2, _ = oracle.conv_state_fwd(x, w, bias, S, apply_silu=True)
    assert u2.reshape(-1)[0] == pytest.approx(silu(z), rel=1e-15)


def test_conv_worked_example_k3(golden_dir):
    """K=3, S=[a,b], x=[c]: z = beta + w0 a + w1 b + w2 c and F = [b, c]."""
    ex = _load(golden_dir, "conv_state_examples.json")["examples"][1]
    K = ex["K"]
    u, F = oracle.conv_state_fwd(np.array(ex["x"]).reshape(1, 1, 1),
                                 np.array(ex["w"]).reshape(1, K),
                                 np.array([ex["bias"]]),
                                 np.array(ex["S"]).reshape(1, 1, K - 1), apply_silu=False)
    assert u.reshape(-1)[0] == ex["z"]
    np.testing.assert_array_equal(F.reshape(-1), ex["F"])


@pytest.mark.parametrize("K,L", [(4, 37), (4, 1), (4, 2), (4, 3), (3, 9), (2, 5), (6, 4)])
def test_conv_matches_numpy_convolve(K, L):
    """Brute force: numpy's textbook convolution over the extended sequence."""
    g = np.random.default_rng(7 + K * 100 + L)
    Bz, D = 2, 5
    x = g.standard_normal((Bz, L, D))
    S = g.standard_normal((Bz, D, K - 1))
    w = g.standard_normal((D, K))
    bias = g.standard_normal(D)
    u, F = oracle.conv_state_fwd(x, w, bias, S)
    for b in range(Bz):
        for d in range(D):
            ext = np.concatenate([S[b, d], x[b, :, d]])
            z = bias[d] + np.convolve(ext, w[d][::-1], mode="valid")
            np.testing.assert_allclose(u[b, :, d], silu(z), rtol=1e-13, atol=1e-15)
            np.testing.assert_array_equal(F[b, d], ext[len(ext) - (K - 1):])


def test_conv_without_state_is_zero_padding():
    """No initial state means S = 0."""
    g = np.random.default_rng(3)
    x = g.standard_normal((1, 6, 3))
    w = g.standard_normal((3, 4))
    u0, F0 = oracle.conv_state_fwd(x, w, None, None)
    u1, F1 = oracle.conv_state_fwd(x, w, np.zeros(3), np.zeros((1, 3, 3)))
    np.testing.assert_array_equal(u0, u1)
    np.testing.assert_array_equal(F0, F1)


def test_conv_k1_is_pointwise_affine():
    g = np.random.default_rng(4)
    x = g.standard_normal((2, 7, 3))
    w = g.standard_normal((3, 1))
    bias = g.standard_normal(3)
    u, F = oracle.conv_state_fwd(x, w, bias, None)
    np.testing.assert_allclose(u, silu(bias + x * w[:, 0]), rtol=1e-14)
    assert F.shape == (2, 3, 0)


def test_conv_empty_sequence_keeps_state():
    g = np.random.default_rng(5)
    S = g.standard_normal((2, 3, 3))
    u, F = oracle.conv_state_fwd(np.zeros((2, 0, 3)), g.standard_normal((3, 4)), None, S)
    assert u.shape == (2, 0, 3)
    np.testing.assert_array_equal(F, S)


# ---------------------------------------------------------------------------
# the recurrence
# ---------------------------------------------------------------------------

def _scan_case(g, Bz=2, L=11, H=4, P=3, N=5, G=2, h0=True):
    u = g.standard_normal((Bz, L, H, P))
    dt = np.log1p(np.exp(g.standard_normal((Bz, L, H)) - 1.0))
    A = -g.uniform(0.05, 1.0, H)
    B = g.standard_normal((Bz, L, G, N))
    C = g.standard_normal((Bz, L, G, N))
    hh = g.standard_normal((Bz, H, P, N)) if h0 else None
    return u, dt, A, B, C, hh


def test_scan_matches_unrolled_eq4():
    """Eq. (4): h_t = sum_s (prod_{r=s+1..t} a_r) B_s x_s + (prod_{r=0..t} a_r) h_{-1},
    y_t = C_t^T h_t, written out as an explicit double sum."""
    g = np.random.default_rng(11)
    Bz, L, H, P, N, G = 2, 9, 4, 3, 5, 2
    u, dt, A, B, C, h0 = _scan_case(g, Bz, L, H, P, N, G)
    y, hT = oracle.ssm_scan(u, dt, A, B, C, h0)
    for b in range(Bz):
        for h in range(H):
            gi = h // (H // G)
            a = np.exp(dt[b, :, h] * A[h])
            for t in range(L):
                ht = np.prod(a[0:t + 1]) * h0[b, h]
                for s in range(t + 1):
                    ht = ht + np.prod(a[s + 1:t + 1]) * np.outer(u[b, s, h], B[b, s, gi])
                np.testing.assert_allclose(y[b, t, h], ht @ C[b, t, gi], rtol=1e-12, atol=1e-12)
                if t == L - 1:
                    np.testing.assert_allclose(hT[b, h], ht, rtol=1e-12, atol=1e-12)


def test_scan_impulse_response_is_product_of_later_decays():
    """An input at s=0 only reaches h_t through a_1 ... a_t (not a_0)."""
    g = np.random.default_rng(12)
    L, H = 8, 1
    dt = g.uniform(0.1, 0.9, (1, L, H))
    A = np.array([-0.7])
    u = np.zeros((1, L, H, 1))
    u[0, 0, 0, 0] = 1.0
    B = np.ones((1, L, 1, 1))
    C = np.ones((1, L, 1, 1))
    y, _ = oracle.ssm_scan(u, dt, A, B, C, None)
    a = np.exp(dt[0, :, 0] * A[0])
    expect = [np.prod(a[1:t + 1]) for t in range(L)]
    np.testing.assert_allclose(y[0, :, 0, 0], expect, rtol=1e-14)


def test_scan_no_decay_is_prefix_sum():
    """A_h = 0 gives a_t = 1: h_t = h0 + cumsum_s x_s B_s^T."""
    g = np.random.default_rng(13)
    u, dt, A, B, C, h0 = _scan_case(g, G=1)
    A = np.zeros_like(A)
    y, hT = oracle.ssm_scan(u, dt, A, B, C, h0)
    upd = np.einsum("blhp,bln->blhpn", u, B[:, :, 0, :])
    h = h0[:, None] + np.cumsum(upd, axis=1)
    np.testing.assert_allclose(hT, h[:, -1], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(y, np.einsum("blhpn,bln->blhp", h, C[:, :, 0, :]),
                               rtol=1e-11, atol=1e-11)


def test_scan_full_decay_forgets_everything():
    """exp(dt*A) underflows to 0: h_t = x_t B_t^T, so y_t = x_t (B_t . C_t)."""
    g = np.random.default_rng(14)
    u, dt, A, B, C, h0 = _scan_case(g, G=1)
    A = np.full_like(A, -1e5)
    y, hT = oracle.ssm_scan(u, dt, A, B, C, h0)
    bc = np.einsum("bln,bln->bl", B[:, :, 0], C[:, :, 0])
    np.testing.assert_allclose(y, u * bc[:, :, None, None], rtol=1e-13)


def test_scan_initial_state_superposition():
    """Eq. (4): y(x, h0) = y(x, 0) + C_t^T (prod_{r<=t} a_r) h0."""
    g = np.random.default_rng(15)
    u, dt, A, B, C, h0 = _scan_case(g, Bz=2, L=23, H=4, P=3, N=6, G=2)
    y1, hT1 = oracle.ssm_scan(u, dt, A, B, C, h0)
    y0, hT0 = oracle.ssm_scan(u, dt, A, B, C, None)
    H, G = 4, 2
    for h in range(H):
        gi = h // (H // G)
        decay = np.exp(np.cumsum(dt[:, :, h] * A[h], axis=1))  # [Bz, L]
        corr = np.einsum("bl,bpn,bln->blp", decay, h0[:, h], C[:, :, gi])
        np.testing.assert_allclose(y1[:, :, h], y0[:, :, h] + corr, rtol=1e-11, atol=1e-11)
        np.testing.assert_allclose(hT1[:, h], hT0[:, h] + decay[:, -1, None, None] * h0[:, h],
                                   rtol=1e-11, atol=1e-11)


def test_state_variance_closed_form(golden_dir):
    """Section 2.4 teaching example: Var(h_t) = (1 - a^{2(t+1)}) / (1 - a^2); at
    a = 0.99 the state reaches ~47.4% of its stationary variance after 32 tokens
    and is near-stationary by 512.  Monte-Carlo over independent heads."""
    ex = _load(golden_dir, "state_variance.json")
    a = ex["a"]
    T = ex["tokens"]
    closed = lambda t: (1 - a ** (2 * (t + 1))) / (1 - a ** 2)
    stat = 1 / (1 - a ** 2)
    # the closed form reproduces the printed fraction
    assert abs(closed(T - 1) / stat - ex["fraction_of_stationary_printed"]) <= ex["printed_precision"]
    assert closed(ex["tokens_near_stationary"] - 1) / stat > 0.999
    n = 1 << 16
    L = ex["tokens_near_stationary"]
    g = np.random.default_rng(16)
    u = g.standard_normal((1, L, n, 1))
    dt = np.ones((1, L, n))
    A = np.full(n, np.log(a))
    one = np.ones((1, L, 1, 1))
    y, _ = oracle.ssm_scan(u, dt, A, one, one, None)
    for t in (T - 1, L - 1):
        v = np.mean(y[0, t, :, 0] ** 2)
        sig = np.sqrt(2.0 / n) * closed(t)
        assert abs(v - closed(t)) < 4 * sig, (t, v, closed(t))


# ---------------------------------------------------------------------------
# state passing
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("split", [1, 2, 3, 17, 31])
def test_segment_equivalence(split):
    """Whole sequence == segment A then segment B started from A's final conv
    and SSM states (S_B = F_A, h0_B = hT_A)."""
    g = np.random.default_rng(20 + split)
    Bz, L, H, P, N, K = 2, 32, 2, 4, 8, 4
    D = H * P
    x = g.standard_normal((Bz, L, D))
    dt = np.log1p(np.exp(g.standard_normal((Bz, L, H)) - 2.0))
    A = -g.uniform(0.01, 1, H)
    B = g.standard_normal((Bz, L, 1, N))
    C = g.standard_normal((Bz, L, 1, N))
    w = g.normal(0, np.sqrt(0.5), (D, K))
    bias = np.full(D, 0.1)
    S0 = g.standard_normal((Bz, D, K - 1))
    h0 = g.normal(0, 0.1, (Bz, H, P, N))
    y, F, hT = oracle.mixer_fwd(x, dt, A, B, C, w, bias, S0, h0)
    sa, sb = slice(0, split), slice(split, L)
    ya, Fa, ha = oracle.mixer_fwd(x[:, sa], dt[:, sa], A, B[:, sa], C[:, sa], w, bias, S0, h0)
    yb, Fb, hb = oracle.mixer_fwd(x[:, sb], dt[:, sb], A, B[:, sb], C[:, sb], w, bias, Fa, ha)
    np.testing.assert_allclose(np.concatenate([ya, yb], axis=1), y, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(Fb, F)
    np.testing.assert_allclose(hb, hT, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("ns", [2, 3, 4, 8])
def test_span_composition_equals_whole(ns):
    """The reading behind the span-parallel forward (Eq. (4): the inherited
    state enters decayed by the total decay of the tokens since): spans run
    from ZERO states, each one's initial state rebuilt afterwards by the
    composition (a1, s1) o (a2, s2) = (a1 a2, a2 s1 + s2) of the earlier spans'
    (exp(sum of l_t), zero-start final state) pairs applied to h0, and each
    span's y rebuilt by running it again from that state, equal the whole
    sequence's y and final state."""
    g = np.random.default_rng(40 + ns)
    Bz, H, P, N = 2, 2, 4, 8
    L = 6 * ns
    Ls = L // ns
    u = g.standard_normal((Bz, L, H, P))
    dt = np.log1p(np.exp(g.standard_normal((Bz, L, H)) - 2.0))
    A = -g.uniform(0.01, 1, H)
    B = g.standard_normal((Bz, L, 1, N))
    C = g.standard_normal((Bz, L, 1, N))
    h0 = g.normal(0, 0.1, (Bz, H, P, N))
    y, hT = oracle.ssm_scan(u, dt, A, B, C, h0)
    h_in = h0.copy()
    ys = []
    for k in range(ns):
        sl = slice(k * Ls, (k + 1) * Ls)
        _, s_k = oracle.ssm_scan(u[:, sl], dt[:, sl], A, B[:, sl], C[:, sl], None)
        a_k = np.exp((dt[:, sl] * A).sum(axis=1))           # [Bz, H]
        y_k, _ = oracle.ssm_scan(u[:, sl], dt[:, sl], A, B[:, sl], C[:, sl], h_in)
        ys.append(y_k)
        h_in = a_k[:, :, None, None] * h_in + s_k
    np.testing.assert_allclose(np.concatenate(ys, axis=1), y, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(h_in, hT, rtol=1e-12, atol=1e-12)


def test_tiny_workload_split_equals_unsplit():
    """The tiny fp32 workload: 64 tokens as two 32-token segments == unsplit."""
    s = synth.WORKLOADS["tiny_f32"]
    p = synth.mixer_params(s)
    st = synth.mixer_initial_states(s)
    segs = [synth.mixer_segment(s, i) for i in range(len(s.segments))]
    cat = {k: np.concatenate([sg[k].f64() for sg in segs], axis=1) for k in segs[0]}
    y, F, hT = oracle.mixer_fwd(cat["x"], cat["dt"], p["A"], cat["B"], cat["C"], p["w"],
                                p["bias"], st["conv_state"], st["h0"])
    S, h = st["conv_state"].f64(), st["h0"].f64()
    ys = []
    for sg in segs:
        yi, S, h = oracle.mixer_fwd(sg["x"], sg["dt"], p["A"], sg["B"], sg["C"], p["w"],
                                    p["bias"], S, h)
        ys.append(yi)
    np.testing.assert_allclose(np.concatenate(ys, axis=1), y, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(S, F)
    np.testing.assert_allclose(h, hT, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# decode update
# ---------------------------------------------------------------------------

def test_circular_slot_example(golden_dir):
    """K=3, S_len=4, p=5: history = logical 3, 4 = slots 3, 0; the new input
    goes to slot 1.  One channel, one-hot weights pick each history value."""
    ex = _load(golden_dir, "circular_slots.json")
    K, S_len, p = ex["K"], ex["S_len"], ex["p"]
    slots = np.array([1.0, 10.0, 100.0, 1000.0])
    pool = slots.reshape(1, 1, S_len)
    xnew = np.array([7.0]).reshape(1, 1, 1)
    one = np.ones((1, 1, 1, 1))
    ssm = np.zeros((1, 1, 1, 1))
    seen = []
    for k in range(K - 1):  # weight k picks the k-th oldest history value
        w = np.zeros((1, K))
        w[0, k] = 1.0
        # a = exp(-1e5) = 0 and B = C = 1: y equals the conv output
        y, cp, sp, nbad = oracle.mixer_update(xnew, w, np.zeros(1), pool, np.array([p]),
                                              np.array([0]), np.ones((1, 1, 1)),
                                              np.array([-1e5]), one, one, ssm)
        assert nbad == 0
        # invert SiLU by matching against the candidate slot values
        cand = [silu(v) for v in slots]
        seen.append(int(np.argmin([abs(c - y[0, 0, 0, 0]) for c in cand])))
        expect_new = slots.copy()
        expect_new[ex["write_slot"]] = 7.0
        np.testing.assert_array_equal(cp.reshape(-1), expect_new)
    assert seen == ex["history_slots"]


def _decode_case(g, Bz=3, pool=5, Lnew=2, H=2, P=3, N=4, K=4, S_len=4, G=1):
    D = H * P
    return dict(
        x=g.standard_normal((Bz, Lnew, D)), w=g.standard_normal((D, K)),
        bias=g.standard_normal(D), conv_pool=g.standard_normal((pool, D, S_len)),
        cache_seqlens=g.integers(0, 50, Bz).astype(np.int32),
        conv_state_indices=g.permutation(pool)[:Bz].astype(np.int32),
        dt=np.log1p(np.exp(g.standard_normal((Bz, Lnew, H)))), A=-g.uniform(0.01, 1, H),
        B=g.standard_normal((Bz, Lnew, G, N)), C=g.standard_normal((Bz, Lnew, G, N)),
        ssm_pool=g.standard_normal((pool, H, P, N)))


@pytest.mark.parametrize("Lnew,S_len,K", [(1, 3, 4), (1, 4, 4), (4, 4, 4), (6, 4, 4),
                                          (3, 7, 4), (2, 2, 3), (5, 1, 2)])
def test_update_equals_forward_from_gathered_state(Lnew, S_len, K):
    """The update on L_new tokens equals the conv-with-state forward plus the
    scan, started from the history read out of the circular slots; the slots
    then hold the newest inputs (x, not y), rows not addressed are untouched."""
    g = np.random.default_rng(30 + Lnew * 10 + S_len)
    c = _decode_case(g, Lnew=Lnew, S_len=S_len, K=K)
    y, cp, sp, nbad = oracle.mixer_update(**c)
    assert nbad == 0
    pool = c["conv_pool"]
    for b, r in enumerate(c["conv_state_indices"]):
        p = int(c["cache_seqlens"][b])
        hist = np.stack([pool[r, :, (p - (K - 1) + j) % S_len] for j in range(K - 1)], axis=-1)
        yb, Fb, hb = oracle.mixer_fwd(c["x"][b:b + 1], c["dt"][b:b + 1], c["A"],
                                      c["B"][b:b + 1], c["C"][b:b + 1], c["w"], c["bias"],
                                      hist[None], c["ssm_pool"][r:r + 1])
        np.testing.assert_allclose(y[b], yb[0], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(sp[r], hb[0], rtol=1e-12, atol=1e-12)
        expect = pool[r].copy()
        for i in range(Lnew):
            expect[:, (p + i) % S_len] = c["x"][b, i]
        np.testing.assert_array_equal(cp[r], expect)
    untouched = np.setdiff1d(np.arange(pool.shape[0]), c["conv_state_indices"])
    np.testing.assert_array_equal(cp[untouched], pool[untouched])
    np.testing.assert_array_equal(sp[untouched], c["ssm_pool"][untouched])


@pytest.mark.parametrize("S_len", [2, 4])
def test_noncircular_single_token_example(S_len):
    """Non-circular mode, K = 3 (the single-token update: the window is the
    newest K-1 stored inputs then x_t; the oldest input is dropped and x_t
    appended; the physical row may be longer than K-1).  Row [.., a, b],
    x = c: one-hot weights pick a, b, c in tap order and the row becomes
    [.., b, c]."""
    K = 3
    row = np.array([1.0, 10.0, 100.0, 1000.0])[-S_len:]
    pool = row.reshape(1, 1, S_len)
    xnew = np.array([7.0]).reshape(1, 1, 1)
    one = np.ones((1, 1, 1, 1))
    picked = []
    for k in range(K):
        w = np.zeros((1, K))
        w[0, k] = 1.0
        # a = exp(-1e5) = 0 and B = C = 1: y equals the conv output
        y, cp, sp, nbad = oracle.mixer_update(xnew, w, np.zeros(1), pool, None, None,
                                              np.ones((1, 1, 1)), np.array([-1e5]), one, one,
                                              np.zeros((1, 1, 1, 1)))
        assert nbad == 0
        picked.append(y[0, 0, 0, 0])
        np.testing.assert_array_equal(cp.reshape(-1), np.concatenate([row[1:], [7.0]]))
    np.testing.assert_allclose(picked, silu(np.array([row[-2], row[-1], 7.0])), rtol=1e-15)


@pytest.mark.parametrize("Lnew,S_len,K", [(1, 3, 4), (2, 4, 4), (4, 4, 4), (6, 4, 4), (3, 7, 4),
                                          (5, 2, 3)])
def test_noncircular_update_equals_forward_from_newest_inputs(Lnew, S_len, K):
    """Non-circular mode on L_new tokens equals the conv-with-state forward
    plus the scan started from the row's newest K-1 inputs; the row then holds
    the last S_len entries of [row, x_0 .. x_{L_new-1}] (x, not y)."""
    g = np.random.default_rng(70 + Lnew * 10 + S_len)
    c = _decode_case(g, Lnew=Lnew, S_len=S_len, K=K)
    c["cache_seqlens"] = None
    y, cp, sp, nbad = oracle.mixer_update(**c)
    assert nbad == 0
    pool = c["conv_pool"]
    for b, r in enumerate(c["conv_state_indices"]):
        hist = pool[r, :, S_len - (K - 1):]
        yb, Fb, hb = oracle.mixer_fwd(c["x"][b:b + 1], c["dt"][b:b + 1], c["A"],
                                      c["B"][b:b + 1], c["C"][b:b + 1], c["w"], c["bias"],
                                      hist[None], c["ssm_pool"][r:r + 1])
        np.testing.assert_allclose(y[b], yb[0], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(sp[r], hb[0], rtol=1e-12, atol=1e-12)
        seq = np.concatenate([pool[r], c["x"][b].T], axis=1)
        np.testing.assert_array_equal(cp[r], seq[:, Lnew:Lnew + S_len])
    untouched = np.setdiff1d(np.arange(pool.shape[0]), c["conv_state_indices"])
    np.testing.assert_array_equal(cp[untouched], pool[untouched])


def test_update_skips_bad_rows():
    g = np.random.default_rng(40)
    c = _decode_case(g)
    c["conv_state_indices"] = np.array([0, 99, 2], np.int32)
    c["cache_seqlens"] = np.array([3, 4, -1], np.int32)
    y, cp, sp, nbad = oracle.mixer_update(**c)
    assert nbad == 2
    assert np.all(y[1] == 0) and np.all(y[2] == 0)
    np.testing.assert_array_equal(cp[2], c["conv_pool"][2])
    assert not np.array_equal(cp[0], c["conv_pool"][0])


def test_update_does_not_depend_on_thread_count():
    g = np.random.default_rng(41)
    c = _decode_case(g, Bz=4, pool=6)
    r1 = oracle.mixer_update(nthreads=1, **c)
    r8 = oracle.mixer_update(nthreads=8, **c)
    for a, b in zip(r1[:3], r8[:3]):
        np.testing.assert_array_equal(a, b)


# ---------------------------------------------------------------------------
# conv backward with state
# ---------------------------------------------------------------------------

def test_conv_bwd_worked_example_k3(golden_dir):
    """The page's single-token check: dS = [w0 d, w1 d + q0], dx = [w2 d + q1]."""
    ex = json.load(open(os.path.join(golden_dir, "conv_state_examples.json")))["backward_examples"][0]
    K = ex["K"]
    x = np.array(ex["x"]).reshape(1, 1, 1)
    S = np.array(ex["S"]).reshape(1, 1, K - 1)
    w = np.array(ex["w"]).reshape(1, K)
    dy = np.array([ex["delta"]]).reshape(1, 1, 1)
    q = np.array(ex["q"]).reshape(1, 1, K - 1)
    dx, dS, dw, db = oracle.conv_state_bwd(x, w, np.array([ex["bias"]]), S, dy, q, apply_silu=False)
    assert dS.ravel().tolist() == ex["dS"]
    assert dx.ravel().tolist() == ex["dx"]
    assert dw.ravel().tolist() == ex["dw"]
    assert db.ravel().tolist() == [ex["dbias"]]


def _conv_loss(x, w, bias, S, dy, q, silu):
    u, F = oracle.conv_state_fwd(x, w, bias, S, silu)
    return float((u * dy).sum() + (F * q).sum())


@pytest.mark.parametrize("K,L,silu", [(4, 6, True), (4, 2, True), (3, 5, False), (2, 1, True)])
def test_conv_bwd_matches_finite_differences(K, L, silu):
    """Central differences of the forward oracle (a loss linear in u and F)."""
    r = np.random.default_rng(7 + K + L)
    Bz, D = 2, 3
    x = r.standard_normal((Bz, L, D))
    w = r.standard_normal((D, K))
    bias = r.standard_normal(D)
    S = r.standard_normal((Bz, D, K - 1))
    dy = r.standard_normal((Bz, L, D))
    q = r.standard_normal((Bz, D, K - 1))
    dx, dS, dw, db = oracle.conv_state_bwd(x, w, bias, S, dy, q, apply_silu=silu)
    eps = 1e-6
    for name, arr, grad in (("x", x, dx), ("S", S, dS), ("w", w, dw), ("bias", bias, db)):
        num = np.empty_like(arr)
        for idx in np.ndindex(arr.shape):
            keep = arr[idx]
            arr[idx] = keep + eps
            lp = _conv_loss(x, w, bias, S, dy, q, silu)
            arr[idx] = keep - eps
            lm = _conv_loss(x, w, bias, S, dy, q, silu)
            arr[idx] = keep
            num[idx] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(grad, num, rtol=1e-6, atol=1e-7, err_msg=name)


@pytest.mark.parametrize("split", [1, 2, 5])
def test_conv_bwd_chunked_equals_whole(split):
    """Segments A then B with S_B = F_A: B's dS is A's dF (the chunked-training
    section), and the pieces reassemble the whole sequence's gradient."""
    r = np.random.default_rng(11 + split)
    Bz, L, D, K = 2, 7, 3, 4
    x = r.standard_normal((Bz, L, D))
    w = r.standard_normal((D, K))
    bias = r.standard_normal(D)
    S = r.standard_normal((Bz, D, K - 1))
    dy = r.standard_normal((Bz, L, D))
    q = r.standard_normal((Bz, D, K - 1))
    dx, dS, dw, db = oracle.conv_state_bwd(x, w, bias, S, dy, q)
    xa, xb = x[:, :split], x[:, split:]
    _, FA = oracle.conv_state_fwd(xa, w, bias, S, True)
    dxb, dSb, dwb, dbb = oracle.conv_state_bwd(xb, w, bias, FA, dy[:, split:], q)
    dxa, dSa, dwa, dba = oracle.conv_state_bwd(xa, w, bias, S, dy[:, :split], dSb)
    np.testing.assert_allclose(np.concatenate([dxa, dxb], axis=1), dx, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dSa, dS, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dwa + dwb, dw, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dba + dbb, db, rtol=1e-12, atol=1e-12)


def test_conv_bwd_empty_sequence_passes_the_state_gradient():
    """L = 0: F = S, so dS = dF and no weight gradient."""
    r = np.random.default_rng(3)
    S = r.standard_normal((2, 3, 3))
    q = r.standard_normal((2, 3, 3))
    dx, dS, dw, db = oracle.conv_state_bwd(np.zeros((2, 0, 3)), r.standard_normal((3, 4)),
                                           np.zeros(3), S, np.zeros((2, 0, 3)), q)
    np.testing.assert_array_equal(dS, q)
    assert not dw.any() and not db.any() and dx.shape == (2, 0, 3)


# ---------------------------------------------------------------------------
# scan backward with state
# ---------------------------------------------------------------------------

def _scan_problem(seed, Bz=2, L=7, H=4, P=3, N=5, G=2):
    r = np.random.default_rng(seed)
    u = r.standard_normal((Bz, L, H, P))
    dt = np.log1p(np.exp(r.standard_normal((Bz, L, H)) - 1.0))
    A = -r.uniform(0.1, 1.0, H)
    B = r.standard_normal((Bz, L, G, N))
    C = r.standard_normal((Bz, L, G, N))
    h0 = r.standard_normal((Bz, H, P, N))
    dy = r.standard_normal((Bz, L, H, P))
    dhT = r.standard_normal((Bz, H, P, N))
    return u, dt, A, B, C, h0, dy, dhT


def _scan_loss(u, dt, A, B, C, h0, dy, dhT):
    y, hT = oracle.ssm_scan(u, dt, A, B, C, h0)
    return float((y * dy).sum() + (hT * dhT).sum())


@pytest.mark.parametrize("name", ["u", "dt", "A", "B", "C", "h0"])
def test_scan_bwd_matches_finite_differences(name):
    """Every gradient against central differences of the (separately pinned)
    forward, for the linear loss <dy, y> + <dhT, hT>."""
    args = list(_scan_problem(11))
    names = ["u", "dt", "A", "B", "C", "h0"]
    du, ddt, dA, dB, dC, dh0 = oracle.ssm_scan_bwd(*args)
    grad = dict(zip(names, (du, ddt, dA, dB, dC, dh0)))[name]
    i = names.index(name)
    x0 = args[i]
    fd = np.zeros_like(x0)
    eps = 1e-6
    for idx in np.ndindex(x0.shape):
        xp = x0.copy(); xp[idx] += eps
        xm = x0.copy(); xm[idx] -= eps
        args[i] = xp; lp = _scan_loss(*args)
        args[i] = xm; lm = _scan_loss(*args)
        fd[idx] = (lp - lm) / (2 * eps)
    args[i] = x0
    np.testing.assert_allclose(grad, fd, rtol=1e-6, atol=1e-6)


def test_scan_bwd_initial_state_closed_form():
    """Eq. (4): the h0 term of y_t is exp(Lam_t) C_t^T h0 and that of hT is
    exp(Lam_{L-1}) h0, so dh0 = exp(Lam_{L-1}) dhT + sum_t exp(Lam_t) dy_t C_t^T,
    Lam_t the inclusive sum of dt_s A_h."""
    u, dt, A, B, C, h0, dy, dhT = _scan_problem(12)
    Bz, L, H, P = u.shape
    G = B.shape[2]
    *_, dh0 = oracle.ssm_scan_bwd(u, dt, A, B, C, h0, dy, dhT)
    lam = np.cumsum(dt * A[None, None, :], axis=1)           # [Bz, L, H]
    g_of_h = np.arange(H) // (H // G)
    Ch = C[:, :, g_of_h, :]                                  # [Bz, L, H, N]
    ref = (np.exp(lam[:, -1])[:, :, None, None] * dhT
           + np.einsum("blh,blhp,blhn->bhpn", np.exp(lam), dy, Ch))
    np.testing.assert_allclose(dh0, ref, rtol=1e-12, atol=1e-12)


def test_scan_bwd_no_decay_closed_forms():
    """A = 0 (a_t = 1): h_t = h0 + sum_{s<=t} x_s B_s^T, so
    dx_s = sum_{t>=s} (C_t . B_s) dy_t + dhT B_s and
    dC_t = (h0 + sum_{s<=t} x_s B_s^T)^T dy_t."""
    u, dt, A, B, C, h0, dy, dhT = _scan_problem(13, G=1)
    A = np.zeros_like(A)
    du, ddt, dA, dB, dC, dh0 = oracle.ssm_scan_bwd(u, dt, A, B, C, h0, dy, dhT)
    Bz, L, H, P = u.shape
    B1, C1 = B[:, :, 0], C[:, :, 0]                          # [Bz, L, N]
    later = np.triu(np.ones((L, L)))                         # [s, t]: t >= s
    GCB = np.einsum("btn,bsn->bst", C1, B1) * later          # (C_t . B_s), t >= s
    ref_dx = np.einsum("bst,bthp->bshp", GCB, dy) + np.einsum("bhpn,bsn->bshp", dhT, B1)
    np.testing.assert_allclose(du, ref_dx, rtol=1e-11, atol=1e-11)
    upto = np.tril(np.ones((L, L)))                          # [t, s]: s <= t
    hs = h0[:, None] + np.einsum("ts,bshp,bsn->bthpn", upto, u, B1)
    ref_dC = np.einsum("bthpn,bthp->btn", hs, dy)[:, :, None, :]
    np.testing.assert_allclose(dC, ref_dC, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(ddt, 0.0, atol=1e-12)        # dl_t times A_h = 0


@pytest.mark.parametrize("split", [1, 3, 6])
def test_scan_bwd_segments_equal_whole(split):
    """Truncated backpropagation made exact: segment B's dh0, fed to segment A
    as its dhT (A's final state is B's initial state), gives the whole
    sequence's gradients."""
    u, dt, A, B, C, h0, dy, dhT = _scan_problem(14)
    whole = oracle.ssm_scan_bwd(u, dt, A, B, C, h0, dy, dhT)
    sl_a, sl_b = slice(0, split), slice(split, None)
    _, hA = oracle.ssm_scan(u[:, sl_a], dt[:, sl_a], A, B[:, sl_a], C[:, sl_a], h0)
    gb = oracle.ssm_scan_bwd(u[:, sl_b], dt[:, sl_b], A, B[:, sl_b], C[:, sl_b], hA, dy[:, sl_b], dhT)
    ga = oracle.ssm_scan_bwd(u[:, sl_a], dt[:, sl_a], A, B[:, sl_a], C[:, sl_a], h0, dy[:, sl_a], gb[5])
    for k in (0, 1, 3, 4):  # du, ddt, dB, dC: per token
        np.testing.assert_allclose(np.concatenate([ga[k], gb[k]], axis=1), whole[k],
                                   rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(ga[2] + gb[2], whole[2], rtol=1e-11, atol=1e-11)  # dA
    np.testing.assert_allclose(ga[5], whole[5], rtol=1e-11, atol=1e-11)          # dh0


def test_scan_bwd_empty_sequence():
    """L = 0: hT = h0, so dh0 = dhT and dA = 0."""
    u, dt, A, B, C, h0, dy, dhT = _scan_problem(15, L=0)
    du, ddt, dA, dB, dC, dh0 = oracle.ssm_scan_bwd(u, dt, A, B, C, h0, dy, dhT)
    np.testing.assert_array_equal(dh0, dhT)
    assert not dA.any() and du.shape[1] == 0


# ---------------------------------------------------------------------------
# state-passing training utilities
# ---------------------------------------------------------------------------

def test_state_reset_rows():
    """A row restarts from zero when its draw is below p (p = 0.1 on the
    pages); 1000 evenly spaced draws reset exactly 100 rows."""
    u = (np.arange(1000) + 0.5) / 1000.0
    h = np.ones((1000, 2, 3, 4))
    c = np.full((1000, 6, 3), 2.0)
    h2, c2 = oracle.state_reset(u, 0.1, h, c)
    zeroed = np.all(h2.reshape(1000, -1) == 0, axis=1)
    assert zeroed.sum() == 100 and np.all(zeroed[:100]) and not zeroed[100:].any()
    np.testing.assert_array_equal(np.all(c2.reshape(1000, -1) == 0, axis=1), zeroed)
    np.testing.assert_array_equal(c2[100:], c[100:])


def test_fitted_noise_weights_follow_eqs_5_6():
    """Eqs. (5)-(6): mu <- 0.9 Mean(hT) + 0.1 mu, var <- 0.9 Var(hT) + 0.1 var
    (the new statistic weighs 1 - beta = 0.9).  Head 0 holds +-3 in equal
    numbers (mean 0, population variance 9), head 1 the constant 2."""
    hT = np.zeros((2, 2, 4, 6))
    hT[:, 0] = 3.0
    hT[:, 0, :2] = -3.0
    hT[:, 1] = 2.0
    m, v = oracle.fitted_noise_update(hT)
    np.testing.assert_allclose(m, [0.0, 2.0], atol=1e-15)
    np.testing.assert_allclose(v, [9.0, 0.0], atol=1e-15)
    m2, v2 = oracle.fitted_noise_update(hT, mu=np.array([10.0, -10.0]), var=np.array([1.0, 5.0]))
    np.testing.assert_allclose(m2, [0.9 * 0.0 + 0.1 * 10.0, 0.9 * 2.0 - 0.1 * 10.0], rtol=1e-15)
    np.testing.assert_allclose(v2, [0.9 * 9.0 + 0.1 * 1.0, 0.1 * 5.0], rtol=1e-15)


def test_fitted_noise_sample_moments():
    """h0 = mu_h + sqrt(var_h) eps: eps = +-1 gives mu +- sigma exactly, and a
    large standard-normal draw reproduces the per-head mean and variance."""
    mu, var = np.array([0.5, -1.0]), np.array([4.0, 0.25])
    e = np.ones((1, 2, 1, 1))
    np.testing.assert_allclose(oracle.fitted_noise_sample(mu, var, e).reshape(2), mu + np.sqrt(var))
    np.testing.assert_allclose(oracle.fitted_noise_sample(mu, var, -e).reshape(2), mu - np.sqrt(var))
    eps = np.random.default_rng(50).standard_normal((64, 2, 16, 32))
    h0 = oracle.fitted_noise_sample(mu, var, eps)
    n = 64 * 16 * 32
    for hh in range(2):
        x = h0[:, hh].ravel()
        assert abs(x.mean() - mu[hh]) < 5 * np.sqrt(var[hh] / n)
        assert abs(x.var() / var[hh] - 1.0) < 5 * np.sqrt(2.0 / n)


@pytest.mark.parametrize("stride", [1, 4, 7, 50])
def test_state_std_trace_matches_scan_prefixes(stride):
    """The diagnostic at each sampled position equals the standard deviation
    of the (separately pinned) scan's final state over that prefix."""
    u, dt, A, B, C, h0, _, _ = _scan_problem(21, L=13)
    tr = oracle.state_std_trace(u, dt, A, B, C, h0, stride)
    Bz, L, H, P = u.shape
    ends = [t for t in range(L) if (t + 1) % stride == 0 or t == L - 1]
    assert tr.shape == (Bz, len(ends), H)
    for k, t in enumerate(ends):
        _, hT = oracle.ssm_scan(u[:, :t + 1], dt[:, :t + 1], A, B[:, :t + 1], C[:, :t + 1], h0)
        np.testing.assert_allclose(tr[:, k], hT.reshape(Bz, H, -1).std(axis=2), rtol=1e-12)


# ---------------------------------------------------------------------------
# prefill into the pool
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("circular", [True, False])
def test_prefill_to_pool_example(circular):
    """K = 3, S_len = 4, prompt x = [a, b, c, d, e] after a zero state: the
    newest four inputs b, c, d, e; circular at length 5 they sit at slots
    1, 2, 3, 0 (row [e, b, c, d]), non-circular oldest first ([b, c, d, e])."""
    x = np.array([1.0, 10.0, 100.0, 1000.0, 10000.0]).reshape(1, 5, 1)
    cp, _, bad = oracle.prefill_to_pool(x, None, 3, None, np.zeros((1, 1, 4)), None,
                                        np.array([5]) if circular else None, None)
    assert bad == 0
    expect = [10000.0, 10.0, 100.0, 1000.0] if circular else [10.0, 100.0, 1000.0, 10000.0]
    np.testing.assert_array_equal(cp.reshape(-1), expect)


@pytest.mark.parametrize("circular", [True, False])
@pytest.mark.parametrize("L,Lnew,S_len,K", [(9, 3, 4, 4), (2, 4, 6, 4), (1, 1, 3, 4), (7, 6, 4, 3)])
def test_prefill_then_update_equals_whole_forward(circular, L, Lnew, S_len, K):
    """A prompt's forward, its state written into the pool, then a decode
    update on the next tokens, equals the forward over the whole sequence
    (the prompt's initial conv and SSM states included)."""
    g = np.random.default_rng(80 + L + 10 * Lnew)
    Bz, pool, H, P, N, G = 3, 5, 2, 3, 4, 1
    D = H * P
    x = g.standard_normal((Bz, L + Lnew, D))
    w, bias = g.standard_normal((D, K)), g.standard_normal(D)
    S0 = g.standard_normal((Bz, D, K - 1))
    h0 = g.standard_normal((Bz, H, P, N))
    dt = np.log1p(np.exp(g.standard_normal((Bz, L + Lnew, H))))
    A = -g.uniform(0.01, 1, H)
    B = g.standard_normal((Bz, L + Lnew, G, N))
    C = g.standard_normal((Bz, L + Lnew, G, N))
    idx = g.permutation(pool)[:Bz].astype(np.int32)
    y_all, _, _ = oracle.mixer_fwd(x, dt, A, B, C, w, bias, S0, h0)
    pre = slice(0, L)
    _, _, hT = oracle.mixer_fwd(x[:, pre], dt[:, pre], A, B[:, pre], C[:, pre], w, bias, S0, h0)
    lens = np.full(Bz, L + 7, np.int32) if circular else None   # any length >= L works
    cp, sp, bad = oracle.prefill_to_pool(x[:, pre], S0, K, hT, g.standard_normal((pool, D, S_len)),
                                         g.standard_normal((pool, H, P, N)), lens, idx)
    assert bad == 0
    post = slice(L, None)
    y, _, _, nbad = oracle.mixer_update(x[:, post], w, bias, cp, lens, idx, dt[:, post], A,
                                        B[:, post], C[:, post], sp)
    assert nbad == 0
    np.testing.assert_allclose(y, y_all[:, post], rtol=1e-10, atol=1e-10)


# ---------------------------------------------------------------------------
# packed sequences in the conv
# ---------------------------------------------------------------------------

def test_packed_conv_does_not_read_across_samples():
    """Samples A = [a1, a2] and B = [b1, b2] packed in one row, K = 3: B's
    first token must not read A's end; one-hot weights pick each tap."""
    x = np.array([1.0, 10.0, 100.0, 1000.0]).reshape(1, 4, 1)
    ids = np.array([[0, 0, 1, 1]])
    got = []
    for k in range(3):
        w = np.zeros((1, 3)); w[0, k] = 1.0
        out, _ = oracle.conv_state_fwd_packed(x, w, None, None, ids, apply_silu=False)
        got.append(out[0, :, 0])
    got = np.array(got)                           # [tap k, token t]
    # token t, tap k reads position t + k - 2 (0 before the row start)
    np.testing.assert_array_equal(got[:, 2], [0.0, 0.0, 100.0])      # b1 alone
    np.testing.assert_array_equal(got[:, 3], [0.0, 100.0, 1000.0])   # b2 reads b1 only
    np.testing.assert_array_equal(got[:, 1], [0.0, 1.0, 10.0])       # a2 reads a1


def test_packed_conv_reused_id_is_not_a_reset():
    """Ids A, B, A: equality alone lets the second A read the first A's input
    (the page's caveat about reused ids)."""
    x = np.array([1.0, 10.0, 100.0]).reshape(1, 3, 1)
    w = np.array([[1.0, 0.0, 0.0]])               # tap 0: position t - 2
    out, _ = oracle.conv_state_fwd_packed(x, w, None, None, np.array([[0, 1, 0]]), apply_silu=False)
    assert out[0, 2, 0] == 1.0


@pytest.mark.parametrize("bounds", [[5], [2, 9], [1, 2, 3], []])
def test_packed_conv_equals_separate_samples(bounds):
    """A packed row equals the samples run one by one: the first continues
    from the state S, every later one starts from a zero state; F is the
    row's last K-1 inputs."""
    g = np.random.default_rng(90 + len(bounds))
    Bz, L, D, K = 2, 12, 5, 4
    x = g.standard_normal((Bz, L, D))
    w, bias, S = g.standard_normal((D, K)), g.standard_normal(D), g.standard_normal((Bz, D, K - 1))
    ids = np.zeros((Bz, L), np.int64)
    for i, s in enumerate(bounds):
        ids[:, s:] = i + 1
    out, F = oracle.conv_state_fwd_packed(x, w, bias, S, ids)
    edges = [0] + bounds + [L]
    for i in range(len(edges) - 1):
        sl = slice(edges[i], edges[i + 1])
        ref, _ = oracle.conv_state_fwd(x[:, sl], w, bias, S if i == 0 else None)
        np.testing.assert_allclose(out[:, sl], ref, rtol=1e-13, atol=1e-13)
    _, F_plain = oracle.conv_state_fwd(x, w, bias, S)
    np.testing.assert_array_equal(F, F_plain)


@pytest.mark.parametrize("bounds", [[3], [1, 2, 9], []])
def test_packed_scan_equals_separate_samples(bounds):
    """A packed row equals its samples scanned one by one (the first from h0,
    the others from zero), and agrees with the unpacked scan without
    boundaries."""
    u, dt, A, B, C, h0, _, _ = _scan_problem(95 + len(bounds), L=12)
    Bz, L = dt.shape[:2]
    ids = np.zeros((Bz, L), np.int64)
    for i, s in enumerate(bounds):
        ids[:, s:] = 5 * (i + 1)
    y, hT = oracle.ssm_scan_packed(u, dt, A, B, C, h0, ids)
    edges = [0] + bounds + [L]
    for i in range(len(edges) - 1):
        sl = slice(edges[i], edges[i + 1])
        yr, hr = oracle.ssm_scan(u[:, sl], dt[:, sl], A, B[:, sl], C[:, sl], h0 if i == 0 else None)
        np.testing.assert_allclose(y[:, sl], yr, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(hT, hr, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# the full Mamba-2 mixer wiring (xBC conv, dt bias + softplus, dt-scaled input,
# D skip, SiLU(z) gate)
# ---------------------------------------------------------------------------

def _m2_inputs(seed, Bz=2, L=13, H=4, P=3, N=5, G=2, K=4, gate=True):
    r = np.random.default_rng(seed)
    D = H * P
    Dt = D + 2 * G * N
    return dict(
        xBC=r.standard_normal((Bz, L, Dt)),
        z=r.standard_normal((Bz, L, D)) if gate else None,
        dt_raw=r.standard_normal((Bz, L, H)) - 2.0,
        dt_bias=r.uniform(-1.0, 1.0, H),
        A=-r.uniform(0.01, 1.0, H),
        D_skip=r.standard_normal(H),
        w=r.standard_normal((Dt, K)) * np.sqrt(0.5),
        bias=np.full(Dt, 0.1),
        conv_state=r.standard_normal((Bz, Dt, K - 1)),
        h0=r.normal(0.0, 0.1, (Bz, H, P, N)),
        H=H, G=G, N=N)


def test_mamba2_zero_gate_gives_zero_output():
    """SiLU(0) = 0: with z = 0 the gated output is exactly zero while the
    state still advances."""
    a = _m2_inputs(1)
    a["z"] = np.zeros_like(a["z"])
    y, _, hT = oracle.mamba2_mixer_fwd(**a)
    assert np.all(y == 0.0)
    _, _, hT_nogate = oracle.mamba2_mixer_fwd(**dict(a, z=None))
    np.testing.assert_array_equal(hT, hT_nogate)


def test_mamba2_equals_plain_scan_of_the_conv_channels():
    """With the conv output split into x, B and C and dt = softplus(dt_raw +
    dt_bias) (numpy logaddexp), the wiring equals the plain scan oracle fed
    x, dt, A, dt-scaled B (one head per group, so dt_t B_t is that head's)
    and C, plus D_h x, times SiLU(z)."""
    a = _m2_inputs(2, H=4, G=4)
    Bz, L, Dt = a["xBC"].shape
    H, G, N = a["H"], a["G"], a["N"]
    D = Dt - 2 * G * N
    P = D // H
    y, F, hT = oracle.mamba2_mixer_fwd(**a)
    u, F_ref = oracle.conv_state_fwd(a["xBC"], a["w"], a["bias"], a["conv_state"])
    x = u[:, :, :D]
    Bm = u[:, :, D:D + G * N].reshape(Bz, L, G, N)
    Cm = u[:, :, D + G * N:].reshape(Bz, L, G, N)
    dt = np.logaddexp(0.0, a["dt_raw"] + a["dt_bias"])          # [Bz, L, H]
    y_s, h_s = oracle.ssm_scan(x, dt, a["A"], Bm * dt[..., None], Cm, a["h0"])
    gate = silu(a["z"]).reshape(Bz, L, H, P)
    y_ref = (y_s + a["D_skip"][None, None, :, None] * x.reshape(Bz, L, H, P)) * gate
    np.testing.assert_allclose(y, y_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(hT, h_s, rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(F, F_ref)


def test_mamba2_dt_bias_shift_invariance():
    """Only dt_raw + dt_bias enters: shifting one by c and the other by -c
    changes nothing."""
    a = _m2_inputs(3)
    y0, _, h0 = oracle.mamba2_mixer_fwd(**a)
    c = 0.375
    y1, _, h1 = oracle.mamba2_mixer_fwd(**dict(a, dt_raw=a["dt_raw"] + c, dt_bias=a["dt_bias"] - c))
    np.testing.assert_allclose(y1, y0, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(h1, h0, rtol=1e-12, atol=1e-14)


def test_mamba2_skip_alone_when_b_channels_are_silent():
    """Zero conv weights and bias on the B channels make B = SiLU(0) = 0; from
    h0 = 0 the state stays zero and y = D_h x SiLU(z) (x the conv output)."""
    a = _m2_inputs(4)
    Bz, L, Dt = a["xBC"].shape
    G, N, H = a["G"], a["N"], a["H"]
    D = Dt - 2 * G * N
    a["w"][D:D + G * N] = 0.0
    a["bias"][D:D + G * N] = 0.0
    a["h0"] = np.zeros_like(a["h0"])
    y, _, hT = oracle.mamba2_mixer_fwd(**a)
    assert np.all(hT == 0.0)
    u, _ = oracle.conv_state_fwd(a["xBC"], a["w"], a["bias"], a["conv_state"])
    P = D // H
    y_ref = (a["D_skip"][None, None, :, None] * u[:, :, :D].reshape(Bz, L, H, P)
             * silu(a["z"]).reshape(Bz, L, H, P))
    np.testing.assert_allclose(y, y_ref, rtol=1e-13, atol=1e-15)


def test_mamba2_large_negative_dt_holds_the_state():
    """dt_raw -> -inf gives dt = softplus(.) -> 0: a = 1 and no input enters,
    so h_t = h0 and y_t = (h0 C_t + D_h x_t) SiLU(z_t)."""
    a = _m2_inputs(5)
    a["dt_raw"] = np.full_like(a["dt_raw"], -800.0)
    y, _, hT = oracle.mamba2_mixer_fwd(**a)
    np.testing.assert_array_equal(hT, a["h0"])
    Bz, L, Dt = a["xBC"].shape
    G, N, H = a["G"], a["N"], a["H"]
    D = Dt - 2 * G * N
    P = D // H
    u, _ = oracle.conv_state_fwd(a["xBC"], a["w"], a["bias"], a["conv_state"])
    Cm = u[:, :, D + G * N:].reshape(Bz, L, G, N)
    g_of_h = np.arange(H) // (H // G)
    hC = np.einsum("bhpn,blhn->blhp", a["h0"], Cm[:, :, g_of_h, :])
    y_ref = (hC + a["D_skip"][None, None, :, None] * u[:, :, :D].reshape(Bz, L, H, P)) \
        * silu(a["z"]).reshape(Bz, L, H, P)
    np.testing.assert_allclose(y, y_ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("cut", [1, 5, 12])
def test_mamba2_segment_equivalence(cut):
    """Whole sequence = first part then the rest from the passed conv state
    (over every xBC channel) and SSM state."""
    a = _m2_inputs(6)
    y, F, hT = oracle.mamba2_mixer_fwd(**a)
    sl = lambda v, s: None if v is None else v[:, s]
    first = dict(a, xBC=a["xBC"][:, :cut], z=sl(a["z"], slice(0, cut)),
                 dt_raw=a["dt_raw"][:, :cut])
    y1, F1, h1 = oracle.mamba2_mixer_fwd(**first)
    second = dict(a, xBC=a["xBC"][:, cut:], z=sl(a["z"], slice(cut, None)),
                  dt_raw=a["dt_raw"][:, cut:], conv_state=F1, h0=h1)
    y2, F2, h2 = oracle.mamba2_mixer_fwd(**second)
    np.testing.assert_allclose(np.concatenate([y1, y2], axis=1), y, rtol=1e-12, atol=1e-13)
    np.testing.assert_array_equal(F2, F)
    np.testing.assert_allclose(h2, hT, rtol=1e-12, atol=1e-14)
