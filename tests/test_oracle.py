"""Pins of the fp64 oracle against what the paper and the mathematics fix.

Every check here compares the oracle with something other than itself: closed
forms, invariants of eqs. 5-10 of "TANGO: Token-Aggregated Nonlinear Gating
Operators ...", an independent formulation (softmax with a null logit, cumulative
sums), or the pair-by-pair definition against the running-sum recurrence.
"""
import numpy as np
import pytest
from scipy.special import softmax

import oracle
from cross_token_gated_gb300 import synth

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def unit_heads(x, H):
    B, T, D = x.shape
    y = x.reshape(B, T, H, D // H)
    y = y / np.maximum(np.linalg.norm(y, axis=-1, keepdims=True), 1e-12)
    return y.reshape(B, T, D)


def rel(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


AGGS = [
    ("tango", lambda q, k, g, v, **kw: oracle.tango(q, k, g, v, **{x: y for x, y in kw.items()
                                                                    if x not in ("window", "phi_mode")})),
    ("wango_direct", oracle.wango_direct),
    ("wango_scan", oracle.wango_scan),
]


# --------------------------------------------------------------- (a) sum to one

@pytest.mark.parametrize("name,fn", AGGS)
@pytest.mark.parametrize("W", [1, 3, 16, 40])
@pytest.mark.parametrize("tau", [0.0, 1.0, 10.0, 20.0])
def test_weights_sum_to_one(name, fn, W, tau):
    """g == 1 gives gbar == 1: the normalised weights of eq. 5 sum to one (no null gate)."""
    B, T, H, dqk, m = 2, 37, 2, 8, 6
    q, k = rnd((B, T, dqk), 1), rnd((B, T, dqk), 2)
    g = np.ones((B, T, m))
    out = fn(q, k, g, None, H=H, tau=tau, window=W, phi_mode=0)
    np.testing.assert_allclose(out, 1.0, rtol=0, atol=1e-13)


@pytest.mark.parametrize("name,fn", AGGS)
def test_weights_with_null_sum_below_one(name, fn):
    """With the null gate, g == 1 gives gbar = 1 - alpha_null, alpha_null in (0, 1),
    and the null weight is the only deficit: gbar(b -> -inf) -> 1."""
    B, T, H, dqk, m = 1, 20, 2, 8, 4
    q, k = rnd((B, T, dqk), 3), rnd((B, T, dqk), 4)
    g = np.ones((B, T, m))
    out = fn(q, k, g, None, H=H, tau=5.0, window=4, null_bias=[0.5, -1.0])
    assert np.all(out < 1.0) and np.all(out > 0.0)
    out_far = fn(q, k, g, None, H=H, tau=5.0, window=4, null_bias=[-200.0, -200.0])
    np.testing.assert_allclose(out_far, 1.0, atol=1e-13)


# ----------------------------------------------------------------- (b) T = 1

@pytest.mark.parametrize("name,fn", AGGS)
def test_single_token_returns_its_gate(name, fn):
    """T = 1: the only visible source is the destination itself, so gbar_0 = g_0."""
    B, H, dqk, m = 3, 2, 8, 10
    q, k, g = rnd((B, 1, dqk), 5), rnd((B, 1, dqk), 6), rnd((B, 1, m), 7)
    out = fn(q, k, g, None, H=H, tau=10.0, window=1)
    np.testing.assert_allclose(out, g, rtol=1e-15, atol=0)
    v = rnd((B, 1, m), 8)
    np.testing.assert_allclose(fn(q, k, g, v, H=H, tau=10.0, window=1), g * v, rtol=1e-15)


@pytest.mark.parametrize("name,fn", AGGS)
def test_single_token_null_closed_form(name, fn):
    """T = 1, q = k: logit = tau, so gbar = g e^tau / (e^tau + e^b) (eq. 5 with n = 1)."""
    B, H, dqk, m = 1, 2, 8, 6
    q = rnd((B, 1, dqk), 9)
    g = rnd((B, 1, m), 10)
    tau, b = 3.0, np.array([0.7, -2.0])
    out = fn(q, q.copy(), g, None, H=H, tau=tau, window=1, null_bias=b)
    m_h = m // H
    for a in range(H):
        expect = g[..., a * m_h:(a + 1) * m_h] * np.exp(tau) / (np.exp(tau) + np.exp(b[a]))
        np.testing.assert_allclose(out[..., a * m_h:(a + 1) * m_h], expect, rtol=1e-14)


# ------------------------------------------------------- (c) W >= T is TANGO

@pytest.mark.parametrize("W", [12, 13, 100])
def test_wango_wide_window_is_tango(W):
    B, T, H, dqk, m = 2, 12, 2, 8, 6
    q, k, g, v = rnd((B, T, dqk), 11), rnd((B, T, dqk), 12), rnd((B, T, m), 13), rnd((B, T, m), 14)
    t = oracle.tango(q, k, g, v, H=H, tau=10.0, null_bias=[0.1, 0.2])
    d = oracle.wango_direct(q, k, g, v, H=H, tau=10.0, window=W, null_bias=[0.1, 0.2])
    s = oracle.wango_scan(q, k, g, v, H=H, tau=10.0, window=W, null_bias=[0.1, 0.2])
    assert np.array_equal(t, d)
    assert rel(s, t) < 1e-13


def test_wango_narrow_window_differs_from_tango():
    """Guard: the pins above are not vacuous (older sources change the result)."""
    B, T, H, dqk, m = 1, 12, 2, 8, 6
    q, k, g = rnd((B, T, dqk), 15), rnd((B, T, dqk), 16), rnd((B, T, m), 17)
    t = oracle.tango(q, k, g, None, H=H, tau=10.0)
    d = oracle.wango_direct(q, k, g, None, H=H, tau=10.0, window=3)
    assert rel(d, t) > 1e-3


# ------------------------------------------- (d) running sums == direct form

@pytest.mark.parametrize("W", [1, 2, 5, 16, 47, 48, 60])
@pytest.mark.parametrize("phi_mode", [0, 1])
@pytest.mark.parametrize("null", [None, [0.3, -0.4]])
def test_scan_matches_direct(W, phi_mode, null):
    B, T, H, dqk, m = 2, 48, 2, 16, 140   # m_h = 70 spans two 64-column work units
    q, k, g, v = rnd((B, T, dqk), 18), rnd((B, T, dqk), 19), rnd((B, T, m), 20), rnd((B, T, m), 21)
    kw = dict(H=H, tau=10.0, window=W, phi_mode=phi_mode, null_bias=null)
    assert rel(oracle.wango_scan(q, k, g, v, **kw), oracle.wango_direct(q, k, g, v, **kw)) < 1e-12


# --------------------------------------------------------- s = 0 closed forms

def test_tango_zero_scale_is_cumulative_mean():
    B, T, H, dqk, m = 2, 30, 2, 8, 6
    q, k, g = rnd((B, T, dqk), 22), rnd((B, T, dqk), 23), rnd((B, T, m), 24)
    expect = np.cumsum(g, axis=1) / np.arange(1, T + 1)[None, :, None]
    assert rel(oracle.tango(q, k, g, None, H=H, tau=0.0), expect) < 1e-13


@pytest.mark.parametrize("phi_mode", [0, 1])
@pytest.mark.parametrize("W", [1, 4, 9])
def test_wango_zero_scale_closed_form(phi_mode, W):
    """tau = 0: window weights are exp(0) = 1; older weights are phi(0).phi(0), which
    is (1 + 1e-4)^2 for eq. 8 and d_h for the literal elu + 1.  So gbar_i is a
    two-level weighted cumulative mean."""
    B, T, H, dqk, m = 1, 25, 2, 8, 6
    d_h = dqk // H
    c = (1.0 + 1e-4) ** 2 if phi_mode == 0 else float(d_h)
    q, k, g = rnd((B, T, dqk), 25), rnd((B, T, dqk), 26), rnd((B, T, m), 27)
    cs = np.concatenate([np.zeros((B, 1, m)), np.cumsum(g, axis=1)], axis=1)
    expect = np.empty_like(g)
    for i in range(T):
        lo = max(0, i - W + 1)
        num = (cs[:, i + 1] - cs[:, lo]) + c * cs[:, lo]
        expect[:, i] = num / ((i + 1 - lo) + c * lo)
    for fn in (oracle.wango_direct, oracle.wango_scan):
        assert rel(fn(q, k, g, None, H=H, tau=0.0, window=W, phi_mode=phi_mode), expect) < 1e-13


def _axis_heads(B, T, H, d_h, axis, sign):
    """Every token's head vector is sign * e_axis (already a unit vector)."""
    x = np.zeros((B, T, H, d_h))
    x[..., axis] = sign
    return x.reshape(B, T, H * d_h)


@pytest.mark.parametrize("phi_mode", [0, 1])
@pytest.mark.parametrize("W", [1, 2, 5])
def test_wango_phi_at_positive_scale_closed_form(phi_mode, W):
    """tau > 0 with q_hat = -e_0 and k_hat = e_1 in every head and token: every cosine is
    0, so each window weight is exp(0) = 1, and every older weight is the feature-map dot
    product of eqs. 8-9 at u = sqrt(tau) q_hat and w = sqrt(tau) k_hat, expanded here by
    hand (u_0 = -sqrt(tau) takes ELU's negative branch e^u - 1, w_1 = +sqrt(tau) the
    identity branch, every other coordinate is 0):
      eq. 8:  [(e^-r + eps)(1 + eps) + (1 + eps)(r + 1 + eps) + (d_h - 2)(1 + eps)^2] / d_h
      elu+1:   e^-r + (r + 1) + (d_h - 2)
    with r = sqrt(tau).  Two heads with different tau fix the per-head sqrt(tau); a
    scaled q/k fixes the unit normalisation in front of it."""
    B, T, H, d_h, m = 1, 7, 2, 4, 6
    eps = 1e-4
    taus = [10.0, 2.25]
    q = _axis_heads(B, T, H, d_h, 0, -3.0)     # normalised to -e_0 inside the oracle
    k = _axis_heads(B, T, H, d_h, 1, 0.5)      # normalised to +e_1
    g = rnd((B, T, m), 31)
    m_h = m // H
    expect = np.empty_like(g)
    for a, tau in enumerate(taus):
        r = np.sqrt(tau)
        if phi_mode == 0:
            c = ((np.exp(-r) + eps) * (1 + eps) + (1 + eps) * (r + 1 + eps)
                 + (d_h - 2) * (1 + eps) ** 2) / d_h
        else:
            c = np.exp(-r) + (r + 1) + (d_h - 2)
        ga = g[..., a * m_h:(a + 1) * m_h]
        for i in range(T):
            lo = max(0, i - W + 1)
            num = ga[:, lo:i + 1].sum(axis=1) + c * ga[:, :lo].sum(axis=1)
            expect[:, i, a * m_h:(a + 1) * m_h] = num / ((i + 1 - lo) + c * lo)
    for fn in (oracle.wango_direct, oracle.wango_scan):
        got = fn(q, k, g, None, H=H, tau=taus, window=W, phi_mode=phi_mode)
        assert rel(got, expect) < 1e-13
    # the older weight differs from both the window weight and the tau = 0 weight, so
    # the case really exercises it
    assert W < T


def test_wango_phi_negative_branch_pin():
    """One more hand value for ELU's negative branch: q_hat = -e_0, k_hat = -e_0 (cosine
    1, so the window weight is e^tau), tau = 4, d_h = 4, eq. 8.  The older weight is
    [(e^-2 + eps)^2 + 3 (1 + eps)^2] / 4 (both vectors on the negative branch)."""
    B, T, H, d_h, m = 1, 3, 1, 4, 2
    eps, tau = 1e-4, 4.0
    q = _axis_heads(B, T, H, d_h, 0, -1.0)
    k = _axis_heads(B, T, H, d_h, 0, -1.0)
    g = rnd((B, T, m), 32)
    c = ((np.exp(-2.0) + eps) ** 2 + 3 * (1 + eps) ** 2) / 4
    wwin = np.exp(tau)
    # W = 1: row 2 has source 2 in the window and sources 0, 1 older
    expect2 = (wwin * g[0, 2] + c * (g[0, 0] + g[0, 1])) / (wwin + 2 * c)
    for fn in (oracle.wango_direct, oracle.wango_scan):
        got = fn(q, k, g, None, H=H, tau=tau, window=1, phi_mode=0)
        assert rel(got[0, 2], expect2) < 1e-13


def test_phi_mode_readings_differ():
    """Guard: the eq. 8 feature map and the literal elu + 1 are different rules."""
    B, T, H, dqk, m = 1, 10, 2, 8, 4
    q, k, g = rnd((B, T, dqk), 28), rnd((B, T, dqk), 29), rnd((B, T, m), 30)
    a = oracle.wango_direct(q, k, g, None, H=H, tau=10.0, window=2, phi_mode=0)
    b = oracle.wango_direct(q, k, g, None, H=H, tau=10.0, window=2, phi_mode=1)
    assert rel(a, b) > 1e-3


# ------------------------------------------ eq. 6 as a softmax with a null logit

def test_tango_is_softmax_with_null_logit():
    """Eq. 6 in eq. 5 equals a softmax over the logits tau q.k and the null logit
    b + log n_i (sec. 2.2), evaluated here with scipy's softmax."""
    B, T, H, dqk, m = 1, 9, 2, 8, 6
    d_h, m_h = dqk // H, m // H
    q, k, g = rnd((B, T, dqk), 31), rnd((B, T, dqk), 32), rnd((B, T, m), 33)
    tau, nb = 7.0, np.array([0.4, -0.3])
    out = oracle.tango(q, k, g, None, H=H, tau=tau, null_bias=nb)
    qn, kn = unit_heads(q, H), unit_heads(k, H)
    for a in range(H):
        sl, gl = slice(a * d_h, (a + 1) * d_h), slice(a * m_h, (a + 1) * m_h)
        for i in range(T):
            logits = tau * kn[0, :i + 1, sl] @ qn[0, i, sl]
            p = softmax(np.append(logits, nb[a] + np.log(i + 1)))
            np.testing.assert_allclose(out[0, i, gl], p[:-1] @ g[0, :i + 1, gl], rtol=1e-12)


# ------------------------------------------------------------ structural pins

@pytest.mark.parametrize("name,fn", AGGS)
def test_causality(name, fn):
    """Changing any source after i leaves gbar_i bit-identical."""
    B, T, H, dqk, m = 1, 20, 2, 8, 6
    q, k, g = rnd((B, T, dqk), 34), rnd((B, T, dqk), 35), rnd((B, T, m), 36)
    base = fn(q, k, g, None, H=H, tau=10.0, window=5)
    cut = 11
    q2, k2, g2 = q.copy(), k.copy(), g.copy()
    q2[:, cut + 1:] += 3.0
    k2[:, cut + 1:] -= 2.0
    g2[:, cut + 1:] *= -5.0
    pert = fn(q2, k2, g2, None, H=H, tau=10.0, window=5)
    assert np.array_equal(base[:, :cut + 1], pert[:, :cut + 1])
    assert not np.array_equal(base[:, cut + 1:], pert[:, cut + 1:])


@pytest.mark.parametrize("name,fn", AGGS)
def test_linear_in_gates_and_features(name, fn):
    """diag(gbar) is a weighted average of diag(g_j) (sec. 2.1): gbar is linear in g,
    and the output gbar * v is linear in v."""
    B, T, H, dqk, m = 1, 16, 2, 8, 6
    q, k = rnd((B, T, dqk), 37), rnd((B, T, dqk), 38)
    g1, g2, v1, v2 = rnd((B, T, m), 39), rnd((B, T, m), 40), rnd((B, T, m), 41), rnd((B, T, m), 42)
    kw = dict(H=H, tau=10.0, window=4, null_bias=[0.0, 1.0])
    lhs = fn(q, k, 2.0 * g1 - 3.0 * g2, None, **kw)
    rhs = 2.0 * fn(q, k, g1, None, **kw) - 3.0 * fn(q, k, g2, None, **kw)
    assert rel(lhs, rhs) < 1e-12
    lhs = fn(q, k, g1, 0.5 * v1 + v2, **kw)
    rhs = 0.5 * fn(q, k, g1, v1, **kw) + fn(q, k, g1, v2, **kw)
    assert rel(lhs, rhs) < 1e-12


def test_tango_identical_keys_is_cumulative_mean():
    """All keys equal: every visible source gets the same weight for any q and tau."""
    B, T, H, dqk, m = 1, 18, 2, 8, 6
    q, g = rnd((B, T, dqk), 43), rnd((B, T, m), 44)
    k = np.broadcast_to(rnd((1, 1, dqk), 45), (B, T, dqk)).copy()
    expect = np.cumsum(g, axis=1) / np.arange(1, T + 1)[None, :, None]
    assert rel(oracle.tango(q, k, g, None, H=H, tau=20.0), expect) < 1e-12


def test_normalisation_scale_invariance():
    """Queries/keys are unit-normalised (sec. 2.1): rescaling them changes nothing,
    and passing pre-normalised vectors with qk_normalized gives the same result."""
    B, T, H, dqk, m = 1, 14, 2, 8, 6
    q, k, g = rnd((B, T, dqk), 46), rnd((B, T, dqk), 47), rnd((B, T, m), 48)
    base = oracle.tango(q, k, g, None, H=H, tau=10.0)
    assert rel(oracle.tango(3.7 * q, 0.2 * k, g, None, H=H, tau=10.0), base) < 1e-13
    pre = oracle.tango(unit_heads(q, H), unit_heads(k, H), g, None, H=H, tau=10.0,
                       qk_normalized=True)
    assert rel(pre, base) < 1e-13


@pytest.mark.parametrize("name,fn", AGGS)
def test_heads_and_batches_independent(name, fn):
    B, T, H, dqk, m = 3, 15, 2, 8, 6
    q, k, g, v = rnd((B, T, dqk), 49), rnd((B, T, dqk), 50), rnd((B, T, m), 51), rnd((B, T, m), 52)
    kw = dict(H=H, tau=10.0, window=4)
    base = fn(q, k, g, v, **kw)
    d_h, m_h = dqk // H, m // H
    swap_qk = np.r_[d_h:dqk, 0:d_h]
    swap_g = np.r_[m_h:m, 0:m_h]
    sw = fn(q[..., swap_qk], k[..., swap_qk], g[..., swap_g], v[..., swap_g], **kw)
    assert np.array_equal(sw, base[..., swap_g])
    one = fn(q[1:2], k[1:2], g[1:2], v[1:2], **kw)
    assert np.array_equal(one, base[1:2])


@pytest.mark.parametrize("which", ["tango", "wango"])
def test_row_sampling_matches_full(which):
    B, T, H, dqk, m = 2, 21, 2, 8, 6
    q, k, g, v = rnd((B, T, dqk), 53), rnd((B, T, dqk), 54), rnd((B, T, m), 55), rnd((B, T, m), 56)
    rows = [0, 5, 20, 21, 33, 41]
    if which == "tango":
        full = oracle.tango(q, k, g, v, H=H, tau=10.0)
        samp = oracle.tango(q, k, g, v, H=H, tau=10.0, rows=rows)
    else:
        full = oracle.wango_direct(q, k, g, v, H=H, tau=10.0, window=3)
        samp = oracle.wango_direct(q, k, g, v, H=H, tau=10.0, window=3, rows=rows)
    assert np.array_equal(samp, full.reshape(B * T, m)[rows])


def test_bf16_inputs_widen_exactly():
    """bf16 bit patterns are widened exactly: the oracle on raw bf16 equals the
    oracle on the same values given as float64."""
    q, k, g, v = synth.agg_inputs(1, 10, 8, 6, seed=3, dtype="bf16")
    raw = [synth.oracle_view(t) for t in (q, k, g, v)]
    wide = [t.double().numpy() for t in (q, k, g, v)]
    a = oracle.tango(*raw, H=2, tau=10.0)
    b = oracle.tango(*wide, H=2, tau=10.0)
    assert np.array_equal(a, b)


# ------------------------------------------------------------ block forward

def _block_np(T, d, dqk, m, seed):
    h, w = synth.block_inputs(1, T, d, dqk, m, seed=seed, dtype="f32")
    return h.double().numpy(), {n: t.double().numpy() for n, t in w.items()}


@pytest.mark.parametrize("mode", [0, 1])
def test_block_single_token_expansion(mode):
    """T = 1 (sec. 2.1 special case): gbar = g, so h+ = h + W_o(SiLU(W_g x) * W_v x)
    with x = RMSNorm(h), written here with numpy matrix products."""
    d, dqk, m, H = 16, 8, 12, 2
    h, w = _block_np(1, d, dqk, m, 60)
    w["gamma"] = 1.0 + 0.1 * rnd(d, 61)
    out = oracle.block_forward(h, w, H=H, tau=10.0, mode=mode, window=1, rms_eps=1e-6)
    x = w["gamma"] * h[0, 0] / np.sqrt(np.mean(h[0, 0] ** 2) + 1e-6)
    a = w["Wg"] @ x
    expect = h[0, 0] + w["Wo"] @ ((a / (1.0 + np.exp(-a))) * (w["Wv"] @ x))
    np.testing.assert_allclose(out[0, 0], expect, rtol=1e-12, atol=1e-12)


def test_block_intermediates_consistent_with_aggregation():
    """The block's aggregation step is the standalone oracle applied to the block's
    own unit q/k, gates and features; h+ - h is W_o u (matrix product in numpy)."""
    T, d, dqk, m, H = 24, 16, 8, 12, 2
    h, w = _block_np(T, d, dqk, m, 62)
    for mode, W in ((0, 1), (1, 5)):
        out, it = oracle.block_forward(h, w, H=H, tau=10.0, mode=mode, window=W,
                                       intermediates=True)
        if mode == 0:
            u = oracle.tango(it["q"], it["k"], it["g"], it["v"], H=H, tau=10.0, qk_normalized=True)
        else:
            u = oracle.wango_scan(it["q"], it["k"], it["g"], it["v"], H=H, tau=10.0, window=W,
                                  qk_normalized=True)
        assert rel(it["u"], u) < 1e-12
        assert rel(out - h, it["u"] @ w["Wo"].T) < 1e-12
        np.testing.assert_allclose(np.linalg.norm(it["q"].reshape(1, T, H, -1), axis=-1), 1.0,
                                   rtol=1e-14)
        assert np.all(it["g"] > -0.2785)   # SiLU's minimum is about -0.27846


def test_block_rope_relative_position():
    """RoPE makes q_i.k_j depend on content and i - j only: with a periodic
    residual stream (period P), scores at (i, j) and (i + P, j + P) agree.  At
    position 0 the rotation is the identity."""
    P, T, d, dqk, m, H = 5, 15, 16, 8, 4, 2
    h, w = _block_np(P, d, dqk, m, 63)
    hp = np.concatenate([h] * (T // P), axis=1)
    _, on = oracle.block_forward(hp, w, H=H, tau=1.0, rope_base=10000.0, intermediates=True)
    _, off = oracle.block_forward(hp, w, H=H, tau=1.0, rope_base=0.0, intermediates=True)
    np.testing.assert_allclose(on["q"][0, 0], off["q"][0, 0], rtol=1e-14)
    d_h = dqk // H
    qh, kh = on["q"].reshape(T, H, d_h), on["k"].reshape(T, H, d_h)
    s = np.einsum("iac,jac->aij", qh, kh)
    for i in range(P, T - P):
        for j in range(i - P + 1):
            np.testing.assert_allclose(s[:, i, j], s[:, i + P, j + P], rtol=1e-10, atol=1e-12)
    assert not np.allclose(on["q"][0, 1], off["q"][0, 1])


def test_model_logits_one_hot_closed_form():
    """h_t = c e_k gives RMSNorm(h_t) = sign(c) sqrt(d) gamma_k e_k (eps = 0); with the
    one-hot tied matrix E[v] = e_(v mod d) the logit of v is that value when
    v mod d == k and 0 otherwise.  Pins the normaliser's sqrt(d), the gain's index and
    the orientation of E."""
    d, vocab = 8, 19
    E = np.zeros((vocab, d))
    E[np.arange(vocab), np.arange(vocab) % d] = 1.0
    gam = 1.0 + np.arange(d) / 10.0
    for k, c in ((3, 2.5), (6, -0.7)):
        h = np.zeros((1, d))
        h[0, k] = c
        got = oracle.final_logits(h, gam, E, rms_eps=0.0)[0]
        want = np.where(np.arange(vocab) % d == k, np.sign(c) * np.sqrt(d) * gam[k], 0.0)
        np.testing.assert_allclose(got, want, rtol=1e-14, atol=1e-14)


def test_model_logits_rmsnorm_scale_invariance():
    """Final RMSNorm then tied logits: logits(c * h) = logits(h) for eps -> 0, and
    logits equal RMSNorm(h) @ E^T (numpy matrix product)."""
    n, d, vocab = 6, 16, 20
    h = rnd((n, d), 64)
    E = rnd((vocab, d), 65)
    gam = 1.0 + 0.1 * rnd(d, 66)
    a = oracle.final_logits(h, gam, E, rms_eps=0.0)
    b = oracle.final_logits(5.0 * h, gam, E, rms_eps=0.0)
    assert rel(a, b) < 1e-13
    x = gam * h / np.sqrt(np.mean(h ** 2, axis=-1, keepdims=True))
    assert rel(a, x @ E.T) < 1e-13
    ids = np.array([[3, 0, 19]])
    np.testing.assert_array_equal(oracle.embed(ids, E), E[ids])


# ------------------------------------------------------------------ model forward

def _model_setup(n_sets, seed=70, d=16, H=2, dqk=8, m=12, vocab=11, B=2, T=7):
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, vocab, size=(B, T))
    E = 0.5 * rng.standard_normal((vocab, d))
    shared = {"gamma": 1.0 + 0.1 * rng.standard_normal(d), "Wq": rng.standard_normal((dqk, d)) / 4,
              "Wk": rng.standard_normal((dqk, d)) / 4}
    sets = [dict(shared, Wg=rng.standard_normal((m, d)) / 4, Wv=rng.standard_normal((m, d)) / 4,
                 Wo=rng.standard_normal((d, m)) / 4) for _ in range(n_sets)]
    gam_f = 1.0 + 0.1 * rng.standard_normal(d)
    return ids, E, gam_f, sets, H


def test_model_default_set_assignment():
    """The revision assigns three narrower gated-projection sets to the first, middle and
    last applications; one set serves every application."""
    assert oracle.default_sets(4, 3) == [0, 1, 1, 2]
    assert oracle.default_sets(8, 3) == [0, 1, 1, 1, 1, 1, 1, 2]
    assert oracle.default_sets(4, 1) == [0, 0, 0, 0]
    with pytest.raises(ValueError):
        oracle.default_sets(4, 2)


def test_model_zero_output_projection_is_identity():
    """W_o = 0 makes every application the identity (h_out = h + W_o u = h), so the model
    reduces to the final RMSNorm of the embeddings against the tied matrix."""
    ids, E, gam_f, sets, H = _model_setup(3)
    for w in sets:
        w["Wo"] = np.zeros_like(w["Wo"])
    got = oracle.model_forward(ids, E, gam_f, sets, H=H, tau=10.0)
    assert rel(got, oracle.final_logits(E[ids], gam_f, E)) < 1e-14


@pytest.mark.parametrize("live,apps", [(0, 1), (1, 2), (2, 1)])
def test_model_sets_applied_first_middle_last(live, apps):
    """With W_o zero in all sets but one, only the applications of that set act: set 0
    once (first), set 1 twice (the two middle applications of four), set 2 once (last)."""
    ids, E, gam_f, sets, H = _model_setup(3, seed=71)
    for s, w in enumerate(sets):
        if s != live:
            w["Wo"] = np.zeros_like(w["Wo"])
    got = oracle.model_forward(ids, E, gam_f, sets, H=H, tau=10.0, n_apps=4)
    h = E[ids]
    for _ in range(apps):
        h = oracle.block_forward(h, sets[live], H=H, tau=10.0)
    assert rel(got, oracle.final_logits(h, gam_f, E)) < 1e-13
    h1 = oracle.block_forward(E[ids], sets[live], H=H, tau=10.0)  # a different count is far off
    if apps != 1:
        assert rel(got, oracle.final_logits(h1, gam_f, E)) > 1e-3


def test_model_prefix_causality():
    """Positions before T' depend only on the first T' tokens (every step is causal), so
    the logits of a prefix run equal the leading rows of the full run."""
    ids, E, gam_f, sets, H = _model_setup(1, seed=72, T=9)
    full = oracle.model_forward(ids, E, gam_f, sets, H=H, tau=10.0, mode=1, window=3)
    pre = oracle.model_forward(ids[:, :4], E, gam_f, sets, H=H, tau=10.0, mode=1, window=3)
    assert rel(pre, full[:, :4]) < 1e-13
    changed = ids.copy()
    changed[:, 6] = (changed[:, 6] + 1) % E.shape[0]
    alt = oracle.model_forward(changed, E, gam_f, sets, H=H, tau=10.0, mode=1, window=3)
    assert rel(alt[:, :6], full[:, :6]) < 1e-13 and rel(alt[:, 6:], full[:, 6:]) > 1e-6
