"""Pins of the oracle's gradients (the derivative of eq. 5 of "TANGO: Token-Aggregated
Nonlinear Gating Operators ..." with TANGO and WANGO weights) against what does not
depend on their formulas:

- central finite differences of the forward oracle, whose own pins are in
  test_oracle.py: for L(x) = sum(dout * u(x)) and a random direction e in one input
  at a time, (L(x + h e) - L(x - h e)) / 2h must equal sum(grad * e);
- closed forms at tau = 0, where every weight is equal: dq = dk = 0 and
  dg_j = sum_{i >= j} dgbar_i / (i + 1) (TANGO);
- dv = dout * gbar, with gbar from the forward oracle.
"""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def forward(kind, q, k, g, v, kw):
    if kind == "tango":
        return oracle.tango(q, k, g, v, **{x: y for x, y in kw.items() if x not in ("window", "phi_mode")})
    return oracle.wango_direct(q, k, g, v, **kw)


def backward(kind, q, k, g, v, dout, kw):
    if kind == "tango":
        return oracle.tango_backward(q, k, g, v, dout, **{x: y for x, y in kw.items()
                                                          if x not in ("window", "phi_mode")})
    return oracle.wango_backward(q, k, g, v, dout, **kw)


CASES = [
    ("tango", dict(tau=10.0)),
    ("tango", dict(tau=[3.0, 12.0], null_bias=[0.3, -1.0])),
    ("wango", dict(tau=10.0, window=1, phi_mode=0)),
    ("wango", dict(tau=10.0, window=3, phi_mode=0)),
    ("wango", dict(tau=[4.0, 9.0], window=4, phi_mode=1, null_bias=[-0.5, 0.2])),
    ("wango", dict(tau=10.0, window=20, phi_mode=0)),     # W >= T: TANGO
]


@pytest.mark.parametrize("with_v", [True, False])
@pytest.mark.parametrize("qk_normalized", [False, True])
@pytest.mark.parametrize("kind,kw", CASES, ids=[f"{c[0]}{i}" for i, c in enumerate(CASES)])
def test_gradients_match_finite_differences(kind, kw, qk_normalized, with_v):
    B, T, H, dqk, m = 2, 9, 2, 8, 6
    q, k = rnd((B, T, dqk), 1), rnd((B, T, dqk), 2)
    if qk_normalized:   # unit vectors per head, as the flag promises
        for x in (q, k):
            y = x.reshape(B, T, H, -1)
            y /= np.linalg.norm(y, axis=-1, keepdims=True)
    g, v, dout = rnd((B, T, m), 3), (rnd((B, T, m), 4) if with_v else None), rnd((B, T, m), 5)
    kw = dict(kw, H=H, qk_normalized=qk_normalized)
    grads = backward(kind, q, k, g, v, dout, kw)
    inputs = {"q": q, "k": k, "g": g, "v": v}
    h = 1e-6
    for name, x in inputs.items():
        if x is None:
            assert grads["d" + name] is None
            continue
        if qk_normalized and name in ("q", "k"):
            continue   # the flag's inputs are constrained to the sphere; checked below
        e = rnd(x.shape, 6 + len(name))
        args = dict(inputs)
        args[name] = x + h * e
        lp = np.sum(dout * forward(kind, args["q"], args["k"], args["g"], args["v"], kw))
        args[name] = x - h * e
        lm = np.sum(dout * forward(kind, args["q"], args["k"], args["g"], args["v"], kw))
        fd = (lp - lm) / (2 * h)
        an = np.sum(grads["d" + name] * e)
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)
    if qk_normalized:
        # on the sphere: a tangent direction e (e . qhat = 0 per head) moves qhat to first
        # order, and the flag's gradient is the one with respect to qhat itself
        for name in ("q", "k"):
            x = inputs[name]
            e = rnd(x.shape, 9 + len(name)).reshape(B, T, H, -1)
            xh = x.reshape(B, T, H, -1)
            e -= xh * np.sum(e * xh, axis=-1, keepdims=True)
            e = e.reshape(x.shape)
            args = dict(inputs)
            vals = []
            for sgn in (1, -1):
                y = (x + sgn * h * e).reshape(B, T, H, -1)
                y = (y / np.linalg.norm(y, axis=-1, keepdims=True)).reshape(x.shape)
                args[name] = y
                vals.append(np.sum(dout * forward(kind, args["q"], args["k"], args["g"], args["v"], kw)))
            fd = (vals[0] - vals[1]) / (2 * h)
            an = np.sum(grads["d" + name] * e)
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)


@pytest.mark.parametrize("kind,kw", [("tango", {}), ("wango", dict(window=3, phi_mode=0)),
                                     ("wango", dict(window=2, phi_mode=1))])
def test_zero_scale_closed_forms(kind, kw):
    """tau = 0: every score is 0 whatever q and k are (and sqrt(tau) = 0 scales the
    feature-map arguments), so dq = dk = 0 exactly; for TANGO every weight is 1/(i+1) and
    dg_j = sum_{i >= j} dgbar_i / (i + 1)."""
    B, T, H, dqk, m = 1, 11, 2, 8, 4
    q, k, g, v, dout = rnd((B, T, dqk), 11), rnd((B, T, dqk), 12), rnd((B, T, m), 13), rnd((B, T, m), 14), \
        rnd((B, T, m), 15)
    d = backward(kind, q, k, g, v, dout, dict(kw, H=H, tau=0.0))
    assert np.all(d["dq"] == 0.0) and np.all(d["dk"] == 0.0)
    if kind == "tango":
        dgb = dout * v
        expect = np.flip(np.cumsum(np.flip(dgb / np.arange(1, T + 1)[None, :, None], axis=1), axis=1), axis=1)
        np.testing.assert_allclose(d["dg"], expect, rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("kind", ["tango", "wango"])
def test_dv_is_dout_times_gbar(kind):
    B, T, H, dqk, m = 2, 7, 2, 8, 6
    q, k, g, v, dout = rnd((B, T, dqk), 21), rnd((B, T, dqk), 22), rnd((B, T, m), 23), rnd((B, T, m), 24), \
        rnd((B, T, m), 25)
    kw = dict(H=H, tau=10.0, window=2, phi_mode=0)
    gbar = forward(kind, q, k, g, None, kw)
    d = backward(kind, q, k, g, v, dout, kw)
    np.testing.assert_allclose(d["dv"], dout * gbar, rtol=1e-13, atol=1e-15)


def test_gradients_are_linear_in_dout():
    B, T, H, dqk, m = 1, 8, 2, 8, 4
    q, k, g, v = rnd((B, T, dqk), 31), rnd((B, T, dqk), 32), rnd((B, T, m), 33), rnd((B, T, m), 34)
    o1, o2 = rnd((B, T, m), 35), rnd((B, T, m), 36)
    kw = dict(H=H, tau=7.0, window=3, phi_mode=0)
    a = oracle.wango_backward(q, k, g, v, o1, **kw)
    b = oracle.wango_backward(q, k, g, v, o2, **kw)
    c = oracle.wango_backward(q, k, g, v, 2 * o1 - o2, **kw)
    for n in ("dq", "dk", "dg", "dv"):
        np.testing.assert_allclose(c[n], 2 * a[n] - b[n], rtol=1e-10, atol=1e-12)


def test_causality_of_gradients():
    """dout at rows < t does not depend on the gates of sources >= t: with dout zero from
    row t on, dg, dq and dk of rows >= t are zero (a source influences later rows only)."""
    B, T, H, dqk, m, t = 1, 10, 2, 8, 4, 6
    q, k, g, v, dout = rnd((B, T, dqk), 41), rnd((B, T, dqk), 42), rnd((B, T, m), 43), rnd((B, T, m), 44), \
        rnd((B, T, m), 45)
    dout[:, t:] = 0.0
    for kind, kw in (("tango", {}), ("wango", dict(window=3, phi_mode=0))):
        d = backward(kind, q, k, g, v, dout, dict(kw, H=H, tau=10.0))
        for n in ("dq", "dk", "dg", "dv"):
            assert np.all(d[n][:, t:] == 0.0), (kind, n)


@pytest.mark.parametrize("kind,kw", [("tango", {}), ("wango", dict(window=5, phi_mode=0)),
                                     ("wango", dict(window=9, phi_mode=1, null_bias=np.array([-1.0, 0.5])))])
def test_rows_variant_equals_the_full_backward(kind, kw):
    """The sampled-row gradients (for long sequences on the GPU side) are the full
    backward's rows, including early sources, the first and last rows, and with unit
    inputs."""
    B, T, H, dqk, m = 2, 23, 2, 8, 6
    rng = np.random.default_rng(5)
    q, k, g, v, dout = (rng.standard_normal(s) for s in [(B, T, dqk)] * 2 + [(B, T, m)] * 3)
    full_fn = oracle.tango_backward if kind == "tango" else oracle.wango_backward
    rows_q = [0, 1, 7, T - 1, T, T + 13, 2 * T - 1]
    rows_k = [0, 3, T - 2, T - 1, T + 2, 2 * T - 1]
    for qn in (False, True):
        unit = lambda x: (x.reshape(B, T, H, -1) / np.linalg.norm(x.reshape(B, T, H, -1), axis=-1,
                                                                   keepdims=True)).reshape(B, T, dqk)
        qq, kk = (unit(q), unit(k)) if qn else (q, k)
        full = full_fn(qq, kk, g, v, dout, H=H, tau=4.0, qk_normalized=qn, **kw)
        part = oracle.backward_rows(kind, qq, kk, g, v, dout, H=H, tau=4.0, rows_q=rows_q, rows_k=rows_k,
                                    qk_normalized=qn, **kw)
        fq, fk = (x.reshape(B * T, -1) for x in (full["dq"], full["dk"]))
        fg, fv = (x.reshape(B * T, -1) for x in (full["dg"], full["dv"]))
        np.testing.assert_allclose(part["dq"], fq[rows_q], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(part["dv"], fv[rows_q], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(part["dk"], fk[rows_k], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(part["dg"], fg[rows_k], rtol=1e-12, atol=1e-12)
