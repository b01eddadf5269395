"""Seeded random configurations against the oracle: the aggregations (both storage types),
their backward (both far-pair paths of WANGO) and the decode step, over shapes that the
fixed cases do not pick: 1-4 heads, head widths 16/32/64, gate widths per head from 16 to
792 (multiples of 8), ragged lengths up to 400 tokens, windows from 1 to past T, score
scales from 1 to 20, with and without the null gate and v.  The configurations are drawn
once from a fixed seed, so every run checks the same ones; the bounds are those of the
fixed-case tests (test_parity_gpu.check, test_backward_gpu.run).  The backward draws run
up to 700 tokens, so that WANGO's far-pair scans (blocks wholly beyond the window's band)
take part.  bf16 draws keep tau <= 10 (fp32 draws go to 20): at tau = 20 the bf16
rounding of qhat and khat moves a logit by up to about tau 2^-8, and fp64 emulations of
the GPU's roundings (bf16 qhat, khat, P and E, exact products) land where the GPU does:
a forward draw (B = 2, T = 143, 4 heads of 290 gates) 1.33 % normwise and 4.46 % per
(row, head), the same figures to four digits; a backward draw (B = 2, T = 584, 24 gate
columns per head, null gate) 2.05 % and 9.1 % in dg, against the GPU's 2.03 % and
9.3 %.  Ten longer backward draws (700-2,500 tokens, windows up to 600; the library's
choice of far-pair path, or one of the two forced) put many blocks beyond the window's
band."""
import numpy as np
import pytest
import torch

import cross_token_gated_gb300 as tg
import oracle
from cross_token_gated_gb300 import synth
from test_backward_gpu import run as run_backward
from test_parity_gpu import abs_inputs, check, pitched, ref_agg_scaled, run_agg, run_decode

pytestmark = pytest.mark.gpu


def _draw(n, seed, backward=False, decode=False):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        H = int(rng.choice([1, 2, 4]))
        d_h = int(rng.choice([16, 32, 64]))
        m_h = 8 * int(rng.integers(2, 100 if not backward else 40))
        if not backward and not decode and rng.random() < 0.2:
            m_h += int(rng.integers(1, 8))  # a head width that is no multiple of 8
        pad = 0
        if m_h % 8 or (not backward and not decode and rng.random() < 0.2):
            pad = (-m_h) % 8 + 8 * int(rng.integers(0, 3))  # a padded per-head pitch
        B = int(rng.integers(1, 4))
        T = int(rng.integers(1, 120 if decode else (700 if backward else 400)))
        if backward:  # mostly WANGO, with windows that leave blocks beyond the band
            kind = "wango" if rng.random() < 0.7 else "tango"
            W = int(rng.integers(1, min(T, 200) + 1))
        else:
            kind = "wango" if decode else str(rng.choice(["tango", "wango"]))
            W = int(rng.integers(1, T + 64))
        dtype = "bf16" if backward else str(rng.choice(["bf16", "f32"]))
        out.append(dict(
            kind=kind, dtype=dtype, B=B, T=T, H=H, dqk=H * d_h, m=H * m_h, W=W,
            s=float(rng.choice([1.0, 4.0, 10.0] if dtype == "bf16" else [1.0, 4.0, 10.0, 20.0])),
            null=bool(rng.random() < 0.3) and not decode, has_v=bool(rng.random() < 0.7),
            phi_mode=int(rng.integers(0, 2)), normalized=bool(rng.random() < 0.3),
            far=str(rng.choice(["scan", "pairs"])), pad=pad, seed=int(rng.integers(0, 1 << 30))))
    return out


def _id(c):
    s = "{kind}-{dtype}-B{B}T{T}H{H}dqk{dqk}m{m}".format(**c)
    if c["kind"] == "wango":
        s += "W{W}-phi{phi_mode}".format(**c)
    return s + "-s{s:g}".format(**c) + ("-null" if c["null"] else "") + ("" if c["has_v"] else "-nov") + \
        (f"-pitch{c['m'] // c['H'] + c['pad']}" if c["pad"] else "") + ("-unit" if c["normalized"] else "")


def _draw_long(n, seed):
    """Backward draws over 700-2,500 tokens: WANGO's older pairs then reach far beyond the
    window's band of blocks."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        H = int(rng.choice([1, 2, 4]))
        d_h = int(rng.choice([16, 32, 64]))
        m_h = 8 * int(rng.integers(2, 48))
        B = int(rng.integers(1, 3))
        T = int(rng.integers(700, 2500))
        W = int(rng.integers(1, 600))
        out.append(dict(kind="wango" if rng.random() < 0.8 else "tango", dtype="bf16", B=B, T=T, H=H,
                        dqk=H * d_h, m=H * m_h, W=W, s=float(rng.choice([1.0, 4.0, 10.0])),
                        null=bool(rng.random() < 0.3), has_v=bool(rng.random() < 0.7),
                        phi_mode=int(rng.integers(0, 2)), normalized=bool(rng.random() < 0.3),
                        far=str(rng.choice(["scan", "pairs", "auto"])), pad=0, seed=int(rng.integers(0, 1 << 30))))
    return out


FWD = _draw(40, 20261202)
BWD = _draw(20, 20261203, backward=True) + _draw_long(10, 888004)
DEC = _draw(12, 20261204, decode=True)


@pytest.mark.parametrize("c", FWD, ids=[_id(c) for c in FWD])
def test_fuzz_aggregation(c):
    B, T, H, m = c["B"], c["T"], c["H"], c["m"]
    q, k, g, v = synth.agg_inputs(B, T, c["dqk"], m, seed=c["seed"], dtype=c["dtype"])
    if c["normalized"]:  # unit vectors per head, rounded to the storage type
        qf, kf = q.double().view(B, T, H, -1), k.double().view(B, T, H, -1)
        q = (qf / qf.norm(dim=-1, keepdim=True)).view(B, T, -1).to(q.dtype)
        k = (kf / kf.norm(dim=-1, keepdim=True)).view(B, T, -1).to(k.dtype)
    if not c["has_v"]:
        v = None
    nb = torch.linspace(-1.5, 0.5, H, dtype=torch.float32) if c["null"] else None
    kw = dict(s=c["s"])
    if c["kind"] == "wango":
        kw["phi_mode"] = c["phi_mode"]
    flags = tg.TG_FLAG_QK_NORMALIZED if c["normalized"] else 0
    if c["pad"]:  # gates at a padded per-head pitch whose padding holds NaN
        m_h = m // H
        pitch = m_h + c["pad"]
        gp = pitched(g, H, pitch, float("nan")).cuda()
        vp = pitched(v, H, pitch, float("nan")).cuda() if v is not None else None
        out = torch.empty_like(gp)
        nbd = nb.cuda() if nb is not None else None
        if c["kind"] == "tango":
            tg.tango_aggregate(q.cuda(), k.cuda(), gp, vp, out, H=H, m_h=m_h, null_bias=nbd, flags=flags, **kw)
        else:
            tg.wango_aggregate(q.cuda(), k.cuda(), gp, vp, out, H=H, window=c["W"], m_h=m_h, null_bias=nbd,
                               flags=flags, **kw)
        st, word = tg.tg_check_device_error()
        assert st == tg.TG_OK, (st, hex(word))
        out = out.view(B, T, H, pitch)[..., :m_h].reshape(B, T, m)
    else:
        out = run_agg(c["kind"], q, k, g, v, H, c["W"], flags=flags,
                      null_bias=nb.cuda() if nb is not None else None, **kw)
    ref_kw = dict(kw, null_bias=nb.double().numpy() if nb is not None else None, qk_normalized=c["normalized"])
    ref, scale = ref_agg_scaled(c["kind"], q, k, g, v, H, c["W"], **ref_kw)
    check(out, ref, c["dtype"], H, scale)


@pytest.mark.parametrize("c", BWD, ids=[_id(c) + (f"-{c['far']}" if c["kind"] == "wango" else "") for c in BWD])
def test_fuzz_backward(c):
    far = c["far"] if c["kind"] == "wango" and c["far"] != "auto" else None
    run_backward(c["kind"], c["B"], c["T"], c["H"], c["dqk"], c["m"], W=c["W"], phi_mode=c["phi_mode"],
                 null=c["null"], has_v=c["has_v"], normalized=c["normalized"], seed=c["seed"], s=c["s"],
                 far=far)


@pytest.mark.parametrize("c", DEC, ids=[_id(c) for c in DEC])
def test_fuzz_decode(c):
    q, k, g, v = synth.agg_inputs(c["B"], c["T"], c["dqk"], c["m"], seed=c["seed"], dtype=c["dtype"])
    if not c["has_v"]:
        v = None
    out = run_decode(q, k, g, v, c["H"], c["W"], s=c["s"], phi_mode=c["phi_mode"])
    kw = dict(H=c["H"], tau=c["s"], window=c["W"], phi_mode=c["phi_mode"])
    ref = oracle.wango_scan(*[synth.oracle_view(t) if t is not None else None for t in (q, k, g, v)], **kw)
    ga, va = abs_inputs(g, v)
    scale = oracle.wango_scan(*[synth.oracle_view(t) if t is not None else None for t in (q, k, ga, va)], **kw)
    check(out, ref, c["dtype"], c["H"], scale)
