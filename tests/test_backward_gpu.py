"""Parity of the aggregation backward (tango_aggregate_backward, wango_aggregate_backward)
with the oracle's fp64 gradients (oracle.tango_backward / oracle.wango_backward: eq. 5
differentiated pair by pair), element by element on seeded inputs.

Bounds per output tensor, with TOL = 2e-2 (bf16 storage, bf16 tensor-core operands,
fp32 accumulation), at tau <= 10 (the benchmark's 10 and below):
- dg, dv: normwise max |gpu - oracle| / max |oracle| <= TOL, and the same ratio within
  each (row, head) <= 2 TOL (as for the forward outputs);
- dq, dk: normwise <= TOL, and per (row, head) max |gpu - oracle| <= TOL * scale, with
  the scale of the sum that forms the gradient.  dq_i sums tau alpha_ij
  (dgbar_i . (g_j - gbar_i)) khat_j over the sources; a relative rounding e of the
  products inside the dot products moves it by at most
      e * tau sum_c |dgbar_ic| (sum_j alpha_ij |g_jc| + |gbar_ic|) / |q_i|,
  which is the scale (the aggregation of |g| gives the inner sum); dk_j likewise sums
  over destinations, with sum_i alpha_ij |dgbar_i| and sum_i alpha_ij |dgbar_i gbar_i|
  (the gate gradients of those two upstream gradients) in place of the aggregations.
  A plain relative bound per row would fail where dq or dk cancels to near zero (a
  peaked softmax, or T = 1, where they vanish), since the rounding of the terms remains.

At the full benchmark width (m = 28,480) the comparison runs on whole sequences of 640
tokens (so the 64-column contraction chunks end inside each head, and the next head's
columns must read as zero); at the full batch and length (B = 8, T = 2,048) the checks
are properties that hold at any size: dv = dout * gbar exactly as the forward's gbar
gives it, sum_j dg_j . g_j = sum_i (dout_i * v_i) . gbar_i (the aggregation is linear
in g), and dq, dk orthogonal to q, k per head (the scores see only unit vectors).
"""
import numpy as np
import pytest
import torch

import cross_token_gated_gb300 as tg
import oracle
from cross_token_gated_gb300 import synth

pytestmark = pytest.mark.gpu

TOL = 2e-2


def as_np(gpu, shape):
    g = gpu.detach().double().cpu().numpy().reshape(shape)
    assert np.all(np.isfinite(g)), "non-finite values in the GPU output"
    return g


def errs(gpu, ref, H, scale=None):
    """Normwise error, and per (row, head) either the relative error (no scale) or the
    largest error over `scale` [rows, H]."""
    g = as_np(gpu, ref.shape)
    d, a = np.abs(g - ref), np.abs(ref)
    n = ref.shape[-1]
    dr, ar = d.reshape(-1, H, n // H), a.reshape(-1, H, n // H)
    out = {"norm": float(d.max() / a.max()) if a.max() > 0 else 0.0, "abs": float(d.max())}
    if scale is None:
        out["row_head"] = float(np.max(dr.max(-1) / np.maximum(ar.max(-1), 1e-30)))
    else:
        out["row_head_cond"] = float(np.max(dr.max(-1) / np.maximum(np.asarray(scale).reshape(-1, H), 1e-30)))
    return out


def grad_scales(kind, view, H, s, W, phi_mode, nbo, normalized):
    """Per (row, head) error scales of dq and dk (see the module docstring), from the
    oracle's forward and gate gradients."""
    q, k, g, v, dout = view
    B, T, dqk = q.shape
    m = g.shape[-1]
    f64 = lambda t: t.astype(np.float64) if t.dtype != np.uint16 else \
        (t.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    gf, doutf = f64(g), f64(dout)
    dgb = doutf * f64(v) if v is not None else doutf
    kw = dict(H=H, tau=s, null_bias=nbo, qk_normalized=normalized)
    if kind == "tango":
        fwd = lambda gg: oracle.tango(q, k, gg, None, **kw)
        bwd = lambda d: oracle.tango_backward(q, k, g, None, d, **kw)["dg"]
    else:
        fwd = lambda gg: oracle.wango_direct(q, k, gg, None, window=W, phi_mode=phi_mode, **kw)
        bwd = lambda d: oracle.wango_backward(q, k, g, None, d, window=W, phi_mode=phi_mode, **kw)["dg"]
    gbar, agg_abs = fwd(g), fwd(np.abs(gf))
    r1, r2 = bwd(np.abs(dgb)), bwd(np.abs(dgb * gbar))
    heads = lambda x: x.reshape(B, T, H, -1)
    nq = np.linalg.norm(heads(f64(q)), axis=-1) if not normalized else 1.0
    nk = np.linalg.norm(heads(f64(k)), axis=-1) if not normalized else 1.0
    sq = s * np.sum(heads(np.abs(dgb)) * (heads(agg_abs) + heads(np.abs(gbar))), axis=-1) / nq
    sk = s * np.sum(heads(r1) * heads(np.abs(gf)) + heads(r2), axis=-1) / nk
    return sq, sk


FAR_FLAGS = {None: 0, "scan": tg.TG_FLAG_BWD_FAR_SCAN, "pairs": tg.TG_FLAG_BWD_FAR_PAIRS}


def run(kind, B, T, H, dqk, m, *, W=16, phi_mode=0, null=False, has_v=True, normalized=False, seed=0, s=10.0,
        far=None):
    """far: how WANGO forms the older pairs beyond the window's band of blocks ("scan":
    running sums, "pairs": pair by pair, None: the library's choice)."""
    q, k, g, v = synth.agg_inputs(B, T, dqk, m, seed=seed, dtype="bf16")
    if normalized:  # unit vectors per head, rounded to bf16
        qf, kf = q.float().view(B, T, H, -1), k.float().view(B, T, H, -1)
        q = (qf / qf.norm(dim=-1, keepdim=True)).view(B, T, dqk).bfloat16()
        k = (kf / kf.norm(dim=-1, keepdim=True)).view(B, T, dqk).bfloat16()
    if not has_v:
        v = None
    dout = synth.upstream_grad(B, T, m, seed=seed + 100)
    nb = torch.linspace(-1.0, 0.5, H, dtype=torch.float32) if null else None
    dev = [t.cuda() if t is not None else None for t in (q, k, g, v, dout)]
    dq, dk = torch.empty_like(dev[0]), torch.empty_like(dev[1])
    dg = torch.empty_like(dev[2])
    dv = torch.empty_like(dev[2]) if has_v else None
    flags = tg.TG_FLAG_QK_NORMALIZED if normalized else 0
    nbd = nb.cuda() if nb is not None else None
    if kind == "tango":
        tg.tango_aggregate_backward(*dev, dq, dk, dg, dv, H=H, s=s, null_bias=nbd, flags=flags)
    else:
        tg.wango_aggregate_backward(*dev, dq, dk, dg, dv, H=H, window=W, s=s, null_bias=nbd, phi_mode=phi_mode,
                                    flags=flags | FAR_FLAGS[far])
    st, word = tg.tg_check_device_error()
    assert st == tg.TG_OK, (st, hex(word))
    view = [synth.oracle_view(t) if t is not None else None for t in (q, k, g, v, dout)]
    nbo = nb.double().numpy() if nb is not None else None
    if kind == "tango":
        ref = oracle.tango_backward(*view, H=H, tau=s, null_bias=nbo, qk_normalized=normalized)
    else:
        ref = oracle.wango_backward(*view, H=H, tau=s, window=W, phi_mode=phi_mode, null_bias=nbo,
                                    qk_normalized=normalized)
    sq, sk = grad_scales(kind, view, H, s, W, phi_mode, nbo, normalized)
    out = {"dq": (dq, sq), "dk": (dk, sk), "dg": (dg, None)}
    if has_v:
        out["dv"] = (dv, None)
    report = {}
    for name, (t, scale) in out.items():
        report[name] = errs(t, ref[name], H, scale)
    for name, e in report.items():
        assert e["norm"] <= TOL, (name, report)
        if "row_head" in e:
            assert e["row_head"] <= 2 * TOL, (name, report)
        else:
            assert e["row_head_cond"] <= TOL, (name, report)
    return report


TANGO_CASES = [
    # B, T, H, dqk, m
    (1, 300, 2, 128, 512),     # ragged tail, 3 destination blocks, two 256-source tiles
    (2, 129, 2, 64, 256),      # d_h = 32, one row past a block
    (1, 70, 1, 16, 64),        # d_h = 16, a single short block
    (1, 520, 2, 128, 1040),    # 5 destination blocks, 3 source tiles, m_h % 64 = 8
    (3, 64, 4, 128, 384),      # four heads of 32
]


@pytest.mark.parametrize("B,T,H,dqk,m", TANGO_CASES)
def test_tango_backward_small(B, T, H, dqk, m):
    run("tango", B, T, H, dqk, m, seed=B * 7 + T)


def test_tango_backward_null_gate_and_no_v():
    run("tango", 1, 300, 2, 128, 512, null=True, seed=3)
    run("tango", 1, 200, 2, 128, 256, has_v=False, seed=4)


def test_tango_backward_unit_inputs():
    run("tango", 2, 150, 2, 128, 256, normalized=True, seed=5)


def test_backward_t1():
    """T = 1: the only weight is the self weight, so gbar = g, dg = dout * v and
    dq = dk = 0 (the conditioned bound then limits the rounding residue)."""
    run("tango", 2, 1, 2, 128, 256, seed=6)
    run("wango", 2, 1, 2, 128, 256, W=1, seed=7)


@pytest.mark.parametrize("W", [1, 16, 200, 1000])
@pytest.mark.parametrize("phi_mode", [0, 1])
@pytest.mark.parametrize("far", ["scan", "pairs"])
def test_wango_backward_small(W, phi_mode, far):
    """T = 300 (3 blocks): W = 1 and 16 leave blocks beyond the band (the scans' far
    pairs, 2 and 1 steps), W = 200 and 1000 none."""
    run("wango", 1, 300, 2, 128, 512, W=W, phi_mode=phi_mode, seed=W + phi_mode, far=far)


@pytest.mark.parametrize("far", ["scan", "pairs"])
def test_wango_backward_shapes(far):
    run("wango", 2, 129, 2, 64, 256, W=40, seed=11, far=far)
    run("wango", 1, 520, 2, 128, 1040, W=256, seed=12, far=far)
    run("wango", 1, 300, 2, 128, 512, W=64, null=True, has_v=False, seed=13, far=far)
    run("wango", 3, 64, 4, 128, 384, W=8, normalized=True, seed=14, far=far)
    # d_h = 16 and 32 through the scans, 5 and 7 blocks, a strip's partial last chunk
    run("wango", 2, 600, 4, 64, 1120, W=100, seed=15, far=far)
    run("wango", 1, 900, 4, 128, 2592, W=130, normalized=True, seed=16, far=far)


@pytest.mark.parametrize("kind,far", [("tango", None), ("wango", "scan"), ("wango", "pairs")])
def test_backward_full_width(kind, far):
    """The 70M-tier gate width (m = 28,480 as two heads of 14,240, i.e. 38 strips of 384
    for the scans at B = 1), one 640-token sequence compared in full."""
    run(kind, 1, 640, 2, 128, 28480, W=256, seed=21, far=far)


@pytest.mark.parametrize("B,T,H,dqk,m,W", [(2, 1500, 2, 128, 4096, 64), (8, 2048, 2, 128, 28480, 256)])
def test_wango_backward_far_paths_agree(B, T, H, dqk, m, W):
    """The scans and the pair path give the same dq and dk within bf16 rounding (the
    pair path rounds X_ij to bf16, the scans their running sums), and dg, dv bit for bit
    (neither depends on the choice): B = 2, T = 1,500, W = 64 (11 blocks beyond the band
    of 1), and the benchmark shape, where the side-1 far rows (the first 13 blocks) are
    beyond the oracle's reach at this size."""
    q, k, g, v = (t.cuda() for t in synth.agg_inputs(B, T, dqk, m, seed=41, dtype="bf16"))
    dout = synth.upstream_grad(B, T, m, seed=42).cuda()
    res = {}
    for far in ("scan", "pairs"):
        dq, dk, dg, dv = (torch.empty_like(x) for x in (q, k, g, g))
        tg.wango_aggregate_backward(q, k, g, v, dout, dq, dk, dg, dv, H=H, window=W, flags=FAR_FLAGS[far])
        st, word = tg.tg_check_device_error()
        assert st == tg.TG_OK, (st, hex(word))
        res[far] = (dq, dk, dg, dv)
    for name, a, b in zip(("dq", "dk"), res["scan"][:2], res["pairs"][:2]):
        e = float((a.float() - b.float()).abs().max() / b.float().abs().max())
        assert e <= TOL, (name, e)
        # per (row, head), against the row's own scale
        d = (a.float() - b.float()).view(B * T, H, -1).abs().amax(-1)
        r = b.float().view(B * T, H, -1).abs().amax(-1)
        assert float((d / (r + 1e-2 * float(r.max()))).max()) <= 4 * TOL, name
    assert torch.equal(res["scan"][2], res["pairs"][2])
    assert torch.equal(res["scan"][3], res["pairs"][3])


@pytest.mark.parametrize("kind", ["tango", "wango"])
def test_backward_full_size_properties(kind):
    """B = 8, T = 2,048, m = 28,480 (the benchmark shape): properties that hold at any size."""
    B, T, H, dqk, m, W = 8, 2048, 2, 128, 28480, 256
    q, k, g, v = (t.cuda() for t in synth.agg_inputs(B, T, dqk, m, seed=31, dtype="bf16"))
    dout = synth.upstream_grad(B, T, m, seed=32).cuda()
    dq, dk, dg, dv = (torch.empty_like(x) for x in (q, k, g, g))
    gbar = torch.empty_like(g)
    if kind == "tango":
        tg.tango_aggregate_backward(q, k, g, v, dout, dq, dk, dg, dv, H=H)
        tg.tango_aggregate(q, k, g, None, gbar, H=H)
    else:
        tg.wango_aggregate_backward(q, k, g, v, dout, dq, dk, dg, dv, H=H, window=W)
        tg.wango_aggregate(q, k, g, None, gbar, H=H, window=W)
    st, word = tg.tg_check_device_error()
    assert st == tg.TG_OK, (st, hex(word))
    for t in (dq, dk, dg, dv):
        assert torch.isfinite(t.float()).all()
    # dv = dout * gbar, each product rounded once to bf16
    assert torch.equal(dv, (dout.float() * gbar.float()).bfloat16())
    # linearity in g: sum_j dg_j . g_j = sum_i (dout_i * v_i) . gbar_i, per (batch, head)
    lhs = (dg.double() * g.double()).view(B, T, H, -1).sum(dim=(1, 3))
    rhs = (dout.double() * v.double() * gbar.double()).view(B, T, H, -1).sum(dim=(1, 3))
    scale = (dout.double() * v.double() * gbar.double()).abs().view(B, T, H, -1).sum(dim=(1, 3))
    assert float(((lhs - rhs).abs() / scale).max()) < 2e-2
    # the scores see unit vectors only: dq . q = 0 and dk . k = 0 per (row, head)
    for d, x in ((dq, q), (dk, k)):
        dd, xx = d.double().view(B, T, H, -1), x.double().view(B, T, H, -1)
        dot = (dd * xx).sum(-1)
        bound = dd.norm(dim=-1) * xx.norm(dim=-1)
        assert float((dot.abs() / bound.clamp_min(1e-30)).max()) < 2e-2


@pytest.mark.parametrize("kind", ["tango", "wango"])
def test_backward_gate_pitch(kind):
    """The backward at the three-set head width m_h = 4,747 with a per-head pitch of
    4,752: NaN in the padding columns of g, v and dout must reach no gradient."""
    B, T, H, dqk, m_h, pitch, W = 1, 260, 2, 128, 4747, 4752, 100
    q, k, g, v = synth.agg_inputs(B, T, dqk, H * m_h, seed=51, dtype="bf16")
    dout = synth.upstream_grad(B, T, H * m_h, seed=52)

    def pad(t):
        out = torch.full((B, T, H, pitch), float("nan"), dtype=t.dtype)
        out[..., :m_h] = t.view(B, T, H, m_h)
        return out.view(B, T, H * pitch).cuda()

    gp, vp, dp_ = pad(g), pad(v), pad(dout)
    qd, kd = q.cuda(), k.cuda()
    dq, dk, dg, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(gp), torch.empty_like(gp)
    if kind == "tango":
        tg.tango_aggregate_backward(qd, kd, gp, vp, dp_, dq, dk, dg, dv, H=H, m_h=m_h)
    else:
        tg.wango_aggregate_backward(qd, kd, gp, vp, dp_, dq, dk, dg, dv, H=H, window=W, m_h=m_h)
    st, word = tg.tg_check_device_error()
    assert st == tg.TG_OK, (st, hex(word))
    view = [synth.oracle_view(t) for t in (q, k, g, v, dout)]
    if kind == "tango":
        ref = oracle.tango_backward(*view, H=H, tau=10.0)
    else:
        ref = oracle.wango_backward(*view, H=H, tau=10.0, window=W)
    sq, sk = grad_scales(kind, view, H, 10.0, W, 0, None, False)
    logical = lambda t: t.view(B, T, H, pitch)[..., :m_h].reshape(B, T, H * m_h)
    for name, t, scale in (("dq", dq, sq), ("dk", dk, sk), ("dg", logical(dg), None), ("dv", logical(dv), None)):
        e = errs(t, ref[name], H, scale)
        assert e["norm"] <= TOL, (name, e)
        assert e.get("row_head", 0.0) <= 2 * TOL and e.get("row_head_cond", 0.0) <= TOL, (name, e)


@pytest.mark.parametrize("kind", ["tango", "wango"])
def test_saved_forward_feeds_the_backward(kind):
    """tango/wango_aggregate_save write u as the plain call does, plus gbar and the row
    denominators; the backward given them (no recomputation of the forward) returns
    exactly the gradients it computes without them.  gbar equals the forward with v = NULL."""
    B, T, H, dqk, m, W = 2, 300, 2, 128, 1040, 100
    q, k, g, v = (t.cuda() for t in synth.agg_inputs(B, T, dqk, m, seed=61, dtype="bf16"))
    dout = synth.upstream_grad(B, T, m, seed=62).cuda()
    u, u_ref, gbar, gbar_ref = (torch.empty_like(g) for _ in range(4))
    den = torch.empty(B, H, T, dtype=torch.float32, device="cuda")
    kw = {} if kind == "tango" else {"window": W}
    fwd = tg.tango_aggregate if kind == "tango" else tg.wango_aggregate
    save = tg.tango_aggregate_save if kind == "tango" else tg.wango_aggregate_save
    bwd = tg.tango_aggregate_backward if kind == "tango" else tg.wango_aggregate_backward
    save(q, k, g, v, u, gbar, den, H=H, **kw)
    fwd(q, k, g, v, u_ref, H=H, **kw)
    fwd(q, k, g, None, gbar_ref, H=H, **kw)
    assert torch.equal(u, u_ref)
    assert torch.equal(gbar, gbar_ref)
    assert bool(torch.isfinite(den).all()) and bool((den > 0).all())
    grads = [[torch.empty_like(x) for x in (q, k, g, g)] for _ in range(2)]
    bwd(q, k, g, v, dout, *grads[0], H=H, **kw)
    bwd(q, k, g, v, dout, *grads[1], H=H, gbar=gbar, den=den, **kw)
    st, word = tg.tg_check_device_error()
    assert st == tg.TG_OK, (st, hex(word))
    for a, b in zip(*grads):
        assert torch.equal(a, b)


@pytest.mark.parametrize("kind,far", [("tango", None), ("wango", "pairs"), ("wango", "scan")])
def test_backward_full_size_sampled_rows(kind, far):
    """B = 8, T = 2,048, m = 28,480 (the benchmark shape, W = 256 for WANGO): dq and dv at
    sampled destinations (first, window and block edges, last, random) and dk, dg at the
    last sources of two sequences, against the oracle's gradients at those rows alone.
    Bounds: normwise over the sample, and per (row, head) for dg and dv."""
    B, T, H, dqk, m, W = 8, 2048, 2, 128, 28480, 256
    q, k, g, v = synth.agg_inputs(B, T, dqk, m, seed=71, dtype="bf16")
    dout = synth.upstream_grad(B, T, m, seed=72)
    dev = [t.cuda() for t in (q, k, g, v, dout)]
    dq, dk, dg, dv = (torch.empty_like(x) for x in (dev[0], dev[1], dev[2], dev[2]))
    if kind == "tango":
        tg.tango_aggregate_backward(*dev, dq, dk, dg, dv, H=H)
    else:
        tg.wango_aggregate_backward(*dev, dq, dk, dg, dv, H=H, window=W, flags=FAR_FLAGS[far])
    st, word = tg.tg_check_device_error()
    assert st == tg.TG_OK, (st, hex(word))
    rng = np.random.default_rng(73)
    rows_q = []
    for b in (0, 5, 7):
        ts = [0, 1, 2, 127, 128, 255, 256, 257, 1024, 2045, 2046, 2047] + list(rng.integers(0, T, 6))
        rows_q += [b * T + int(t) for t in ts]
    rows_k = [b * T + t for b in (2, 7) for t in (T - 1, T - 2, T - 5, T - 9, T - 14)]
    view = [synth.oracle_view(t) for t in (q, k, g, v, dout)]
    kw = {} if kind == "tango" else {"window": W}
    ref = oracle.backward_rows(kind, *view, H=H, tau=10.0, rows_q=rows_q, rows_k=rows_k, **kw)
    got = {"dq": dq.view(B * T, -1)[rows_q], "dv": dv.view(B * T, -1)[rows_q],
           "dk": dk.view(B * T, -1)[rows_k], "dg": dg.view(B * T, -1)[rows_k]}
    for name, t in got.items():
        e = errs(t, ref[name], H)
        assert e["norm"] <= TOL, (name, e)
        if name in ("dg", "dv"):
            assert e["row_head"] <= 2 * TOL, (name, e)


@pytest.mark.parametrize("kind,far", [("tango", None), ("wango", "scan"), ("wango", "pairs")])
def test_backward_bounded_wait_timeout_reports_status(kind, far):
    """TG_FLAG_DEBUG_TIMEOUT arms the hook of the backward's own tensor-core kernels (the
    pair gradients, dq/dk and, on the scan path, the running-sum scans): each MMA issuer
    first waits on a barrier that nothing signals, runs out (1 ms), records a timeout
    (kernel code 5) and every role leaves its loops.  The forward kernels that the call
    also runs get no flag.  The context stays usable: the next call is correct."""
    B, T, H, dqk, m, W = 1, 700, 2, 128, 512, 16  # W = 16: blocks beyond the band, so scans
    q, k, g, v = synth.agg_inputs(B, T, dqk, m, seed=31, dtype="bf16")
    dout = synth.upstream_grad(B, T, m, seed=131)
    dev = [t.cuda() for t in (q, k, g, v, dout)]
    dq, dk, dg, dv = (torch.empty_like(dev[i]) for i in (0, 1, 2, 2))
    flags = tg.TG_FLAG_DEBUG_TIMEOUT | FAR_FLAGS[far]
    if kind == "tango":
        tg.tango_aggregate_backward(*dev, dq, dk, dg, dv, H=H, flags=flags)
    else:
        tg.wango_aggregate_backward(*dev, dq, dk, dg, dv, H=H, window=W, flags=flags)
    st, word = tg.tg_check_device_error()
    assert st == tg.TG_ERR_TIMEOUT
    assert word & 1 and (word >> 8) & 0xFF == 5, hex(word)
    assert tg.tg_check_device_error() == (tg.TG_OK, 0)
    run(kind, B, T, H, dqk, m, W=W, seed=31, far=far)
