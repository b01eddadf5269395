"""Parity of the CUDA path with the fp64 oracle, element by element, on seeded inputs.

Tolerances (stated for the path): max |gpu - oracle| / max |oracle| per output tensor
must be <= 1e-4 for fp32 storage (CUDA-core fp32 arithmetic) and <= 2e-2 for bf16
storage (bf16 tensor-core operands, fp32 accumulation).  The oracle reads exactly the
values the GPU reads (bf16 inputs are widened, not re-rounded).
"""
import numpy as np
import pytest
import torch

import cross_token_gated_gb300 as tg
import oracle
from cross_token_gated_gb300 import synth

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}


def rel_err(gpu: torch.Tensor, ref: np.ndarray) -> float:
    g = gpu.detach().double().cpu().numpy().reshape(ref.shape)
    assert np.all(np.isfinite(g)), "non-finite values in the GPU output"
    return float(np.max(np.abs(g - ref)) / max(np.max(np.abs(ref)), 1e-30))


def run_agg(kind, q, k, g, v, H, W=16, **kw):
    qd, kd, gd = q.cuda(), k.cuda(), g.cuda()
    vd = v.cuda() if v is not None else None
    out = torch.empty_like(gd)
    if kind == "tango":
        tg.tango_aggregate(qd, kd, gd, vd, out, H=H, **kw)
    else:
        tg.wango_aggregate(qd, kd, gd, vd, out, H=H, window=W, **kw)
    st, word = tg.tg_check_device_error()
    assert st == tg.TG_OK, (st, hex(word))
    return out


def ref_agg(kind, q, k, g, v, H, W=16, s=10.0, rows=None, **kw):
    args = [synth.oracle_view(t) if t is not None else None for t in (q, k, g, v)]
    if kind == "tango":
        return oracle.tango(*args, H=H, tau=s, rows=rows, **kw)
    return oracle.wango_direct(*args, H=H, tau=s, window=W, rows=rows, **kw)


# (B, T, H, d_qk, m, W): tiny oracle config, ragged T, ragged gate tiles, several W
SMALL = [
    (1, 64, 2, 32, 256, 16),      # the tiny oracle configuration
    (1, 1, 2, 32, 256, 16),       # T = 1
    (2, 63, 2, 128, 144, 1),      # W = 1: every earlier source is older
    (3, 65, 2, 64, 272, 64),      # W = T - 1
    (1, 200, 2, 128, 1040, 200),  # W = T: no older prefix
    (2, 130, 4, 128, 544, 300),   # W > T, four heads of d_h = 32
    (1, 300, 2, 128, 2096, 129),  # ragged window boundary
    (1, 700, 2, 128, 272, 200),   # two mixed blocks in a row, window > one block
    (2, 520, 2, 64, 144, 100),    # W < block: the diagonal block is mixed too
    (1, 700, 2, 128, 272, 400),   # five source blocks per destination block
    (1, 700, 2, 64, 144, 700),    # W = T: every earlier block is a source block
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("kind", ["tango", "wango"])
@pytest.mark.parametrize("case", SMALL, ids=[f"B{c[0]}T{c[1]}H{c[2]}dqk{c[3]}m{c[4]}W{c[5]}" for c in SMALL])
def test_agg_parity_small(kind, dtype, case):
    B, T, H, dqk, m, W = case
    q, k, g, v = synth.agg_inputs(B, T, dqk, m, seed=T + m, dtype=dtype)
    out = run_agg(kind, q, k, g, v, H, W)
    ref = ref_agg(kind, q, k, g, v, H, W)
    assert rel_err(out, ref) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("kind", ["tango", "wango"])
def test_agg_null_gate_tau_array_and_gbar_output(kind, dtype):
    """Per-head tau from device memory, the null gate on, v = NULL (out = gbar), and
    pre-normalised q/k passed with TG_FLAG_QK_NORMALIZED."""
    B, T, H, dqk, m, W = 2, 150, 2, 128, 512, 40
    q, k, g, _ = synth.agg_inputs(B, T, dqk, m, seed=7, dtype=dtype)
    tau = torch.tensor([10.0, 4.0], device="cuda")
    nb = torch.tensor([-1.0, 0.5], device="cuda")
    out = run_agg(kind, q, k, g, None, H, W, tau=tau, null_bias=nb)
    ref = ref_agg(kind, q, k, g, None, H, W, s=[10.0, 4.0], null_bias=[-1.0, 0.5])
    assert rel_err(out, ref) <= TOL[dtype]
    # unit vectors in, no normalisation inside
    qn = q.double().reshape(B, T, H, -1)
    qn = (qn / qn.norm(dim=-1, keepdim=True)).reshape(B, T, dqk).to(q.dtype)
    kn = k.double().reshape(B, T, H, -1)
    kn = (kn / kn.norm(dim=-1, keepdim=True)).reshape(B, T, dqk).to(k.dtype)
    out2 = run_agg(kind, qn, kn, g, None, H, W, tau=tau, null_bias=nb, flags=tg.TG_FLAG_QK_NORMALIZED)
    ref2 = ref_agg(kind, qn, kn, g, None, H, W, s=[10.0, 4.0], null_bias=[-1.0, 0.5], qk_normalized=True)
    assert rel_err(out2, ref2) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("kind", ["tango", "wango"])
def test_agg_weights_sum_to_one_on_gpu(kind, dtype):
    """g == 1 gives gbar == 1 on the GPU path too (the denominator is the sum of the
    very weights applied to g)."""
    B, T, H, dqk, m, W = 1, 333, 2, 128, 256, 70
    q, k, _, _ = synth.agg_inputs(B, T, dqk, m, seed=11, dtype=dtype)
    g = torch.ones(B, T, m, dtype=q.dtype)
    out = run_agg(kind, q, k, g, None, H, W)
    tol = 1e-5 if dtype == "f32" else 8e-3
    assert (out.float() - 1).abs().max().item() <= tol


@pytest.mark.parametrize("kind", ["tango", "wango"])
def test_agg_parity_70m_shape_sampled(kind):
    """bf16 at the 70M-tier aggregation shape (B=8, T=2048, m=28480, q/k width 128,
    W=256): oracle rows sampled at the sequence ends, the window and tile boundaries,
    plus random rows."""
    B, T, H, dqk, m, W = 8, 2048, 2, 128, 28480, 256
    q, k, g, v = synth.agg_inputs(B, T, dqk, m, seed=0, dtype="bf16")
    out = run_agg(kind, q, k, g, v, H, W)
    extra = [0, 1, 127, 128, 255, 256, 257, 383, 384, 2047, 7 * T + 2047, 3 * T + 1000]
    rows = synth.random_rows(B, T, 40, seed=1, extra=extra)
    ref = ref_agg(kind, q, k, g, v, H, W, rows=rows)
    got = out.reshape(B * T, m)[torch.from_numpy(rows).cuda()]
    assert rel_err(got, ref) <= TOL["bf16"]


@pytest.mark.parametrize("kind", ["tango", "wango"])
def test_agg_parity_long_context_sampled(kind):
    """bf16 at the long-context shape (B=1, T=8192, m=28480, q/k width 128, W=256).
    Few strips for many destination blocks: the WANGO kernel splits each strip into
    segments, and a later segment starts by rebuilding the state.  Oracle rows are
    sampled around the segment and window boundaries."""
    B, T, H, dqk, m, W = 1, 8192, 2, 128, 28480, 256
    q, k, g, v = synth.agg_inputs(B, T, dqk, m, seed=3, dtype="bf16")
    out = run_agg(kind, q, k, g, v, H, W)
    extra = [0, 255, 256, 4095, 4096, 4097, 4223, 4224, 4351, 4352, 8191]
    rows = synth.random_rows(B, T, 24, seed=2, extra=extra)
    ref = ref_agg(kind, q, k, g, v, H, W, rows=rows)
    got = out.reshape(B * T, m)[torch.from_numpy(rows).cuda()]
    assert rel_err(got, ref) <= TOL["bf16"]


# ------------------------------------------------------------------ block forward

def run_block(h, w, H, mode, W, **kw):
    hd = h.cuda()
    wd = {n: t.cuda() for n, t in w.items()}
    out = torch.empty_like(hd)
    tg.tango_block_forward(hd, wd, out, H=H, mode=mode, window=W, **kw)
    st, word = tg.tg_check_device_error()
    assert st == tg.TG_OK, (st, hex(word))
    return out


def ref_block(h, w, H, mode, W, batches=None, s=10.0):
    wv = {n: synth.oracle_view(t) for n, t in w.items()}
    return oracle.block_forward(synth.oracle_view(h), wv, H=H, tau=s, mode=mode, window=W,
                                batches=batches, rope_base=10000.0, rms_eps=1e-6)


@pytest.mark.parametrize("mode", [0, 1])
def test_block_tiny_fp32(mode):
    """The tiny oracle configuration: B=1, T=64, d=64, m=256, q/k width 32, W=16, fp32."""
    B, T, d, dqk, m, H, W = 1, 64, 64, 32, 256, 2, 16
    h, w = synth.block_inputs(B, T, d, dqk, m, seed=0, dtype="f32")
    out = run_block(h, w, H, mode, W)
    ref = ref_block(h, w, H, mode, W)
    h64 = h.double().numpy()
    assert rel_err(out, ref) <= 1e-4
    assert rel_err(out.cpu().double() - torch.from_numpy(h64), ref - h64) <= 1e-4


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("shape", [(2, 100, 128, 64, 512, 2, 32), (1, 257, 128, 128, 1040, 2, 100)])
def test_block_bf16_small(mode, shape):
    B, T, d, dqk, m, H, W = shape
    h, w = synth.block_inputs(B, T, d, dqk, m, seed=5, dtype="bf16")
    out = run_block(h, w, H, mode, W)
    ref = ref_block(h, w, H, mode, W)
    h64 = h.double().numpy()
    assert rel_err(out, ref) <= TOL["bf16"]
    assert rel_err(out.cpu().double() - torch.from_numpy(h64), ref - h64) <= TOL["bf16"]


@pytest.mark.parametrize("mode", [0, 1])
def test_block_output_gemm_many_tiles(mode):
    """d=1024 and B*T=5000 rows give 40 row blocks of 4 output tiles, 160 tiles for 152
    SMs: the persistent output GEMM takes a second tile on some CTAs, with K = m = 256
    (4 k-blocks a tile).  Every row is compared, the last row block being ragged (8 rows)."""
    B, T, d, dqk, m, H, W = 2, 2500, 1024, 128, 256, 2, 100
    h, w = synth.block_inputs(B, T, d, dqk, m, seed=11, dtype="bf16")
    out = run_block(h, w, H, mode, W)
    ref = ref_block(h, w, H, mode, W)
    h64 = h.double().numpy()
    assert rel_err(out, ref) <= TOL["bf16"]
    assert rel_err(out.cpu().double() - torch.from_numpy(h64), ref - h64) <= TOL["bf16"]


@pytest.mark.parametrize("mode", [0, 1])
def test_block_160m_tier_widths(mode):
    """The 160M tier's widths (d=768, F=52,176; H=2 heads of 64, m_h=26,088, W=256), one
    sequence of 300 tokens compared in full: K = 768 in the projection, three 256-column
    tiles in the output GEMM, 102 gate tiles per head in the aggregation."""
    B, T, d, dqk, m, H, W = 1, 300, 768, 128, 52176, 2, 256
    h, w = synth.block_inputs(B, T, d, dqk, m, seed=13, dtype="bf16")
    out = run_block(h, w, H, mode, W)
    ref = ref_block(h, w, H, mode, W)
    h64 = h.double().numpy()
    assert rel_err(out, ref) <= TOL["bf16"]
    assert rel_err(out.cpu().double() - torch.from_numpy(h64), ref - h64) <= TOL["bf16"]


def test_block_70m_shape_sampled_sequences():
    """The benchmarked configuration (B=8, T=2048, d=512, m=28480, q/k width 128, TANGO,
    bf16): sequences 0 and 7 compared in full against the oracle."""
    B, T, d, dqk, m, H = 8, 2048, 512, 128, 28480, 2
    h, w = synth.block_inputs(B, T, d, dqk, m, seed=0, dtype="bf16")
    out = run_block(h, w, H, 0, 1)
    ref = ref_block(h, w, H, 0, 1, batches=[0, 7])
    got = out[[0, 7]]
    h64 = h[[0, 7]].double().numpy()
    assert rel_err(got, ref) <= TOL["bf16"]
    assert rel_err(got.cpu().double() - torch.from_numpy(h64), ref - h64) <= TOL["bf16"]


def test_bounded_wait_timeout_reports_status():
    """TG_FLAG_DEBUG_TIMEOUT makes the TANGO kernel wait on a barrier that nothing
    signals; the bounded wait runs out, the kernel records a timeout and returns, and
    the context stays usable for the next call."""
    B, T, H, dqk, m = 1, 256, 2, 128, 512
    q, k, g, v = synth.agg_inputs(B, T, dqk, m, seed=3, dtype="bf16")
    qd, kd, gd, vd = q.cuda(), k.cuda(), g.cuda(), v.cuda()
    out = torch.empty_like(gd)
    tg.tango_aggregate(qd, kd, gd, vd, out, H=H, flags=tg.TG_FLAG_DEBUG_TIMEOUT)
    st, word = tg.tg_check_device_error()
    assert st == tg.TG_ERR_TIMEOUT
    assert word & 1 and (word >> 8) & 0xFF == 1
    assert tg.tg_check_device_error() == (tg.TG_OK, 0)      # the word was cleared
    out = run_agg("tango", q, k, g, v, H)
    assert rel_err(out, ref_agg("tango", q, k, g, v, H)) <= TOL["bf16"]


# ------------------------------------------------------------------ model forward

def model_tol(dtype, n_apps=4):
    """Tolerance of the model's logits: the per-operation bound times sqrt(n_apps).  Each
    application adds its own storage roundings (h, x, q, k, g, v, u) and the residual
    path carries earlier errors forward, so independent per-application errors add in
    quadrature.  Measured on GB300 (bf16, d=128): max relative error 0.4-0.85 % after one
    application and 1.1-2.4 % after four; RMS 0.55 % -> 1.2 %, the sqrt(4) growth."""
    return TOL[dtype] * float(np.sqrt(n_apps))


def model_setup(B, T, d, dqk, m, vocab, n_sets, seed, dtype):
    """Token ids, the tied embedding N(0, 0.02^2), unit final gain and n_sets weight sets
    that share gamma, W_q and W_k (each set owns W_g, W_v, W_o)."""
    ids, E = synth.model_inputs(B, T, d, vocab, seed=seed, dtype=dtype)
    _, w = synth.block_inputs(1, 1, d, dqk, m, seed=seed + 1, dtype=dtype)
    sets = [w] + [dict(w, **synth.gated_set(d, m, seed + 2 + k, dtype=dtype)) for k in range(n_sets - 1)]
    gam_f = synth.cast(np.ones(d, dtype=np.float32), dtype)
    return ids, E, gam_f, sets


def run_model(ids, E, gam_f, sets, H, mode, W, n_apps=4):
    B, T = ids.shape
    logits = torch.empty(B, T, E.shape[0], dtype=E.dtype, device="cuda")
    tg.tango_model_forward(ids.to(torch.int32).cuda(), E.cuda(), gam_f.cuda(),
                           [{n: t.cuda() for n, t in w.items()} for w in sets], logits, H=H, n_apps=n_apps,
                           mode=mode, window=W)
    st, word = tg.tg_check_device_error()
    assert st == tg.TG_OK, (st, hex(word))
    return logits


def ref_model(ids, E, gam_f, sets, H, mode, W, n_apps=4):
    return oracle.model_forward(ids.numpy(), synth.oracle_view(E), synth.oracle_view(gam_f),
                                [{n: synth.oracle_view(t) for n, t in w.items()} for w in sets], H=H,
                                tau=10.0, n_apps=n_apps, mode=mode, window=W, rope_base=10000.0,
                                rms_eps=1e-6, final_rms_eps=1e-6)


@pytest.mark.parametrize("mode", [0, 1])
def test_model_tiny_fp32(mode):
    """Four applications of the tiny block (d=64, m=256, q/k width 32, W=16) with a
    1,000-entry tied embedding, fp32, every logit compared."""
    ids, E, gam_f, sets = model_setup(1, 64, 64, 32, 256, 1000, 1, seed=40, dtype="f32")
    out = run_model(ids, E, gam_f, sets, 2, mode, 16)
    assert rel_err(out, ref_model(ids, E, gam_f, sets, 2, mode, 16)) <= model_tol("f32")


@pytest.mark.parametrize("mode", [0, 1])
def test_model_bf16_small(mode):
    ids, E, gam_f, sets = model_setup(2, 100, 128, 64, 512, 1000, 1, seed=41, dtype="bf16")
    out = run_model(ids, E, gam_f, sets, 2, mode, 32)
    assert rel_err(out, ref_model(ids, E, gam_f, sets, 2, mode, 32)) <= model_tol("bf16")
    # one application alone meets the per-operation bound
    one = run_model(ids, E, gam_f, sets, 2, mode, 32, n_apps=1)
    assert rel_err(one, ref_model(ids, E, gam_f, sets, 2, mode, 32, n_apps=1)) <= TOL["bf16"]


@pytest.mark.parametrize("mode", [0, 1])
def test_model_three_sets_unaligned_gate_width(mode):
    """Three gated-projection sets (first / middle / last applications) with a head gate
    width of 47, which the bf16 block pads to 48 internally."""
    ids, E, gam_f, sets = model_setup(2, 150, 128, 64, 94, 1000, 3, seed=42, dtype="bf16")
    out = run_model(ids, E, gam_f, sets, 2, mode, 64)
    assert rel_err(out, ref_model(ids, E, gam_f, sets, 2, mode, 64)) <= model_tol("bf16")
    # the assignment matters: swapping the first and last sets changes the logits
    swapped = run_model(ids, E, gam_f, [sets[2], sets[1], sets[0]], 2, mode, 64)
    assert rel_err(swapped, ref_model(ids, E, gam_f, sets, 2, mode, 64)) > 3 * model_tol("bf16")


@pytest.mark.parametrize("m,n_sets", [(28480, 1), (9494, 3)])
def test_model_shared_block_config_sampled(m, n_sets):
    """The shared-block model configuration: B=16, T=1024, d=512, q/k width 128, four
    TANGO applications, 32,768-entry tied embedding, bf16; one set of m=28,480 or three
    sets of m=9,494.  Sequences 0 and 15 are compared on their first 128 positions,
    which by causality the oracle computes from those positions' tokens alone."""
    B, T, d, dqk, vocab, Tp = 16, 1024, 512, 128, 32768, 128
    ids, E, gam_f, sets = model_setup(B, T, d, dqk, m, vocab, n_sets, seed=43, dtype="bf16")
    out = run_model(ids, E, gam_f, sets, 2, 0, 1)
    got = out[[0, 15], :Tp]
    ref = ref_model(ids[[0, 15], :Tp], E, gam_f, sets, 2, 0, 1)
    assert rel_err(got, ref) <= model_tol("bf16")


@pytest.mark.parametrize("mode", [0, 1])
def test_block_paper_head_geometry(mode):
    """The paper's own head geometry (sec. 2.3: H=16 heads of d_h=32, F=28,480, i.e. 1,780
    gate columns per head, which the bf16 block pads to 1,784; WANGO window 64), d=512,
    T=300 (ragged), every output compared."""
    B, T, d, dqk, m, H, W = 1, 300, 512, 512, 28480, 16, 64
    h, w = synth.block_inputs(B, T, d, dqk, m, seed=11, dtype="bf16")
    out = run_block(h, w, H, mode, W)
    ref = ref_block(h, w, H, mode, W)
    h64 = h.double().numpy()
    assert rel_err(out, ref) <= TOL["bf16"]
    assert rel_err(out.cpu().double() - torch.from_numpy(h64), ref - h64) <= TOL["bf16"]


# ------------------------------------------------------------------ WANGO decode step

def run_decode(q, k, g, v, H, W, **kw):
    """Feeds the sequence one position at a time through wango_decode_step."""
    B, T, dqk = q.shape
    m = g.shape[-1]
    qd, kd, gd = q.cuda(), k.cuda(), g.cuda()
    vd = v.cuda() if v is not None else None
    out = torch.empty_like(gd)
    st = tg.decode_state(B, H, dqk, m, window=W, dtype=tg._dtype_code(gd))
    step_out = torch.empty(B, m, dtype=gd.dtype, device="cuda")
    for i in range(T):
        tg.wango_decode_step(qd[:, i].contiguous(), kd[:, i].contiguous(), gd[:, i].contiguous(),
                             vd[:, i].contiguous() if vd is not None else None, step_out, st, i, H=H, window=W,
                             **kw)
        out[:, i] = step_out
    status, word = tg.tg_check_device_error()
    assert status == tg.TG_OK, (status, hex(word))
    return out


@pytest.mark.parametrize("dtype,case", [
    ("bf16", (2, 100, 2, 32, 256, 16)),
    ("bf16", (1, 64, 2, 32, 256, 1)),      # W = 1: every earlier source is older
    ("bf16", (2, 80, 2, 64, 144, 200)),    # W > T: no older prefix
    ("bf16", (1, 600, 2, 128, 2048, 256)),  # the benchmark window, three steps of state
    ("f32", (1, 50, 2, 32, 256, 7)),
    # per-column gate path: 8-column groups straddle heads (the paper's m_h = 1,780), an
    # odd bf16 width with unaligned rows, an fp32 width that is no multiple of 8
    ("bf16", (2, 90, 2, 64, 3560, 40)),
    ("bf16", (1, 50, 2, 32, 206, 12)),
    ("f32", (1, 60, 2, 32, 150, 9)),
])
def test_decode_steps_match_the_whole_sequence(dtype, case):
    """T decode steps reproduce every row of WANGO over the whole sequence (the oracle's
    running-sum evaluation of eq. 10)."""
    B, T, H, dqk, m, W = case
    q, k, g, v = synth.agg_inputs(B, T, dqk, m, seed=21, dtype=dtype)
    out = run_decode(q, k, g, v, H, W)
    ref = oracle.wango_scan(*[synth.oracle_view(t) for t in (q, k, g, v)], H=H, tau=10.0, window=W)
    assert rel_err(out, ref) <= TOL[dtype]


def test_decode_null_gate_tau_array_and_gbar():
    B, T, H, dqk, m, W = 2, 70, 2, 64, 256, 20
    q, k, g, _ = synth.agg_inputs(B, T, dqk, m, seed=22, dtype="bf16")
    tau = torch.tensor([3.0, 12.0], dtype=torch.float32)
    nb = torch.tensor([-1.0, 0.5], dtype=torch.float32)
    out = run_decode(q, k, g, None, H, W, tau=tau.cuda(), null_bias=nb.cuda(), phi_mode=1)
    ref = oracle.wango_scan(*[synth.oracle_view(t) for t in (q, k, g)], None, H=H, tau=tau.numpy(), window=W,
                            null_bias=nb.numpy(), phi_mode=1)
    assert rel_err(out, ref) <= TOL["bf16"]


def test_wango_segments_hand_over_the_state():
    """160 gate strips for 152 SMs and 8 destination blocks: the launcher splits every
    strip into four segments of two blocks, and each later segment starts from the state
    its predecessor hands over through global memory.  Every row compared against the
    oracle's running sums."""
    B, T, H, dqk, m, W = 1, 1024, 2, 128, 20480, 256
    q, k, g, v = synth.agg_inputs(B, T, dqk, m, seed=31, dtype="bf16")
    out = run_agg("wango", q, k, g, v, H, W)
    ref = oracle.wango_scan(*[synth.oracle_view(t) for t in (q, k, g, v)], H=H, tau=10.0, window=W)
    assert rel_err(out, ref) <= TOL["bf16"]
