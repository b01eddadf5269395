"""Parity of the CUDA path with the fp64 oracle, element by element, on seeded inputs.

Bounds, checked by `check` on every output tensor (the oracle reads exactly the values
the GPU reads: bf16 inputs are widened, not re-rounded):
- normwise: max |gpu - oracle| / max |oracle| <= TOL, i.e. 1e-4 for fp32 storage (CUDA
  core fp32 arithmetic) and 2e-2 for bf16 storage (bf16 tensor-core operands, fp32
  accumulation);
- per row and head (the gate columns of one head in one output row): the same ratio
  within each, <= 2 TOL.  A row holds far fewer elements than the tensor, so its
  largest value sits closer to its typical ones; this keeps an error confined to rows
  or heads of small magnitude from hiding behind the tensor's largest values;
- element-wise, for aggregation outputs: |gpu - oracle| / scale <= COND_TOL, where
  scale = sum_j alpha_ij |g_j| |v_i| is the oracle's own aggregation of |g| and |v|
  (the weights alpha do not depend on g).  A weighted average computed with relative
  weight errors e_j is off by sum_j alpha_j e_j (g_j - gbar), at most 2 max|e| times
  that scale, so this bound holds element by element, even where the output is near
  zero through cancellation.  In bf16 the weights carry the rounding of qhat, khat (a
  logit error of up to tau 2^-8) and of P (2^-9).
The plain element-wise ratio |gpu - oracle| / (|oracle| + 1e-3 rms(oracle)) is
computed and reported (TG_PARITY_REPORT) but not bounded: an
output element that cancels to near zero keeps the absolute error of the weights, and
the ratio then measures the cancellation, not the kernel.  With TG_PARITY_REPORT=<path>
every check appends its figures as one JSON line to that file.
"""
import json
import os

import numpy as np
import pytest
import torch

import cross_token_gated_gb300 as tg
import oracle
from cross_token_gated_gb300 import synth

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}
COND_TOL = {"f32": 1e-4, "bf16": 4e-2}


def as_f64(gpu: torch.Tensor, shape) -> np.ndarray:
    g = gpu.detach().double().cpu().numpy().reshape(shape)
    assert np.all(np.isfinite(g)), "non-finite values in the GPU output"
    return g


def rel_err(gpu: torch.Tensor, ref: np.ndarray) -> float:
    """Normwise relative error max |gpu - ref| / max |ref| over the whole tensor."""
    g = as_f64(gpu, ref.shape)
    return float(np.max(np.abs(g - ref)) / max(np.max(np.abs(ref)), 1e-30))


def errors(gpu: torch.Tensor, ref: np.ndarray, H: int = 1, scale=None) -> dict:
    """Normwise, worst per-(row, head), plain element-wise and (with `scale`)
    condition-normalised element-wise errors.  Rows are the last axis; H splits it into
    heads of equal width."""
    g = as_f64(gpu, ref.shape)
    d = np.abs(g - ref)
    a = np.abs(ref)
    n = ref.shape[-1]
    H = H if n % H == 0 else 1
    dr, ar = d.reshape(-1, H, n // H), a.reshape(-1, H, n // H)
    rms = float(np.sqrt(np.mean(ref * ref)))
    out = {"norm": float(d.max() / max(a.max(), 1e-30)),
           "row_head": float(np.max(dr.max(-1) / np.maximum(ar.max(-1), 1e-30))),
           "elem_rms": float(np.max(d / (a + 1e-3 * rms)))}
    if scale is not None:
        out["elem_cond"] = float(np.max(d / np.maximum(np.asarray(scale).reshape(ref.shape), 1e-30)))
    return out


def check(gpu: torch.Tensor, ref: np.ndarray, dtype: str, H: int = 1, scale=None):
    e = errors(gpu, ref, H, scale)
    path = os.environ.get("TG_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(dict(test=os.environ.get("PYTEST_CURRENT_TEST", ""), dtype=dtype, **e)) + "\n")
    assert e["norm"] <= TOL[dtype], ("normwise", e)
    assert e["row_head"] <= 2 * TOL[dtype], ("per row and head", e)
    if scale is not None:
        assert e["elem_cond"] <= COND_TOL[dtype], ("element-wise", e)


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


def abs_inputs(g, v):
    """|g| and |v| (exact in either storage type): the oracle's aggregation of them is the
    element-wise error scale sum_j alpha_ij |g_j| |v_i|."""
    return g.abs(), (v.abs() if v is not None else None)


def ref_agg_scaled(kind, q, k, g, v, H, W=16, **kw):
    """(oracle output, element-wise error scale) for one aggregation."""
    ga, va = abs_inputs(g, v)
    return ref_agg(kind, q, k, g, v, H, W, **kw), ref_agg(kind, q, k, ga, va, H, W, **kw)


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
    ref, scale = ref_agg_scaled(kind, q, k, g, v, H, W)
    check(out, ref, dtype, H, scale)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("case", SMALL, ids=[f"B{c[0]}T{c[1]}H{c[2]}dqk{c[3]}m{c[4]}W{c[5]}" for c in SMALL])
def test_wango_plain_elu_feature_map(dtype, case):
    """phi_mode = 1, the literal phi(u) = elu(u) + 1 of the benchmark configurations
    (no epsilon, no 1/sqrt(d_h)), through the same kernels: the feature-map pre-pass
    computes Fq and Fk with it, and every older-prefix weight and the state read-out use
    them."""
    B, T, H, dqk, m, W = case
    q, k, g, v = synth.agg_inputs(B, T, dqk, m, seed=T + m + 1, dtype=dtype)
    out = run_agg("wango", q, k, g, v, H, W, phi_mode=1)
    ref, scale = ref_agg_scaled("wango", q, k, g, v, H, W, phi_mode=1)
    check(out, ref, dtype, H, scale)


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
    ref, scale = ref_agg_scaled(kind, q, k, g, None, H, W, s=[10.0, 4.0], null_bias=[-1.0, 0.5])
    check(out, ref, dtype, H, scale)
    # unit vectors in, no normalisation inside
    qn = q.double().reshape(B, T, H, -1)
    qn = (qn / qn.norm(dim=-1, keepdim=True)).reshape(B, T, dqk).to(q.dtype)
    kn = k.double().reshape(B, T, H, -1)
    kn = (kn / kn.norm(dim=-1, keepdim=True)).reshape(B, T, dqk).to(k.dtype)
    out2 = run_agg(kind, qn, kn, g, None, H, W, tau=tau, null_bias=nb, flags=tg.TG_FLAG_QK_NORMALIZED)
    ref2, scale2 = ref_agg_scaled(kind, qn, kn, g, None, H, W, s=[10.0, 4.0], null_bias=[-1.0, 0.5],
                                  qk_normalized=True)
    check(out2, ref2, dtype, H, scale2)


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
    ref, scale = ref_agg_scaled(kind, q, k, g, v, H, W, rows=rows)
    got = out.reshape(B * T, m)[torch.from_numpy(rows).cuda()]
    check(got, ref, "bf16", H, scale)


def test_wango_70m_shape_plain_elu_sampled():
    """The WANGO benchmark configuration as written (phi = elu + 1 on the 64 feature
    dimensions of each head): B=8, T=2048, m=28480, W=256, bf16, sampled rows."""
    B, T, H, dqk, m, W = 8, 2048, 2, 128, 28480, 256
    q, k, g, v = synth.agg_inputs(B, T, dqk, m, seed=4, dtype="bf16")
    out = run_agg("wango", q, k, g, v, H, W, phi_mode=1)
    extra = [0, 255, 256, 257, 383, 384, 1000, 2047, 5 * T + 300, 7 * T + 2047]
    rows = synth.random_rows(B, T, 30, seed=5, extra=extra)
    ref, scale = ref_agg_scaled("wango", q, k, g, v, H, W, rows=rows, phi_mode=1)
    got = out.reshape(B * T, m)[torch.from_numpy(rows).cuda()]
    check(got, ref, "bf16", H, scale)


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
    ref, scale = ref_agg_scaled(kind, q, k, g, v, H, W, rows=rows)
    got = out.reshape(B * T, m)[torch.from_numpy(rows).cuda()]
    check(got, ref, "bf16", H, scale)


# ------------------------------------------------------------------ block forward

def run_block(h, w, H, mode, W, **kw):
    hd = h.cuda()
    wd = {n: t.cuda() for n, t in w.items()}
    out = torch.empty_like(hd)
    tg.tango_block_forward(hd, wd, out, H=H, mode=mode, window=W, **kw)
    st, word = tg.tg_check_device_error()
    assert st == tg.TG_OK, (st, hex(word))
    return out


def ref_block(h, w, H, mode, W, batches=None, s=10.0, phi_mode=0):
    wv = {n: synth.oracle_view(t) for n, t in w.items()}
    return oracle.block_forward(synth.oracle_view(h), wv, H=H, tau=s, mode=mode, window=W, phi_mode=phi_mode,
                                batches=batches, rope_base=10000.0, rms_eps=1e-6)


@pytest.mark.parametrize("mode", [0, 1])
def test_block_tiny_fp32(mode):
    """The tiny oracle configuration: B=1, T=64, d=64, m=256, q/k width 32, W=16, fp32."""
    B, T, d, dqk, m, H, W = 1, 64, 64, 32, 256, 2, 16
    h, w = synth.block_inputs(B, T, d, dqk, m, seed=0, dtype="f32")
    out = run_block(h, w, H, mode, W)
    ref = ref_block(h, w, H, mode, W)
    h64 = h.double().numpy()
    check(out, ref, "f32")
    check(out.cpu().double() - torch.from_numpy(h64), ref - h64, "f32")


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("shape", [(2, 100, 128, 64, 512, 2, 32), (1, 257, 128, 128, 1040, 2, 100)])
def test_block_bf16_small(mode, shape):
    B, T, d, dqk, m, H, W = shape
    h, w = synth.block_inputs(B, T, d, dqk, m, seed=5, dtype="bf16")
    out = run_block(h, w, H, mode, W)
    ref = ref_block(h, w, H, mode, W)
    h64 = h.double().numpy()
    check(out, ref, "bf16")
    check(out.cpu().double() - torch.from_numpy(h64), ref - h64, "bf16")


@pytest.mark.parametrize("shape", [(2, 100, 128, 64, 512, 2, 32), (1, 600, 512, 128, 28480, 2, 256)])
def test_block_wango_plain_elu(shape):
    """The WANGO block with phi = elu + 1 (the benchmark configuration's feature map):
    a small shape, and one 600-token sequence at the 70M-tier widths with W=256, every
    output compared."""
    B, T, d, dqk, m, H, W = shape
    h, w = synth.block_inputs(B, T, d, dqk, m, seed=6, dtype="bf16")
    out = run_block(h, w, H, 1, W, phi_mode=1)
    ref = ref_block(h, w, H, 1, W, phi_mode=1)
    h64 = h.double().numpy()
    check(out, ref, "bf16")
    check(out.cpu().double() - torch.from_numpy(h64), ref - h64, "bf16")


@pytest.mark.parametrize("shape", [(2, 100, 128, 64, 512, 2, 32), (1, 2048, 512, 128, 4096, 2, 256),
                                   (1, 300, 768, 128, 2 * 4747, 2, 64)])
def test_block_wango_fused_v_and_separate_v(shape):
    """With TG_FLAG_FUSED_V the WANGO block forms v = W_v x inside the aggregation kernel
    (v never stored); by default v comes from the projection GEMM.  Both are compared with
    the oracle in full, on shapes that cover 2 and 12 chunks of the residual width, strips
    split into segments (few strips, long sequence), and the padded per-head gate pitch
    (m_h = 4,747); the two paths compute v with the same chunks in the same order, so
    their outputs agree to within a bf16 rounding of the residual."""
    B, T, d, dqk, m, H, W = shape
    h, w = synth.block_inputs(B, T, d, dqk, m, seed=17, dtype="bf16")
    fused = run_block(h, w, H, 1, W, flags=tg.TG_FLAG_FUSED_V)
    separate = run_block(h, w, H, 1, W)
    ref = ref_block(h, w, H, 1, W)
    h64 = h.double().numpy()
    for out in (fused, separate):
        check(out, ref, "bf16")
        check(out.cpu().double() - torch.from_numpy(h64), ref - h64, "bf16")
    diff = (fused.double() - separate.double()).abs().max().item()
    assert diff <= 2 * 2.0 ** -8 * h.double().abs().max().item(), diff


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
    check(out, ref, "bf16")
    check(out.cpu().double() - torch.from_numpy(h64), ref - h64, "bf16")


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
    check(out, ref, "bf16")
    check(out.cpu().double() - torch.from_numpy(h64), ref - h64, "bf16")


def test_block_70m_shape_sampled_sequences():
    """The benchmarked configuration (B=8, T=2048, d=512, m=28480, q/k width 128, TANGO,
    bf16): sequences 0 and 7 compared in full against the oracle."""
    B, T, d, dqk, m, H = 8, 2048, 512, 128, 28480, 2
    h, w = synth.block_inputs(B, T, d, dqk, m, seed=0, dtype="bf16")
    out = run_block(h, w, H, 0, 1)
    ref = ref_block(h, w, H, 0, 1, batches=[0, 7])
    got = out[[0, 7]]
    h64 = h[[0, 7]].double().numpy()
    check(got, ref, "bf16")
    check(got.cpu().double() - torch.from_numpy(h64), ref - h64, "bf16")


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
    ref, scale = ref_agg_scaled("tango", q, k, g, v, H)
    check(out, ref, "bf16", H, scale)


@pytest.mark.parametrize("T,m", [(700, 1040), (1024, 20480)])
def test_bounded_wait_timeout_reports_status_wango(T, m):
    """The same hook in the WANGO gate-strip kernel: its MMA issuer waits on a barrier
    that nothing signals, runs out (1 ms), records a timeout and every role leaves its
    loops.  The second shape splits the strips into segments, so later segments also
    give up (bounded) on the state their aborted predecessors never hand over.  The
    context stays usable: the next call is correct."""
    B, H, dqk, W = 1, 2, 128, 256
    q, k, g, v = synth.agg_inputs(B, T, dqk, m, seed=8, dtype="bf16")
    qd, kd, gd, vd = q.cuda(), k.cuda(), g.cuda(), v.cuda()
    out = torch.empty_like(gd)
    tg.wango_aggregate(qd, kd, gd, vd, out, H=H, window=W, flags=tg.TG_FLAG_DEBUG_TIMEOUT)
    st, word = tg.tg_check_device_error()
    assert st == tg.TG_ERR_TIMEOUT
    assert word & 1 and (word >> 8) & 0xFF == 2
    assert tg.tg_check_device_error() == (tg.TG_OK, 0)
    out = run_agg("wango", q, k, g, v, H, W)
    rows = synth.random_rows(B, T, 12, seed=9, extra=[0, 255, 256, T - 1])
    ref, scale = ref_agg_scaled("wango", q, k, g, v, H, W, rows=rows)
    check(out.reshape(B * T, m)[torch.from_numpy(rows).cuda()], ref, "bf16", H, scale)


def test_bounded_wait_timeout_reports_status_gemm():
    """In tango_block_forward the flag arms the hook of the projection GEMM only: its
    MMA issuer waits on a barrier that nothing signals, runs out (1 ms), and the GEMM
    records its timeout (kernel code 3).  The rest of the block then runs on whatever
    the workspace held, without faults; the next block call is correct."""
    B, T, d, dqk, m, H = 1, 256, 512, 128, 1024, 2
    h, w = synth.block_inputs(B, T, d, dqk, m, seed=12, dtype="bf16")
    hd = h.cuda()
    wd = {n: t.cuda() for n, t in w.items()}
    out = torch.empty_like(hd)
    tg.tango_block_forward(hd, wd, out, H=H, flags=tg.TG_FLAG_DEBUG_TIMEOUT)
    st, word = tg.tg_check_device_error()
    assert st == tg.TG_ERR_TIMEOUT
    assert word & 1 and (word >> 8) & 0xFF == 3
    assert tg.tg_check_device_error() == (tg.TG_OK, 0)
    out = run_block(h, w, H, 0, 1)
    check(out, ref_block(h, w, H, 0, 1), "bf16")


# ------------------------------------------------------------------ model forward

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


# The model's logits are held to the same bounds as one operation.  In bf16 they are met
# at the benchmark's widths: four applications at d = 512 and m >= 4,096.  At smaller
# widths (d = 128, or m in the hundreds) bf16 storage of the GEMM operands alone, x and u,
# gives 1.5-2.7 % after four applications, whether the residual stream is bf16 or fp32:
# the output projection's sum over m averages fewer independent roundings.

@pytest.mark.parametrize("mode", [0, 1])
def test_model_tiny_fp32(mode):
    """Four applications of the tiny block (d=64, m=256, q/k width 32, W=16) with a
    1,000-entry tied embedding, fp32, every logit compared."""
    ids, E, gam_f, sets = model_setup(1, 64, 64, 32, 256, 1000, 1, seed=40, dtype="f32")
    out = run_model(ids, E, gam_f, sets, 2, mode, 16)
    check(out, ref_model(ids, E, gam_f, sets, 2, mode, 16), "f32")


@pytest.mark.parametrize("mode", [0, 1])
def test_model_bf16_small(mode):
    """Four applications at d=512, m=4,096 (two heads of 2,048 gates), T=100, every
    logit compared; one application alone too."""
    ids, E, gam_f, sets = model_setup(2, 100, 512, 128, 4096, 1000, 1, seed=41, dtype="bf16")
    out = run_model(ids, E, gam_f, sets, 2, mode, 32)
    check(out, ref_model(ids, E, gam_f, sets, 2, mode, 32), "bf16")
    one = run_model(ids, E, gam_f, sets, 2, mode, 32, n_apps=1)
    check(one, ref_model(ids, E, gam_f, sets, 2, mode, 32, n_apps=1), "bf16")


@pytest.mark.parametrize("mode", [0, 1])
def test_model_three_sets_unaligned_gate_width(mode):
    """Three gated-projection sets (first / middle / last applications) of m=9,494, i.e.
    a head gate width of 4,747, which the bf16 block pads to 4,752 internally; T=150,
    every logit compared."""
    ids, E, gam_f, sets = model_setup(2, 150, 512, 128, 9494, 1000, 3, seed=42, dtype="bf16")
    out = run_model(ids, E, gam_f, sets, 2, mode, 64)
    ref = ref_model(ids, E, gam_f, sets, 2, mode, 64)
    check(out, ref, "bf16")
    # the assignment matters: swapping the first and last sets changes the logits
    swapped = run_model(ids, E, gam_f, [sets[2], sets[1], sets[0]], 2, mode, 64)
    assert rel_err(swapped, ref) > 3 * TOL["bf16"]


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
    check(got, ref, "bf16")


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
    check(out, ref, "bf16")
    check(out.cpu().double() - torch.from_numpy(h64), ref - h64, "bf16")


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
    # one sequence: 64-column blocks that straddle two heads, and a window wider than the
    # 9-slot register batch of the ring (W + 8 = 608 slots: several batches)
    ("bf16", (1, 120, 2, 64, 272, 24)),
    ("bf16", (1, 700, 2, 64, 512, 600)),
    ("bf16", (4, 60, 2, 64, 512, 16)),     # four sequences: the plain launch
    ("bf16", (3, 50, 2, 64, 256, 41)),     # the last group of 8 still waiting at the end
    ("f32", (3, 60, 2, 64, 256, 20)),      # three sequences in fp32: the plain launch's vectors
    ("bf16", (4, 80, 1, 128, 512, 30)),    # one head of 128: two batches of 4 state rows a thread
])
def test_decode_steps_match_the_whole_sequence(dtype, case):
    """T decode steps reproduce every row of WANGO over the whole sequence (the oracle's
    running-sum evaluation of eq. 10).  Sources that left the window enter S in groups of
    8, so every case with T > W + 8 crosses several group boundaries, and W = 1 folds
    the current token's own group."""
    B, T, H, dqk, m, W = case
    q, k, g, v = synth.agg_inputs(B, T, dqk, m, seed=21, dtype=dtype)
    out = run_decode(q, k, g, v, H, W)
    ref = oracle.wango_scan(*[synth.oracle_view(t) for t in (q, k, g, v)], H=H, tau=10.0, window=W)
    scale = oracle.wango_scan(*[synth.oracle_view(t) for t in (q, k, *abs_inputs(g, v))], H=H, tau=10.0,
                              window=W)
    check(out, ref, dtype, H, scale)


def test_decode_null_gate_tau_array_and_gbar():
    B, T, H, dqk, m, W = 2, 70, 2, 64, 256, 20
    q, k, g, _ = synth.agg_inputs(B, T, dqk, m, seed=22, dtype="bf16")
    tau = torch.tensor([3.0, 12.0], dtype=torch.float32)
    nb = torch.tensor([-1.0, 0.5], dtype=torch.float32)
    out = run_decode(q, k, g, None, H, W, tau=tau.cuda(), null_bias=nb.cuda(), phi_mode=1)
    kw = dict(H=H, tau=tau.numpy(), window=W, null_bias=nb.numpy(), phi_mode=1)
    ref = oracle.wango_scan(*[synth.oracle_view(t) for t in (q, k, g)], None, **kw)
    scale = oracle.wango_scan(*[synth.oracle_view(t) for t in (q, k, g.abs())], None, **kw)
    check(out, ref, "bf16", H, scale)


def test_wango_segments_hand_over_the_state():
    """160 gate strips for 152 SMs and 8 destination blocks: the launcher splits every
    strip into four segments of two blocks, and each later segment starts from the state
    its predecessor hands over through global memory.  Every row compared against the
    oracle's running sums."""
    B, T, H, dqk, m, W = 1, 1024, 2, 128, 20480, 256
    q, k, g, v = synth.agg_inputs(B, T, dqk, m, seed=31, dtype="bf16")
    out = run_agg("wango", q, k, g, v, H, W)
    ref = oracle.wango_scan(*[synth.oracle_view(t) for t in (q, k, g, v)], H=H, tau=10.0, window=W)
    scale = oracle.wango_scan(*[synth.oracle_view(t) for t in (q, k, *abs_inputs(g, v))], H=H, tau=10.0,
                              window=W)
    check(out, ref, "bf16", H, scale)


def pitched(t, H, pitch, fill):
    """[B, T, H*m_h] -> [B, T, H*pitch] with each head's gates first and `fill` after them."""
    B, T, m = t.shape
    m_h = m // H
    out = torch.full((B, T, H, pitch), fill, dtype=t.dtype)
    out[..., :m_h] = t.view(B, T, H, m_h)
    return out.view(B, T, H * pitch)


@pytest.mark.parametrize("kind,W", [("tango", 1), ("wango", 16), ("wango", 300)])
@pytest.mark.parametrize("dtype,pitch", [("bf16", 4752), ("f32", 4750)])
def test_agg_gate_pitch(kind, W, dtype, pitch):
    """The revision's three-set head width m_h = 4,747 through the aggregate calls at a
    padded per-head pitch (m_pitch): the padding columns of g and v hold NaN, which must
    reach no gate column (the padding columns of the output are unspecified)."""
    B, T, H, dqk, m_h = 1, 300, 2, 128, 4747
    q, k, g, v = synth.agg_inputs(B, T, dqk, H * m_h, seed=41, dtype=dtype)
    gp, vp = (pitched(t, H, pitch, float("nan")).cuda() for t in (g, v))
    out = torch.full_like(gp, 7.0)
    kw = dict(H=H, m_h=m_h)
    if kind == "tango":
        tg.tango_aggregate(q.cuda(), k.cuda(), gp, vp, out, **kw)
    else:
        tg.wango_aggregate(q.cuda(), k.cuda(), gp, vp, out, window=W, **kw)
    st, word = tg.tg_check_device_error()
    assert st == tg.TG_OK, (st, hex(word))
    o4 = out.view(B, T, H, pitch)
    got = o4[..., :m_h].reshape(B, T, H * m_h)
    ref, scale = ref_agg_scaled(kind, q, k, g, v, H, W)
    check(got, ref, dtype, H=H, scale=scale)
    if dtype == "f32":  # bf16 stores 16-byte vectors, which may run into the padding
        assert bool((o4[..., m_h:] == 7.0).all())


def _bf16(x: np.ndarray) -> np.ndarray:
    """Round to bf16 (nearest even) and widen back to fp64."""
    return torch.from_numpy(np.asarray(x, dtype=np.float64)).float().bfloat16().double().numpy()


def _widen(x: np.ndarray) -> np.ndarray:
    """The oracle view of a bf16 tensor (its raw 16-bit patterns) widened to fp64."""
    return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("case", [(2, 143, 4, 64, 1152), (1, 300, 2, 128, 1040), (1, 1, 2, 32, 256)])
def test_tango_matches_its_rounding_points(case):
    """The bf16 TANGO path against an fp64 emulation of the rounding points the kernel
    documents (qhat and khat in bf16, each weight rounded to bf16 before it is summed into
    the denominator and multiplied with g, gbar rounded to bf16, u = gbar * v rounded to
    bf16), in bf16 steps of the output: what is left is the fp32 accumulation order and
    the exponential's last bits, so a wrong mask, index or rounding point would show."""
    B, T, H, dqk, m = case
    s = 10.0
    q, k, g, v = synth.agg_inputs(B, T, dqk, m, seed=B * T + m, dtype="bf16")
    out = run_agg("tango", q, k, g, v, H, s=s)
    qv, kv, gv, vv = (_widen(synth.oracle_view(t)) for t in (q, k, g, v))
    d_h, m_h = dqk // H, m // H
    emu = np.zeros((B, T, m))
    causal = np.tril(np.ones((T, T)))
    for b in range(B):
        for a in range(H):
            qa, ka = qv[b, :, a * d_h:(a + 1) * d_h], kv[b, :, a * d_h:(a + 1) * d_h]
            qh = _bf16(qa / np.maximum(np.linalg.norm(qa, axis=1, keepdims=True), 1e-12))
            kh = _bf16(ka / np.maximum(np.linalg.norm(ka, axis=1, keepdims=True), 1e-12))
            P = _bf16(np.exp(s * (qh @ kh.T - 1.0))) * causal
            gbar = _bf16((P @ gv[b, :, a * m_h:(a + 1) * m_h]) / P.sum(1)[:, None])
            emu[b, :, a * m_h:(a + 1) * m_h] = _bf16(gbar * vv[b, :, a * m_h:(a + 1) * m_h])
    # distances in bf16 steps (units in the last place) between the GPU's u and the
    # emulation rounded to bf16
    def key(t):
        b = t.contiguous().view(torch.int16).to(torch.int32)
        return torch.where(b < 0, -(b & 0x7FFF), b)
    emu16 = torch.from_numpy(emu.reshape(-1)).bfloat16()
    ulps = (key(out.cpu().reshape(-1)) - key(emu16)).abs()
    got = as_f64(out, emu.shape)
    stats = {"differ": float((ulps > 0).double().mean()), "over1": float((ulps > 1).double().mean()),
             "norm": float(np.abs(got - emu16.double().numpy().reshape(emu.shape)).max() / np.abs(emu).max())}
    print("distance to the emulation:", stats)
    # almost every element is the same bf16 value (measured: all but 0.01-0.1 %); where a
    # weight's rounding flips, the output moves by a fraction of a bf16 step of the
    # largest outputs (measured 5.8e-4 of the largest)
    assert stats["differ"] <= 5e-3 and stats["norm"] <= 2.0 ** -9, stats


@pytest.mark.parametrize("case,null", [((1, 300, 2, 128, 1040, 16), False), ((1, 300, 2, 128, 1040, 100), False),
                                       ((2, 520, 2, 64, 272, 256), False), ((1, 700, 2, 128, 272, 200), False),
                                       ((1, 600, 4, 64, 128, 300), True)])  # d_h = 16, null gate
def test_wango_matches_its_rounding_points(case, null):
    """The bf16 WANGO path against an fp64 emulation of the rounding points its kernels
    document: Fq = bf16(e^-tau phi(sqrt(tau) qhat)) and Fk = bf16(phi(sqrt(tau) khat))
    from bf16 unit vectors; for destination block ib the source blocks jlo(ib)..ib give
    bf16 weights (window pairs exp(tau (qhat.khat - 1)), older pairs Fq.Fk, zero after
    the row), every older block through the state S = sum Fk g^T read out as Fq .
    bf16(S); the denominator sums the rounded weights, Fq . z (z the sums of the rounded
    Fk below the window) and, with the null gate, (i + 1) e^(b - tau); gbar and u rounded
    to bf16.  Compared in bf16 steps of the output, like the TANGO case."""
    B, T, H, dqk, m, W = case
    s = 10.0
    q, k, g, v = synth.agg_inputs(B, T, dqk, m, seed=B * T + m + W, dtype="bf16")
    nb = np.linspace(-1.0, 0.5, H) if null else np.full(H, -np.inf)
    out = run_agg("wango", q, k, g, v, H, W, s=s,
                  null_bias=torch.tensor(nb, dtype=torch.float32).cuda() if null else None)
    qv, kv, gv, vv = (_widen(synth.oracle_view(t)) for t in (q, k, g, v))
    d_h, m_h = dqk // H, m // H
    nblk = -(-T // 128)

    def phi(u):  # eq. 8
        return np.maximum(np.where(u > 0, u + 1.0, np.exp(np.minimum(u, 0.0))) + 1e-4, 1e-4) / np.sqrt(d_h)

    emu = np.zeros((B, T, m))
    for b in range(B):
        for a in range(H):
            qa, ka = qv[b, :, a * d_h:(a + 1) * d_h], kv[b, :, a * d_h:(a + 1) * d_h]
            ga, va = gv[b, :, a * m_h:(a + 1) * m_h], vv[b, :, a * m_h:(a + 1) * m_h]
            qh = _bf16(qa / np.maximum(np.linalg.norm(qa, axis=1, keepdims=True), 1e-12))
            kh = _bf16(ka / np.maximum(np.linalg.norm(ka, axis=1, keepdims=True), 1e-12))
            fq = _bf16(np.exp(-s) * phi(np.sqrt(s) * qh))
            fk = _bf16(phi(np.sqrt(s) * kh))
            zb = np.array([fk[128 * j:min(T, 128 * j + 128)].sum(0) for j in range(nblk)])
            for ib in range(nblk):
                i0, i1 = 128 * ib, min(T, 128 * ib + 128)
                jlo = max(0, 128 * ib - W + 1) // 128
                j0 = 128 * jlo
                ii = np.arange(i0, i1)[:, None]
                jj = np.arange(j0, i1)[None, :]
                win = _bf16(np.exp(s * (qh[i0:i1] @ kh[j0:i1].T - 1.0)))
                old = _bf16(fq[i0:i1] @ fk[j0:i1].T)
                P = np.where(jj > ii, 0.0, np.where(jj >= ii - W + 1, win, old))
                S = _bf16(fk[:j0].T @ ga[:j0])           # the state before the block, as read out
                z = zb[:jlo].sum(0)
                num = P @ ga[j0:i1] + fq[i0:i1] @ S
                den = P.sum(1) + fq[i0:i1] @ z + (np.arange(i0, i1) + 1.0) * np.exp(nb[a] - s)
                emu[b, i0:i1, a * m_h:(a + 1) * m_h] = _bf16(_bf16(num / den[:, None]) * va[i0:i1])

    def key(t):
        b_ = t.contiguous().view(torch.int16).to(torch.int32)
        return torch.where(b_ < 0, -(b_ & 0x7FFF), b_)
    emu16 = torch.from_numpy(emu.reshape(-1)).bfloat16()
    ulps = (key(out.cpu().reshape(-1)) - key(emu16)).abs()
    got = as_f64(out, emu.shape)
    stats = {"differ": float((ulps > 0).double().mean()), "over1": float((ulps > 1).double().mean()),
             "norm": float(np.abs(got - emu16.double().numpy().reshape(emu.shape)).max() / np.abs(emu).max())}
    print("distance to the emulation:", stats)
    # measured: 0.1-1.7 % of the outputs differ (the fp32 state and accumulation orders
    # flip a bf16 rounding now and then), normwise at most 1.2e-3
    assert stats["differ"] <= 5e-2 and stats["norm"] <= 2.0 ** -8, stats
