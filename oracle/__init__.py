"""fp64 CPU oracle for the cross-token gate aggregation of "TANGO: Token-Aggregated
Nonlinear Gating Operators for Natural and Formal Language Modeling".

TEST INFRASTRUCTURE ONLY.  The test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  Nothing here is shared with,
or called by, the CUDA path (``cross_token_gated_gb300``).

Arrays are numpy arrays: float64, float32, or uint16 holding raw bf16 bit
patterns.  They are widened exactly to fp64 inside the C code (``oracle.c``).

Pins: every function here is checked against closed forms, invariants and the
paper's printed figures in ``tests/test_oracle.py``; none is unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

F64, F32, BF16 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library with gcc (OpenMP when available)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            vp, i, d, ll = ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_longlong
            agg = [i] * 5
            lib.oracle_tango.argtypes = agg + [vp, i, vp, i, vp, i, vp, i, vp, vp, i, vp, ll, vp]
            lib.oracle_wango_direct.argtypes = agg + [i, i] + [vp, i, vp, i, vp, i, vp, i, vp, vp, i,
                                                            vp, ll, vp]
            lib.oracle_wango_scan.argtypes = agg + [i, i] + [vp, i, vp, i, vp, i, vp, i, vp, vp, i, vp]
            lib.oracle_block_forward.argtypes = ([i] * 9 + [d, d] + [vp] * 6 + [i] + [vp, i, vp, vp]
                                                 + [vp, i, vp] + [vp] * 5)
            bwd = [vp, i, vp, i, vp, i, vp, i, vp, i, vp, vp, i, vp, vp, vp, vp]
            lib.oracle_tango_backward.argtypes = agg + bwd
            lib.oracle_wango_backward.argtypes = agg + [i, i] + bwd
            lib.oracle_agg_backward_rows.argtypes = ([i] * 8 + [vp, i, vp, i, vp, i, vp, i, vp, i, vp, vp, i]
                                                     + [vp, i, vp, i, vp, vp, vp, vp])
            lib.oracle_embed.argtypes = [ll, vp, i, i, vp, i, vp]
            lib.oracle_final_logits.argtypes = [ll, i, i, vp, vp, i, d, vp, i, vp]
            for name in ("oracle_tango", "oracle_wango_direct", "oracle_wango_scan",
                         "oracle_block_forward", "oracle_embed", "oracle_final_logits",
                         "oracle_tango_backward", "oracle_wango_backward", "oracle_agg_backward_rows",
                         "oracle_num_threads"):
                getattr(lib, name).restype = ctypes.c_int
            _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def _arr(x):
    """(pointer, dtype code, keep-alive array) for an input array or None."""
    if x is None:
        return None, F64, None
    a = np.ascontiguousarray(x)
    if a.dtype == np.float64:
        code = F64
    elif a.dtype == np.float32:
        code = F32
    elif a.dtype == np.uint16:
        code = BF16
    else:
        raise TypeError(f"oracle input dtype {a.dtype} (want float64, float32 or uint16 bf16 bits)")
    return a.ctypes.data, code, a


def _f64(x, n=None):
    if x is None:
        return None, None
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64).reshape(-1))
    if n is not None and a.size != n:
        raise ValueError(f"expected {n} values, got {a.size}")
    return a.ctypes.data, a


def _rows(rows):
    if rows is None:
        return None, 0, None
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
    return r.ctypes.data, int(r.size), r


def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"{what} failed with status {rc}")


def _tau_vec(tau, H):
    t = np.full(H, float(tau)) if np.isscalar(tau) else np.asarray(tau, dtype=np.float64)
    if t.size != H:
        raise ValueError("tau must be a scalar or have H entries")
    return t


def tango(q, k, g, v, *, H, tau, null_bias=None, qk_normalized=False, rows=None):
    """TANGO aggregation (eqs. 5-6).  q, k: [B, T, dqk]; g, v: [B, T, m] (v may be None,
    then the result is gbar).  rows: optional flat indices b*T+i.  Returns fp64
    [B, T, m] (all rows) or [len(rows), m]."""
    B, T, dqk = q.shape
    m = g.shape[-1]
    qp, qd, qa = _arr(q); kp, kd, ka = _arr(k); gp, gd, ga = _arr(g); vp_, vd, va = _arr(v)
    tp, ta = _f64(_tau_vec(tau, H), H)
    bp, ba = _f64(null_bias, H)
    rp, nr, ra = _rows(rows)
    out = np.empty((nr if rows is not None else B * T, m), dtype=np.float64)
    rc = _load().oracle_tango(B, T, H, dqk, m, qp, qd, kp, kd, gp, gd, vp_, vd, tp, bp,
                              int(bool(qk_normalized)), rp, nr, out.ctypes.data)
    _check(rc, "oracle_tango")
    return out if rows is not None else out.reshape(B, T, m)


def wango_direct(q, k, g, v, *, H, tau, window, phi_mode=0, null_bias=None,
                 qk_normalized=False, rows=None):
    """WANGO aggregation evaluated pair by pair in O(T^2) (eqs. 5-9)."""
    B, T, dqk = q.shape
    m = g.shape[-1]
    qp, qd, qa = _arr(q); kp, kd, ka = _arr(k); gp, gd, ga = _arr(g); vp_, vd, va = _arr(v)
    tp, ta = _f64(_tau_vec(tau, H), H)
    bp, ba = _f64(null_bias, H)
    rp, nr, ra = _rows(rows)
    out = np.empty((nr if rows is not None else B * T, m), dtype=np.float64)
    rc = _load().oracle_wango_direct(B, T, H, dqk, m, int(window), int(phi_mode), qp, qd, kp, kd,
                                     gp, gd, vp_, vd, tp, bp, int(bool(qk_normalized)), rp, nr,
                                     out.ctypes.data)
    _check(rc, "oracle_wango_direct")
    return out if rows is not None else out.reshape(B, T, m)


def _backward(fn, extra, q, k, g, v, dout, H, tau, null_bias, qk_normalized):
    B, T, dqk = q.shape
    m = g.shape[-1]
    qp, qd, qa = _arr(q); kp, kd, ka = _arr(k); gp, gd, ga = _arr(g); vp_, vd, va = _arr(v)
    op, od, oa = _arr(dout)
    tp, ta = _f64(_tau_vec(tau, H), H)
    bp, ba = _f64(null_bias, H)
    dq = np.empty((B, T, dqk)); dk = np.empty((B, T, dqk))
    dg = np.empty((B, T, m)); dv = np.zeros((B, T, m))
    rc = getattr(_load(), fn)(B, T, H, dqk, m, *extra, qp, qd, kp, kd, gp, gd, vp_, vd, op, od, tp, bp,
                              int(bool(qk_normalized)), dq.ctypes.data, dk.ctypes.data, dg.ctypes.data,
                              dv.ctypes.data)
    _check(rc, fn)
    return {"dq": dq, "dk": dk, "dg": dg, "dv": dv if v is not None else None}


def tango_backward(q, k, g, v, dout, *, H, tau, null_bias=None, qk_normalized=False):
    """Gradients of L = sum(dout * u) for the TANGO aggregation u (eqs. 5-6) with respect
    to q, k, g and v (dv is None when v is None, i.e. u = gbar).  Returns a dict of fp64
    arrays dq, dk [B, T, dqk] and dg, dv [B, T, m]."""
    return _backward("oracle_tango_backward", (), q, k, g, v, dout, H, tau, null_bias, qk_normalized)


def wango_backward(q, k, g, v, dout, *, H, tau, window, phi_mode=0, null_bias=None, qk_normalized=False):
    """Gradients of L = sum(dout * u) for the WANGO aggregation (eqs. 5-9), pair by pair."""
    return _backward("oracle_wango_backward", (int(window), int(phi_mode)), q, k, g, v, dout, H, tau,
                     null_bias, qk_normalized)


def backward_rows(kind, q, k, g, v, dout, *, H, tau, rows_q, rows_k, window=1, phi_mode=0, null_bias=None,
                  qk_normalized=False):
    """The gradients of tango_backward / wango_backward (kind "tango" or "wango") at
    selected rows only: dq, dv [len(rows_q), .] for destination rows and dk, dg
    [len(rows_k), .] for source rows (row = b * T + t).  dk of a source needs every later
    destination's gbar, so early sources cost about as much as the full backward."""
    B, T, dqk = q.shape
    m = g.shape[-1]
    qp, qd, qa = _arr(q); kp, kd, ka = _arr(k); gp, gd, ga = _arr(g); vp_, vd, va = _arr(v)
    op, od, oa = _arr(dout)
    tp, ta = _f64(_tau_vec(tau, H), H)
    bp, ba = _f64(null_bias, H)
    rq = np.ascontiguousarray(np.asarray(rows_q, dtype=np.int64))
    rk = np.ascontiguousarray(np.asarray(rows_k, dtype=np.int64))
    dq = np.empty((len(rq), dqk)); dv = np.zeros((len(rq), m))
    dk = np.empty((len(rk), dqk)); dg = np.empty((len(rk), m))
    rc = _load().oracle_agg_backward_rows(0 if kind == "tango" else 1, B, T, H, dqk, m, int(window), int(phi_mode),
                                          qp, qd, kp, kd, gp, gd, vp_, vd, op, od, tp, bp, int(bool(qk_normalized)),
                                          rq.ctypes.data, len(rq), rk.ctypes.data, len(rk), dq.ctypes.data,
                                          dv.ctypes.data, dk.ctypes.data, dg.ctypes.data)
    _check(rc, "oracle_agg_backward_rows")
    return {"dq": dq, "dk": dk, "dg": dg, "dv": dv if v is not None else None}


def wango_scan(q, k, g, v, *, H, tau, window, phi_mode=0, null_bias=None, qk_normalized=False):
    """WANGO aggregation through the running sums S, z of eq. 10 (all rows)."""
    B, T, dqk = q.shape
    m = g.shape[-1]
    qp, qd, qa = _arr(q); kp, kd, ka = _arr(k); gp, gd, ga = _arr(g); vp_, vd, va = _arr(v)
    tp, ta = _f64(_tau_vec(tau, H), H)
    bp, ba = _f64(null_bias, H)
    out = np.empty((B, T, m), dtype=np.float64)
    rc = _load().oracle_wango_scan(B, T, H, dqk, m, int(window), int(phi_mode), qp, qd, kp, kd,
                                   gp, gd, vp_, vd, tp, bp, int(bool(qk_normalized)),
                                   out.ctypes.data)
    _check(rc, "oracle_wango_scan")
    return out


def block_forward(h, weights, *, H, tau, mode=0, window=1, phi_mode=0, null_bias=None,
                  rms_eps=1e-6, rope_base=10000.0, batches=None, intermediates=False):
    """One block application (eqs. 2-10) for the sequences in ``batches`` (default all).

    h: [B, T, d]; weights: dict with gamma [d], Wq/Wk [dqk, d], Wg/Wv [m, d], Wo [d, m],
    all of one dtype.  Returns h_out [nb, T, d] fp64, or (h_out, dict of q, k, g, v, u)
    when ``intermediates`` is set."""
    B, T, d = h.shape
    dqk = weights["Wq"].shape[0]
    m = weights["Wg"].shape[0]
    batches = list(range(B)) if batches is None else list(batches)
    nb = len(batches)
    ws = [_arr(weights[n]) for n in ("gamma", "Wq", "Wk", "Wg", "Wv", "Wo")]
    codes = {w[1] for w in ws}
    if len(codes) != 1:
        raise TypeError("all block weights must share one dtype")
    hp, hd, ha = _arr(h)
    tp, ta = _f64(_tau_vec(tau, H), H)
    bp, ba = _f64(null_bias, H)
    bt = np.ascontiguousarray(np.asarray(batches, dtype=np.int64))
    h_out = np.empty((nb, T, d), dtype=np.float64)
    inter = {}
    ptrs = []
    for name, width in (("q", dqk), ("k", dqk), ("g", m), ("v", m), ("u", m)):
        if intermediates:
            inter[name] = np.empty((nb, T, width), dtype=np.float64)
            ptrs.append(inter[name].ctypes.data)
        else:
            ptrs.append(None)
    rc = _load().oracle_block_forward(B, T, d, H, dqk, m, int(mode), int(window), int(phi_mode),
                                      float(rms_eps), float(rope_base),
                                      *[w[0] for w in ws], ws[0][1], hp, hd, tp, bp,
                                      bt.ctypes.data, nb, h_out.ctypes.data, *ptrs)
    _check(rc, "oracle_block_forward")
    return (h_out, inter) if intermediates else h_out


def embed(ids, E):
    """Token-embedding lookup with the tied matrix E [vocab, d]."""
    ids = np.ascontiguousarray(np.asarray(ids, dtype=np.int64))
    vocab, d = E.shape
    ep, ed, ea = _arr(E)
    out = np.empty(ids.shape + (d,), dtype=np.float64)
    _check(_load().oracle_embed(ids.size, ids.ctypes.data, d, vocab, ep, ed, out.ctypes.data),
           "oracle_embed")
    return out


def final_logits(h, gamma, E, *, rms_eps=1e-6):
    """Final RMSNorm and tied-embedding logits.  h: [..., d] fp64; returns [..., vocab]."""
    h = np.ascontiguousarray(np.asarray(h, dtype=np.float64))
    vocab, d = E.shape
    n = h.size // d
    gp, gd, ga = _arr(gamma)
    ep, ed, ea = _arr(E)
    out = np.empty(h.shape[:-1] + (vocab,), dtype=np.float64)
    _check(_load().oracle_final_logits(n, d, vocab, h.ctypes.data, gp, gd, float(rms_eps), ep, ed,
                                       out.ctypes.data), "oracle_final_logits")
    return out


def default_sets(n_apps, n_sets):
    """Set of each application when the caller gives no table: set 0 throughout for one
    set; for three sets (the revision's abstract and Table 2: narrower gated-projection
    sets for the first, middle and last applications) set 0 first, set 2 last and set 1
    in between."""
    if n_sets == 1:
        return [0] * n_apps
    if n_sets != 3:
        raise ValueError("no default assignment for this many sets")
    return [0 if r == 0 else (2 if r == n_apps - 1 else 1) for r in range(n_apps)]


def model_forward(ids, E, final_gamma, sets, *, H, tau, n_apps=4, set_of_app=None, mode=0, window=1,
                  phi_mode=0, null_bias=None, rms_eps=1e-6, final_rms_eps=1e-6, rope_base=10000.0):
    """The shared-block language model (sec. 2.3 eq. 11): h^(0) = E[ids]; n_apps block
    applications, application r with weight set set_of_app[r]; then the final RMSNorm
    and the tied logits.  Nothing is added between applications.  ids [nb, T'];
    returns logits [nb, T', vocab] in fp64.  By causality the logits of the first T'
    positions depend only on the first T' ids, so a prefix of a longer sequence may be
    passed."""
    ids = np.asarray(ids, dtype=np.int64)
    table = default_sets(n_apps, len(sets)) if set_of_app is None else list(set_of_app)
    h = embed(ids, E)
    for r in range(n_apps):
        h = block_forward(h, sets[table[r]], H=H, tau=tau, mode=mode, window=window, phi_mode=phi_mode,
                          null_bias=null_bias, rms_eps=rms_eps, rope_base=rope_base)
    return final_logits(h, final_gamma, E, rms_eps=final_rms_eps)


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
