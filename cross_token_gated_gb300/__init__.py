"""GB300-native cross-token gate aggregation (TANGO / WANGO).

Python binding of the C-ABI library declared in ``include/tango.h``.  The binding
only marshals arguments: every step of the path runs in the library's CUDA
kernels.  PyTorch supplies device memory and streams.  There is no fallback: if
the library cannot be loaded, every call raises.

Functions (same names as the C ABI):
  tango_aggregate, tango_aggregate_noalloc, wango_aggregate, tango_aggregate_save,
  wango_aggregate_save, tango_aggregate_backward, wango_aggregate_backward, wango_decode_step, tango_block_forward, tango_model_forward,
  tg_workspace_size, tg_status_string, tg_check_device_error, tg_version
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

from . import build as _build

TG_OK, TG_ERR_INVALID_ARG, TG_ERR_UNSUPPORTED, TG_ERR_WORKSPACE, TG_ERR_CUDA, TG_ERR_TIMEOUT, \
    TG_ERR_DEVICE = range(7)
TG_F32, TG_BF16 = 0, 1
TG_FLAG_QK_NORMALIZED = 0x1
TG_FLAG_DEBUG_TIMEOUT = 0x100
TG_FLAG_FUSED_V = 0x200
TG_FLAG_BWD_FAR_SCAN = 0x400
TG_FLAG_BWD_FAR_PAIRS = 0x800
TG_MODE_TANGO, TG_MODE_WANGO = 0, 1
TG_WS_TANGO, TG_WS_WANGO, TG_WS_BLOCK, TG_WS_MODEL, TG_WS_DECODE, TG_WS_TANGO_BWD, TG_WS_WANGO_BWD = range(7)

HEADER = os.path.join(_build.INCLUDE, "tango.h")


class TgError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} (status {status})")
        self.status = status


class tg_agg_params(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("H", ctypes.c_int), ("d_qk", ctypes.c_int),
                ("m", ctypes.c_int), ("s", ctypes.c_float), ("tau", ctypes.c_void_p),
                ("null_bias", ctypes.c_void_p), ("window", ctypes.c_int), ("phi_mode", ctypes.c_int),
                ("flags", ctypes.c_uint), ("dtype", ctypes.c_int), ("m_pitch", ctypes.c_int)]


class tg_block_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("rms_gamma", "Wq", "Wk", "Wg", "Wv", "Wo")]


class tg_block_params(ctypes.Structure):
    _fields_ = [("agg", tg_agg_params), ("d", ctypes.c_int), ("mode", ctypes.c_int),
                ("rms_eps", ctypes.c_float), ("rope_base", ctypes.c_float)]


class tg_model_weights(ctypes.Structure):
    _fields_ = [("embedding", ctypes.c_void_p), ("final_gamma", ctypes.c_void_p),
                ("sets", ctypes.POINTER(tg_block_weights))]


class tg_model_params(ctypes.Structure):
    _fields_ = [("block", tg_block_params), ("vocab", ctypes.c_int), ("n_apps", ctypes.c_int),
                ("n_sets", ctypes.c_int), ("set_of_app", ctypes.POINTER(ctypes.c_int)),
                ("final_rms_eps", ctypes.c_float)]


_lib = None
_lock = threading.Lock()


def declared_functions() -> list[str]:
    """Names of the functions include/tango.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Loads (building in-tree first if needed) the C-ABI library."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if build_if_missing:
            _build.build()
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"CUDA library {_build.LIB} is missing; build it with "
                               "`python -m cross_token_gated_gb300.build` (needs nvcc)")
        lib = ctypes.CDLL(_build.LIB)
        vp, sz = ctypes.c_void_p, ctypes.c_size_t
        P = ctypes.POINTER
        for name in ("tango_aggregate", "wango_aggregate"):
            f = getattr(lib, name)
            f.argtypes = [P(tg_agg_params), vp, vp, vp, vp, vp, vp, sz, vp]
            f.restype = ctypes.c_int
        for name in ("tango_aggregate_backward", "wango_aggregate_backward"):
            f = getattr(lib, name)
            f.argtypes = [P(tg_agg_params), vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
            f.restype = ctypes.c_int
        for name in ("tango_aggregate_save", "wango_aggregate_save"):
            f = getattr(lib, name)
            f.argtypes = [P(tg_agg_params), vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
            f.restype = ctypes.c_int
        lib.tango_aggregate_noalloc.argtypes = [P(tg_agg_params), vp, vp, vp, vp, vp, vp]
        lib.tango_aggregate_noalloc.restype = ctypes.c_int
        lib.tango_block_forward.argtypes = [P(tg_block_params), P(tg_block_weights), vp, vp, vp, sz, vp]
        lib.tango_block_forward.restype = ctypes.c_int
        lib.wango_decode_step.argtypes = [P(tg_agg_params), ctypes.c_longlong, vp, vp, vp, vp, vp, vp, sz, vp]
        lib.wango_decode_step.restype = ctypes.c_int
        lib.tango_model_forward.argtypes = [P(tg_model_params), P(tg_model_weights), vp, vp, vp, sz, vp]
        lib.tango_model_forward.restype = ctypes.c_int
        lib.tg_workspace_size.argtypes = [ctypes.c_int, vp]
        lib.tg_workspace_size.restype = sz
        lib.tg_status_string.argtypes = [ctypes.c_int]
        lib.tg_status_string.restype = ctypes.c_char_p
        lib.tg_check_device_error.argtypes = [vp, P(ctypes.c_uint)]
        lib.tg_check_device_error.restype = ctypes.c_int
        lib.tg_version.argtypes = []
        lib.tg_version.restype = ctypes.c_int
        _lib = lib
        return lib


# ------------------------------------------------------------------ marshalling

def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return TG_F32
    if t.dtype == torch.bfloat16:
        return TG_BF16
    raise TypeError(f"unsupported storage dtype {t.dtype} (float32 or bfloat16)")


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def agg_params(B, T, H, d_qk, m, *, dtype, s=10.0, tau=None, null_bias=None, window=1, phi_mode=0,
               flags=0, m_pitch=0) -> tg_agg_params:
    return tg_agg_params(B, T, H, d_qk, m, float(s), _ptr(tau), _ptr(null_bias), int(window),
                         int(phi_mode), int(flags), int(dtype), int(m_pitch))


def _gate_width(g, H, m_h):
    """(m, m_pitch) for a gate tensor of last dimension H * pitch: the logical total width
    H * m_h and the per-head pitch (0 when dense)."""
    width = g.shape[-1]
    if m_h is None:
        return width, 0
    if width % H != 0:
        raise ValueError("gate tensor width must be H * m_pitch")
    return H * int(m_h), width // H


def status_string(status: int) -> str:
    return load().tg_status_string(int(status)).decode()


tg_status_string = status_string


def tg_workspace_size(which: int, params) -> int:
    return int(load().tg_workspace_size(int(which), ctypes.byref(params)))


def tg_check_device_error(stream=None):
    """(status, raw word) after synchronising the stream."""
    word = ctypes.c_uint(0)
    st = load().tg_check_device_error(_stream(stream), ctypes.byref(word))
    return st, word.value


def tg_version() -> int:
    return int(load().tg_version())


def _workspace(nbytes: int, device, ws):
    if nbytes == 0:
        return None
    if ws is not None:
        return ws
    return torch.empty(nbytes + 256, dtype=torch.uint8, device=device)


def _ws_ptr(ws):
    if ws is None:
        return None, 0
    p = ws.data_ptr()
    aligned = (p + 255) & ~255
    return aligned, ws.numel() - (aligned - p)


def _aggregate(fn_name, q, k, g, v, out, *, H, s, tau, null_bias, window, phi_mode, flags, ws, stream, m_h=None,
               saved=None):
    B, T, d_qk = q.shape
    m, pitch = _gate_width(g, H, m_h)
    p = agg_params(B, T, H, d_qk, m, dtype=_dtype_code(g), s=s, tau=tau, null_bias=null_bias,
                   window=window, phi_mode=phi_mode, flags=flags, m_pitch=pitch)
    which = TG_WS_TANGO if fn_name.startswith("tango") else TG_WS_WANGO
    need = load().tg_workspace_size(which, ctypes.byref(p))
    wbuf = _workspace(need, g.device, ws)
    wp, wn = _ws_ptr(wbuf)
    extra = () if saved is None else (_ptr(saved[0]), _ptr(saved[1]))
    st = getattr(load(), fn_name)(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(g), _ptr(v), _ptr(out), *extra, wp, wn,
                                  _stream(stream))
    if st != TG_OK:
        raise TgError(st, fn_name)
    return out


def tango_aggregate(q, k, g, v, out, *, H, s=10.0, tau=None, null_bias=None, flags=0, ws=None,
                    stream=None, m_h=None):
    """Full-prefix aggregation (eqs. 5-6).  q, k [B, T, d_qk]; g, v, out [B, T, m] on the
    device, one storage dtype.  v may be None (then out = gbar).  With m_h given, the gate
    tensors are [B, T, H * pitch] and each head's m_h gates sit at a pitch of
    g.shape[-1] / H columns (m_pitch in tango.h)."""
    return _aggregate("tango_aggregate", q, k, g, v, out, H=H, s=s, tau=tau, null_bias=null_bias,
                      window=1, phi_mode=0, flags=flags, ws=ws, stream=stream, m_h=m_h)


def wango_aggregate(q, k, g, v, out, *, H, window, s=10.0, tau=None, null_bias=None, phi_mode=0,
                    flags=0, ws=None, stream=None, m_h=None):
    """Windowed aggregation (eqs. 7-10); arguments as for tango_aggregate."""
    return _aggregate("wango_aggregate", q, k, g, v, out, H=H, s=s, tau=tau, null_bias=null_bias,
                      window=window, phi_mode=phi_mode, flags=flags, ws=ws, stream=stream, m_h=m_h)


def tango_aggregate_save(q, k, g, v, out, gbar, den, *, H, s=10.0, tau=None, null_bias=None, flags=0, ws=None,
                         stream=None, m_h=None):
    """tango_aggregate that also writes gbar (laid out as out) and den (float32 [B, H, T])
    for the backward (bf16)."""
    return _aggregate("tango_aggregate_save", q, k, g, v, out, H=H, s=s, tau=tau, null_bias=null_bias, window=1,
                      phi_mode=0, flags=flags, ws=ws, stream=stream, m_h=m_h, saved=(gbar, den))


def wango_aggregate_save(q, k, g, v, out, gbar, den, *, H, window, s=10.0, tau=None, null_bias=None, phi_mode=0,
                         flags=0, ws=None, stream=None, m_h=None):
    """wango_aggregate that also writes gbar and den for the backward (bf16)."""
    return _aggregate("wango_aggregate_save", q, k, g, v, out, H=H, s=s, tau=tau, null_bias=null_bias,
                      window=window, phi_mode=phi_mode, flags=flags, ws=ws, stream=stream, m_h=m_h,
                      saved=(gbar, den))


def _aggregate_backward(fn_name, q, k, g, v, dout, dq, dk, dg, dv, *, H, s, tau, null_bias, window, phi_mode,
                        flags, ws, stream, m_h=None, gbar=None, den=None):
    B, T, d_qk = q.shape
    m, pitch = _gate_width(g, H, m_h)
    p = agg_params(B, T, H, d_qk, m, dtype=_dtype_code(g), s=s, tau=tau, null_bias=null_bias,
                   window=window, phi_mode=phi_mode, flags=flags, m_pitch=pitch)
    which = TG_WS_TANGO_BWD if fn_name == "tango_aggregate_backward" else TG_WS_WANGO_BWD
    need = load().tg_workspace_size(which, ctypes.byref(p))
    wbuf = _workspace(need, g.device, ws)
    wp, wn = _ws_ptr(wbuf)
    st = getattr(load(), fn_name)(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(g), _ptr(v), _ptr(dout), _ptr(gbar),
                                  _ptr(den), _ptr(dq), _ptr(dk), _ptr(dg), _ptr(dv), wp, wn, _stream(stream))
    if st != TG_OK:
        raise TgError(st, fn_name)
    return dq, dk, dg, dv


def tango_aggregate_backward(q, k, g, v, dout, dq, dk, dg, dv, *, H, s=10.0, tau=None, null_bias=None, flags=0,
                             ws=None, stream=None, m_h=None, gbar=None, den=None):
    """Gradients of sum(dout * tango_aggregate(q, k, g, v)) with respect to q, k, g, v
    (bf16).  dq, dk [B, T, d_qk] and dg, dv [B, T, m] are written; v and dv may be None."""
    return _aggregate_backward("tango_aggregate_backward", q, k, g, v, dout, dq, dk, dg, dv, H=H, s=s, tau=tau,
                               null_bias=null_bias, window=1, phi_mode=0, flags=flags, ws=ws, stream=stream,
                               m_h=m_h, gbar=gbar, den=den)


def wango_aggregate_backward(q, k, g, v, dout, dq, dk, dg, dv, *, H, window, s=10.0, tau=None, null_bias=None,
                             phi_mode=0, flags=0, ws=None, stream=None, m_h=None, gbar=None, den=None):
    """Gradients of sum(dout * wango_aggregate(q, k, g, v)); arguments as for
    tango_aggregate_backward."""
    return _aggregate_backward("wango_aggregate_backward", q, k, g, v, dout, dq, dk, dg, dv, H=H, s=s, tau=tau,
                               null_bias=null_bias, window=window, phi_mode=phi_mode, flags=flags, ws=ws,
                               stream=stream, m_h=m_h, gbar=gbar, den=den)


def tango_aggregate_noalloc(q, k, g, v, out, *, H, s=10.0, tau=None, null_bias=None, flags=0,
                            stream=None):
    """tango_aggregate without a workspace: the library's fixed device scratch array is
    used instead (for callers that cannot allocate device memory).  Raises TgError with
    TG_ERR_WORKSPACE when the problem needs more scratch than TG_NOALLOC_SCRATCH_BYTES."""
    B, T, d_qk = q.shape
    m = g.shape[-1]
    p = agg_params(B, T, H, d_qk, m, dtype=_dtype_code(g), s=s, tau=tau, null_bias=null_bias, flags=flags)
    st = load().tango_aggregate_noalloc(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(g), _ptr(v), _ptr(out),
                                        _stream(stream))
    if st != TG_OK:
        raise TgError(st, "tango_aggregate_noalloc")
    return out


TG_NOALLOC_SCRATCH_BYTES = 16 << 20


def block_params(B, T, d, H, d_qk, m, *, dtype, mode=TG_MODE_TANGO, s=10.0, tau=None, null_bias=None,
                 window=1, phi_mode=0, rms_eps=1e-6, rope_base=10000.0, flags=0) -> tg_block_params:
    return tg_block_params(agg_params(B, T, H, d_qk, m, dtype=dtype, s=s, tau=tau, null_bias=null_bias,
                                      window=window, phi_mode=phi_mode, flags=flags), int(d), int(mode),
                           float(rms_eps), float(rope_base))


def tango_block_forward(h, weights, h_out, *, H, mode=TG_MODE_TANGO, s=10.0, tau=None, null_bias=None,
                        window=1, phi_mode=0, rms_eps=1e-6, rope_base=10000.0, flags=0, ws=None, stream=None):
    """One block application (eqs. 2-10).  h, h_out [B, T, d]; weights: dict with gamma,
    Wq, Wk, Wg, Wv, Wo device tensors of h's dtype.  h_out may be h.  flags: 0,
    TG_FLAG_DEBUG_TIMEOUT (the projection GEMM's test hook) and/or TG_FLAG_FUSED_V
    (WANGO: v formed inside the aggregation instead of by the projection GEMM)."""
    B, T, d = h.shape
    d_qk, m = weights["Wq"].shape[0], weights["Wg"].shape[0]
    p = block_params(B, T, d, H, d_qk, m, dtype=_dtype_code(h), mode=mode, s=s, tau=tau,
                     null_bias=null_bias, window=window, phi_mode=phi_mode, rms_eps=rms_eps,
                     rope_base=rope_base, flags=flags)
    w = tg_block_weights(*[_ptr(weights[n]) for n in ("gamma", "Wq", "Wk", "Wg", "Wv", "Wo")])
    need = load().tg_workspace_size(TG_WS_BLOCK, ctypes.byref(p))
    wbuf = _workspace(need, h.device, ws)
    wp, wn = _ws_ptr(wbuf)
    st = load().tango_block_forward(ctypes.byref(p), ctypes.byref(w), _ptr(h), _ptr(h_out), wp, wn,
                                    _stream(stream))
    if st != TG_OK:
        raise TgError(st, "tango_block_forward")
    return h_out


def block_workspace(B, T, d, H, d_qk, m, *, dtype, mode=TG_MODE_TANGO, window=1, device="cuda"):
    """Allocates a workspace tensor large enough for tango_block_forward."""
    p = block_params(B, T, d, H, d_qk, m, dtype=dtype, mode=mode, window=window)
    return _workspace(tg_workspace_size(TG_WS_BLOCK, p), device, None)


def model_params(B, T, d, H, d_qk, m, vocab, *, dtype, n_apps=4, n_sets=1, set_of_app=None,
                 mode=TG_MODE_TANGO, s=10.0, tau=None, null_bias=None, window=1, phi_mode=0, rms_eps=1e-6,
                 rope_base=10000.0, final_rms_eps=1e-6):
    """tg_model_params; the returned structure keeps its set_of_app array alive."""
    table = None
    if set_of_app is not None:
        table = (ctypes.c_int * len(set_of_app))(*[int(x) for x in set_of_app])
    p = tg_model_params(block_params(B, T, d, H, d_qk, m, dtype=dtype, mode=mode, s=s, tau=tau,
                                     null_bias=null_bias, window=window, phi_mode=phi_mode, rms_eps=rms_eps,
                                     rope_base=rope_base),
                        int(vocab), int(n_apps), int(n_sets),
                        ctypes.cast(table, ctypes.POINTER(ctypes.c_int)) if table is not None else None,
                        float(final_rms_eps))
    p._table = table
    return p


def tango_model_forward(ids, embedding, final_gamma, sets, logits, *, H, n_apps=4, set_of_app=None,
                        mode=TG_MODE_TANGO, s=10.0, tau=None, null_bias=None, window=1, phi_mode=0,
                        rms_eps=1e-6, rope_base=10000.0, final_rms_eps=1e-6, ws=None, stream=None):
    """The shared-block language model (sec. 2.3): embedding, n_apps block applications,
    final RMSNorm, tied logits.  ids: device int32 [B, T]; embedding [vocab, d];
    final_gamma [d]; sets: list of weight dicts (gamma, Wq, Wk, Wg, Wv, Wo) of one gate
    width; logits [B, T, vocab], written."""
    if ids.dtype != torch.int32:
        raise TypeError("ids must be an int32 tensor")
    B, T = ids.shape
    vocab, d = embedding.shape
    d_qk, m = sets[0]["Wq"].shape[0], sets[0]["Wg"].shape[0]
    p = model_params(B, T, d, H, d_qk, m, vocab, dtype=_dtype_code(embedding), n_apps=n_apps,
                     n_sets=len(sets), set_of_app=set_of_app, mode=mode, s=s, tau=tau, null_bias=null_bias,
                     window=window, phi_mode=phi_mode, rms_eps=rms_eps, rope_base=rope_base,
                     final_rms_eps=final_rms_eps)
    arr = (tg_block_weights * len(sets))(
        *[tg_block_weights(*[_ptr(w[n]) for n in ("gamma", "Wq", "Wk", "Wg", "Wv", "Wo")]) for w in sets])
    w = tg_model_weights(_ptr(embedding), _ptr(final_gamma), ctypes.cast(arr, ctypes.POINTER(tg_block_weights)))
    need = load().tg_workspace_size(TG_WS_MODEL, ctypes.byref(p))
    wbuf = _workspace(need, ids.device, ws)
    wp, wn = _ws_ptr(wbuf)
    st = load().tango_model_forward(ctypes.byref(p), ctypes.byref(w), _ptr(ids), _ptr(logits), wp, wn,
                                    _stream(stream))
    if st != TG_OK:
        raise TgError(st, "tango_model_forward")
    return logits


def decode_state(B, H, d_qk, m, *, window, dtype, device="cuda"):
    """Allocates a state buffer for wango_decode_step (cleared by the step at pos 0)."""
    p = agg_params(B, 1, H, d_qk, m, dtype=dtype, window=window)
    return _workspace(tg_workspace_size(TG_WS_DECODE, p), device, None)


def wango_decode_step(q, k, g, v, out, state, pos, *, H, window, s=10.0, tau=None, null_bias=None,
                      phi_mode=0, flags=0, stream=None):
    """One autoregressive WANGO step for B sequences at position pos.  q, k [B, d_qk];
    g, v, out [B, m]; state from decode_state(), kept between steps (pos = 0, 1, ...)."""
    B, d_qk = q.shape
    m = g.shape[-1]
    p = agg_params(B, 1, H, d_qk, m, dtype=_dtype_code(g), s=s, tau=tau, null_bias=null_bias, window=window,
                   phi_mode=phi_mode, flags=flags)
    wp, wn = _ws_ptr(state)
    st = load().wango_decode_step(ctypes.byref(p), int(pos), _ptr(q), _ptr(k), _ptr(g), _ptr(v), _ptr(out),
                                  wp, wn, _stream(stream))
    if st != TG_OK:
        raise TgError(st, "wango_decode_step")
    return out
