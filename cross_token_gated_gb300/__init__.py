"""GB300-native cross-token gate aggregation (TANGO / WANGO).

Python binding of the C-ABI library declared in ``include/tango.h``.  The binding
only marshals arguments: every step of the path runs in the library's CUDA
kernels.  PyTorch supplies device memory and streams.  There is no fallback: if
the library cannot be loaded, every call raises.

Functions (same names as the C ABI):
  tango_aggregate, tango_aggregate_noalloc, wango_aggregate, tango_block_forward,
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
TG_MODE_TANGO, TG_MODE_WANGO = 0, 1
TG_WS_TANGO, TG_WS_WANGO, TG_WS_BLOCK = 0, 1, 2

HEADER = os.path.join(_build.INCLUDE, "tango.h")


class TgError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} (status {status})")
        self.status = status


class tg_agg_params(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("H", ctypes.c_int), ("d_qk", ctypes.c_int),
                ("m", ctypes.c_int), ("s", ctypes.c_float), ("tau", ctypes.c_void_p),
                ("null_bias", ctypes.c_void_p), ("window", ctypes.c_int), ("phi_mode", ctypes.c_int),
                ("flags", ctypes.c_uint), ("dtype", ctypes.c_int)]


class tg_block_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("rms_gamma", "Wq", "Wk", "Wg", "Wv", "Wo")]


class tg_block_params(ctypes.Structure):
    _fields_ = [("agg", tg_agg_params), ("d", ctypes.c_int), ("mode", ctypes.c_int),
                ("rms_eps", ctypes.c_float), ("rope_base", ctypes.c_float)]


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
        lib.tango_aggregate_noalloc.argtypes = [P(tg_agg_params), vp, vp, vp, vp, vp, vp]
        lib.tango_aggregate_noalloc.restype = ctypes.c_int
        lib.tango_block_forward.argtypes = [P(tg_block_params), P(tg_block_weights), vp, vp, vp, sz, vp]
        lib.tango_block_forward.restype = ctypes.c_int
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
               flags=0) -> tg_agg_params:
    return tg_agg_params(B, T, H, d_qk, m, float(s), _ptr(tau), _ptr(null_bias), int(window),
                         int(phi_mode), int(flags), int(dtype))


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


def _aggregate(fn_name, q, k, g, v, out, *, H, s, tau, null_bias, window, phi_mode, flags, ws, stream):
    B, T, d_qk = q.shape
    m = g.shape[-1]
    p = agg_params(B, T, H, d_qk, m, dtype=_dtype_code(g), s=s, tau=tau, null_bias=null_bias,
                   window=window, phi_mode=phi_mode, flags=flags)
    which = TG_WS_TANGO if fn_name == "tango_aggregate" else TG_WS_WANGO
    need = load().tg_workspace_size(which, ctypes.byref(p))
    wbuf = _workspace(need, g.device, ws)
    wp, wn = _ws_ptr(wbuf)
    st = getattr(load(), fn_name)(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(g), _ptr(v), _ptr(out), wp, wn,
                                  _stream(stream))
    if st != TG_OK:
        raise TgError(st, fn_name)
    return out


def tango_aggregate(q, k, g, v, out, *, H, s=10.0, tau=None, null_bias=None, flags=0, ws=None,
                    stream=None):
    """Full-prefix aggregation (eqs. 5-6).  q, k [B, T, d_qk]; g, v, out [B, T, m] on the
    device, one storage dtype.  v may be None (then out = gbar)."""
    return _aggregate("tango_aggregate", q, k, g, v, out, H=H, s=s, tau=tau, null_bias=null_bias,
                      window=1, phi_mode=0, flags=flags, ws=ws, stream=stream)


def wango_aggregate(q, k, g, v, out, *, H, window, s=10.0, tau=None, null_bias=None, phi_mode=0,
                    flags=0, ws=None, stream=None):
    """Windowed aggregation (eqs. 7-10); arguments as for tango_aggregate."""
    return _aggregate("wango_aggregate", q, k, g, v, out, H=H, s=s, tau=tau, null_bias=null_bias,
                      window=window, phi_mode=phi_mode, flags=flags, ws=ws, stream=stream)


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
                 window=1, phi_mode=0, rms_eps=1e-6, rope_base=10000.0) -> tg_block_params:
    return tg_block_params(agg_params(B, T, H, d_qk, m, dtype=dtype, s=s, tau=tau, null_bias=null_bias,
                                      window=window, phi_mode=phi_mode), int(d), int(mode), float(rms_eps),
                           float(rope_base))


def tango_block_forward(h, weights, h_out, *, H, mode=TG_MODE_TANGO, s=10.0, tau=None, null_bias=None,
                        window=1, phi_mode=0, rms_eps=1e-6, rope_base=10000.0, ws=None, stream=None):
    """One block application (eqs. 2-10).  h, h_out [B, T, d]; weights: dict with gamma,
    Wq, Wk, Wg, Wv, Wo device tensors of h's dtype.  h_out may be h."""
    B, T, d = h.shape
    d_qk, m = weights["Wq"].shape[0], weights["Wg"].shape[0]
    p = block_params(B, T, d, H, d_qk, m, dtype=_dtype_code(h), mode=mode, s=s, tau=tau,
                     null_bias=null_bias, window=window, phi_mode=phi_mode, rms_eps=rms_eps,
                     rope_base=rope_base)
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
