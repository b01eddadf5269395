"""Host-side checks of the C-ABI library: it loads without a GPU, exports every
function include/tango.h declares, and rejects bad arguments before launching."""
import ctypes

import pytest

import cross_token_gated_gb300 as tg


def test_exports_every_declared_function(lib):
    names = tg.declared_functions()
    assert {"tango_aggregate", "wango_aggregate", "tango_block_forward", "tg_workspace_size",
            "tg_status_string", "tg_check_device_error", "tg_version"} <= set(names)
    raw = tg.load()
    for n in names:
        assert hasattr(raw, n), f"library does not export {n}"


def test_exports_no_undeclared_c_function(lib):
    """The C ABI is exactly the header: every exported function with C linkage (an
    unmangled name) is declared in include/tango.h; internal helpers stay internal."""
    import shutil
    import subprocess

    from cross_token_gated_gb300 import build
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm is not installed")
    out = subprocess.run([nm, "-D", "--defined-only", build.LIB], capture_output=True, text=True, check=True).stdout
    c_funcs = {parts[2] for parts in (line.split() for line in out.splitlines())
               if len(parts) == 3 and parts[1] == "T" and not parts[2].startswith("_Z")}
    assert c_funcs == set(tg.declared_functions())


def test_status_strings(lib):
    for st in range(7):
        assert tg.status_string(st)
    assert tg.status_string(99) == "unknown status"
    assert tg.tg_version() >= 100


def _agg(**kw):
    base = dict(B=2, T=64, H=2, d_qk=128, m=256, dtype=tg.TG_BF16, s=10.0, window=16)
    base.update(kw)
    B, T, H, d_qk, m = (base.pop(x) for x in ("B", "T", "H", "d_qk", "m"))
    return tg.agg_params(B, T, H, d_qk, m, **base)


def test_workspace_sizes(lib):
    p = _agg()
    # two normalised copies of q and k, each 256-byte aligned
    assert tg.tg_workspace_size(tg.TG_WS_TANGO, p) == 2 * 2 * 64 * 128 * 2
    p = _agg(flags=tg.TG_FLAG_QK_NORMALIZED)
    assert tg.tg_workspace_size(tg.TG_WS_TANGO, p) == 0
    bp = tg.block_params(8, 2048, 512, 2, 128, 28480, dtype=tg.TG_BF16)
    need = tg.tg_workspace_size(tg.TG_WS_BLOCK, bp)
    BT = 8 * 2048
    assert need == BT * 2 * (512 + 2 * 128 + 2 * 28480)
    assert tg.tg_workspace_size(tg.TG_WS_TANGO, _agg(H=3)) == 0        # invalid -> 0
    assert tg.tg_workspace_size(7, p) == 0


@pytest.mark.parametrize("kw,status", [
    (dict(B=0), tg.TG_ERR_INVALID_ARG),
    (dict(T=0), tg.TG_ERR_INVALID_ARG),
    (dict(H=3), tg.TG_ERR_INVALID_ARG),             # d_qk % H != 0
    (dict(m=255), tg.TG_ERR_INVALID_ARG),           # m % H != 0
    (dict(s=25.0), tg.TG_ERR_INVALID_ARG),          # tau cap of eq. 4
    (dict(s=-1.0), tg.TG_ERR_INVALID_ARG),
    (dict(window=0), tg.TG_ERR_INVALID_ARG),
    (dict(phi_mode=2), tg.TG_ERR_INVALID_ARG),
    (dict(flags=0x80), tg.TG_ERR_INVALID_ARG),
    (dict(dtype=5), tg.TG_ERR_INVALID_ARG),
    (dict(d_qk=96, H=2), tg.TG_ERR_UNSUPPORTED),    # bf16 head width 48
    (dict(m=2 * 4747), tg.TG_ERR_UNSUPPORTED),      # bf16 head gate width not a multiple of 8
])
def test_invalid_arguments_rejected_on_host(lib, kw, status):
    p = _agg(**kw)
    raw = tg.load()
    dummy = 256  # never dereferenced: validation fails first
    st = raw.wango_aggregate(ctypes.byref(p), dummy, dummy, dummy, dummy, dummy, None, 0, None)
    assert st == status


def test_null_pointers_and_workspace(lib):
    raw = tg.load()
    p = _agg()
    assert raw.tango_aggregate(None, 256, 256, 256, 256, 256, None, 0, None) == tg.TG_ERR_INVALID_ARG
    assert raw.tango_aggregate(ctypes.byref(p), None, 256, 256, 256, 256, None, 0, None) == \
        tg.TG_ERR_INVALID_ARG
    # misaligned bf16 tensor
    assert raw.tango_aggregate(ctypes.byref(p), 258, 256, 256, 256, 256, None, 0, None) == \
        tg.TG_ERR_UNSUPPORTED
    # workspace required but missing / too small / misaligned
    need = tg.tg_workspace_size(tg.TG_WS_TANGO, p)
    assert raw.tango_aggregate(ctypes.byref(p), 256, 256, 256, 256, 256, None, 0, None) == tg.TG_ERR_WORKSPACE
    assert raw.tango_aggregate(ctypes.byref(p), 256, 256, 256, 256, 256, 4096, need - 1, None) == \
        tg.TG_ERR_WORKSPACE
    assert raw.tango_aggregate(ctypes.byref(p), 256, 256, 256, 256, 256, 4096 + 16, need, None) == \
        tg.TG_ERR_WORKSPACE


def test_block_validation(lib):
    raw = tg.load()
    w = tg.tg_block_weights(*([256] * 6))
    bp = tg.block_params(1, 8, 64, 2, 32, 256, dtype=tg.TG_BF16, rms_eps=0.0)
    assert raw.tango_block_forward(ctypes.byref(bp), ctypes.byref(w), 256, 256, None, 0, None) == \
        tg.TG_ERR_INVALID_ARG
    bp = tg.block_params(1, 8, 64, 2, 32, 256, dtype=tg.TG_BF16, mode=5)
    assert raw.tango_block_forward(ctypes.byref(bp), ctypes.byref(w), 256, 256, None, 0, None) == \
        tg.TG_ERR_INVALID_ARG
    bp = tg.block_params(1, 8, 60, 2, 32, 256, dtype=tg.TG_BF16)   # bf16 needs d % 64 == 0
    assert raw.tango_block_forward(ctypes.byref(bp), ctypes.byref(w), 256, 256, None, 0, None) == \
        tg.TG_ERR_UNSUPPORTED
    bp = tg.block_params(1, 8, 64, 2, 32, 256, dtype=tg.TG_BF16)
    w0 = tg.tg_block_weights(256, 256, None, 256, 256, 256)
    assert raw.tango_block_forward(ctypes.byref(bp), ctypes.byref(w0), 256, 256, None, 0, None) == \
        tg.TG_ERR_INVALID_ARG
    assert raw.tango_block_forward(ctypes.byref(bp), ctypes.byref(w), 256, 256, None, 0, None) == \
        tg.TG_ERR_WORKSPACE


def test_block_pads_unaligned_head_gate_width(lib):
    """The block accepts a bf16 head gate width that is not a multiple of 8 (the
    three-set width 9,494 = 2 x 4,747): its g and u use a pitch of 4,752 per head and the
    padded W_g, W_v, W_o copies sit at the end of the workspace."""
    B, T, d, dqk, H = 2, 64, 512, 128, 2
    BT = B * T
    bp = tg.block_params(B, T, d, H, dqk, 2 * 4747, dtype=tg.TG_BF16)
    mp = 2 * 4752
    def a256(x):
        return (x + 255) // 256 * 256
    want = a256(BT * d * 2) + 2 * a256(BT * dqk * 2) + 2 * a256(BT * mp * 2) + 3 * a256(mp * d * 2)
    assert tg.tg_workspace_size(tg.TG_WS_BLOCK, bp) == want
    # fp32 runs on the CUDA cores at the caller's width: no padding, no copies
    bp = tg.block_params(B, T, d, H, dqk, 2 * 4747, dtype=tg.TG_F32)
    assert tg.tg_workspace_size(tg.TG_WS_BLOCK, bp) == \
        a256(BT * d * 4) + 2 * a256(BT * dqk * 4) + 2 * a256(BT * 2 * 4747 * 4)


def test_block_qk_width_rule(lib):
    """bf16 blocks take q and k in one 256-column projection tile (d_qk <= 128) or in
    256-column tiles (d_qk a multiple of 256, e.g. the paper's 16 heads of 32)."""
    for dqk, H, ok in ((128, 2, True), (512, 16, True), (256, 8, True), (384, 12, False)):
        bp = tg.block_params(2, 64, 512, H, dqk, 256 * H, dtype=tg.TG_BF16)
        assert (tg.tg_workspace_size(tg.TG_WS_BLOCK, bp) > 0) == ok, dqk


def _model(**kw):
    base = dict(B=2, T=64, d=512, H=2, d_qk=128, m=256, vocab=1000, dtype=tg.TG_BF16)
    base.update(kw)
    args = [base.pop(x) for x in ("B", "T", "d", "H", "d_qk", "m", "vocab")]
    return tg.model_params(*args, **base)


def test_model_workspace_and_validation(lib):
    raw = tg.load()
    p = _model()
    bp = tg.block_params(2, 64, 512, 2, 128, 256, dtype=tg.TG_BF16)
    hb = 2 * 64 * 512 * 2
    assert tg.tg_workspace_size(tg.TG_WS_MODEL, p) == 2 * hb + tg.tg_workspace_size(tg.TG_WS_BLOCK, bp)
    for bad, status in [(dict(vocab=0), tg.TG_ERR_INVALID_ARG),
                        (dict(n_apps=0), tg.TG_ERR_INVALID_ARG),
                        (dict(n_apps=65), tg.TG_ERR_INVALID_ARG),
                        (dict(n_sets=2), tg.TG_ERR_INVALID_ARG),          # no default for two sets
                        (dict(n_sets=3, set_of_app=[0, 1, 3, 2]), tg.TG_ERR_INVALID_ARG),
                        (dict(final_rms_eps=0.0), tg.TG_ERR_INVALID_ARG),
                        (dict(vocab=1001), tg.TG_ERR_UNSUPPORTED),        # bf16 logits pitch
                        (dict(d=60), tg.TG_ERR_UNSUPPORTED)]:
        q = _model(**bad)
        assert tg.tg_workspace_size(tg.TG_WS_MODEL, q) == 0
        sets = (tg.tg_block_weights * 1)(tg.tg_block_weights(*([256] * 6)))
        w = tg.tg_model_weights(256, 256, ctypes.cast(sets, ctypes.POINTER(tg.tg_block_weights)))
        assert raw.tango_model_forward(ctypes.byref(q), ctypes.byref(w), 256, 256, None, 0, None) == status
    assert tg.tg_workspace_size(tg.TG_WS_MODEL, _model(n_sets=2, set_of_app=[0, 1, 1, 0])) > 0
    assert tg.tg_workspace_size(tg.TG_WS_MODEL, _model(vocab=1001, dtype=tg.TG_F32)) > 0
    sets = (tg.tg_block_weights * 1)(tg.tg_block_weights(*([256] * 6)))
    w = tg.tg_model_weights(256, None, ctypes.cast(sets, ctypes.POINTER(tg.tg_block_weights)))
    assert raw.tango_model_forward(ctypes.byref(p), ctypes.byref(w), 256, 256, None, 0, None) == \
        tg.TG_ERR_INVALID_ARG
    w = tg.tg_model_weights(256, 256, ctypes.cast(sets, ctypes.POINTER(tg.tg_block_weights)))
    assert raw.tango_model_forward(ctypes.byref(p), ctypes.byref(w), 256, 256, None, 0, None) == \
        tg.TG_ERR_WORKSPACE


def test_binding_has_no_fallback(monkeypatch, tmp_path):
    """Without the library the binding raises instead of computing anything itself."""
    monkeypatch.setattr(tg, "_lib", None)
    monkeypatch.setattr(tg._build, "LIB", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        tg.load(build_if_missing=False)
    monkeypatch.undo()


def test_decode_state_size_and_validation(lib):
    """The decode state: S [B, d_h, m] and z (two buffers, by step parity) in f32, the
    ring of R = W + 8 unit keys and gates (storage type: the window plus the sources that
    left it and wait to be folded into S in a group of 8), and per-step scratch (ring
    weights, q's feature map, the group's key feature maps, 8 partial sums and the
    older-prefix term per head), each region 256-byte aligned."""
    raw = tg.load()
    B, H, dqk, m, W = 2, 2, 128, 512, 16
    R = W + 8
    p = tg.agg_params(B, 1, H, dqk, m, dtype=tg.TG_BF16, window=W)
    def a256(x):
        return (x + 255) // 256 * 256
    d_h = dqk // H
    want = (a256(B * d_h * m * 4) + a256(2 * B * H * d_h * 4) + a256(B * H * R * d_h * 2) + a256(B * R * m * 2)
            + a256(B * H * R * 4) + a256(B * H * d_h * 4) + a256(B * H * 8 * d_h * 4) + a256(B * H * 8 * 4)
            + a256(B * H * 4))
    assert tg.tg_workspace_size(tg.TG_WS_DECODE, p) == want
    for bad in (dict(window=0), dict(phi_mode=3), dict(flags=tg.TG_FLAG_DEBUG_TIMEOUT)):
        q = tg.agg_params(B, 1, H, dqk, m, dtype=tg.TG_BF16, **dict(dict(window=W), **bad))
        assert tg.tg_workspace_size(tg.TG_WS_DECODE, q) == 0
        assert raw.wango_decode_step(ctypes.byref(q), 0, 256, 256, 256, None, 256, None, 0, None) == \
            tg.TG_ERR_INVALID_ARG
    assert raw.wango_decode_step(ctypes.byref(p), -1, 256, 256, 256, None, 256, None, 0, None) == \
        tg.TG_ERR_INVALID_ARG
    assert raw.wango_decode_step(ctypes.byref(p), 0, 256, 256, 256, None, 256, None, 0, None) == \
        tg.TG_ERR_WORKSPACE


def test_backward_validation_and_workspace(lib):
    """The backward entry points validate on the host: bf16 only, only the unit-input
    flag, v needed for dv, aligned pointers, a workspace that holds the recomputed
    forward, E and the bf16 pair gradients of B * H * T_pad^2 entries."""
    raw = tg.load()
    p = _agg(B=2, T=300, H=2, d_qk=128, m=512)
    for which in (tg.TG_WS_TANGO_BWD, tg.TG_WS_WANGO_BWD):
        need = tg.tg_workspace_size(which, p)
        assert need >= 2 * 2 * 384 * 384 * 2 + 2 * 300 * 512 * 2 * 2
    assert tg.tg_workspace_size(tg.TG_WS_WANGO_BWD, p) > tg.tg_workspace_size(tg.TG_WS_TANGO_BWD, p)
    assert tg.tg_workspace_size(tg.TG_WS_TANGO_BWD, _agg(dtype=tg.TG_F32)) == 0
    a = [256] * 5 + [None, None] + [256] * 4   # q k g v dout, no saved gbar/den, dq dk dg dv
    for fn in (raw.tango_aggregate_backward, raw.wango_aggregate_backward):
        assert fn(ctypes.byref(_agg(dtype=tg.TG_F32)), *a, None, 0, None) == tg.TG_ERR_UNSUPPORTED
        # the test hook passes validation (it arms the backward's own kernels); the call then
        # stops at the missing workspace, before any launch
        assert fn(ctypes.byref(_agg(flags=tg.TG_FLAG_DEBUG_TIMEOUT)), *a, None, 0, None) == tg.TG_ERR_WORKSPACE
        assert fn(ctypes.byref(_agg(B=0)), *a, None, 0, None) == tg.TG_ERR_INVALID_ARG
        # dv without v
        assert fn(ctypes.byref(p), 256, 256, 256, None, 256, None, None, 256, 256, 256, 256, None, 0, None) == \
            tg.TG_ERR_INVALID_ARG
        # misaligned dout
        assert fn(ctypes.byref(p), 256, 256, 256, 256, 264, None, None, 256, 256, 256, 256, None, 0, None) == \
            tg.TG_ERR_UNSUPPORTED
        # a saved gbar without its denominators
        assert fn(ctypes.byref(p), 256, 256, 256, 256, 256, 256, None, 256, 256, 256, 256, None, 0, None) == \
            tg.TG_ERR_INVALID_ARG
        assert fn(ctypes.byref(p), *a, None, 0, None) == tg.TG_ERR_WORKSPACE
    # the far-pair choice: WANGO only, not both at once
    both = tg.TG_FLAG_BWD_FAR_SCAN | tg.TG_FLAG_BWD_FAR_PAIRS
    assert raw.wango_aggregate_backward(ctypes.byref(_agg(flags=both)), *a, None, 0, None) == tg.TG_ERR_INVALID_ARG
    assert raw.tango_aggregate_backward(ctypes.byref(_agg(flags=tg.TG_FLAG_BWD_FAR_SCAN)), *a, None, 0, None) == \
        tg.TG_ERR_INVALID_ARG
    assert tg.tg_workspace_size(tg.TG_WS_WANGO_BWD, _agg(flags=both)) == 0
    for fn in (raw.tango_aggregate_save, raw.wango_aggregate_save):
        assert fn(ctypes.byref(p), 256, 256, 256, 256, 256, None, 256, None, 0, None) == tg.TG_ERR_INVALID_ARG
        assert fn(ctypes.byref(_agg(dtype=tg.TG_F32)), 256, 256, 256, 256, 256, 256, 256, None, 0, None) == \
            tg.TG_ERR_UNSUPPORTED
        assert fn(ctypes.byref(p), 256, 256, 256, 256, 256, 256, 256, None, 0, None) == tg.TG_ERR_WORKSPACE


def test_gate_pitch_validation(lib):
    """A per-head gate pitch: at least m_h, a multiple of 8 in bf16; it lets the
    revision's three-set width (m_h = 4,747) run in bf16; blocks and decode steps take
    none."""
    raw = tg.load()
    a = [256] * 5
    dense = _agg(m=2 * 4747)
    assert raw.tango_aggregate(ctypes.byref(dense), *a, None, 0, None) == tg.TG_ERR_UNSUPPORTED
    for fn in (raw.tango_aggregate, raw.wango_aggregate):
        ok = _agg(m=2 * 4747, m_pitch=4752)
        assert fn(ctypes.byref(ok), *a, None, 0, None) == tg.TG_ERR_WORKSPACE   # valid: only the workspace is missing
        assert fn(ctypes.byref(_agg(m=2 * 4747, m_pitch=4740)), *a, None, 0, None) == tg.TG_ERR_INVALID_ARG
        assert fn(ctypes.byref(_agg(m=2 * 4747, m_pitch=4750)), *a, None, 0, None) == tg.TG_ERR_UNSUPPORTED
        assert fn(ctypes.byref(_agg(m=2 * 4747, m_pitch=4750, dtype=tg.TG_F32)), *a, None, 0, None) == \
            tg.TG_ERR_WORKSPACE
    for which in (tg.TG_WS_TANGO_BWD, tg.TG_WS_WANGO_BWD):
        assert tg.tg_workspace_size(which, _agg(m=2 * 4747, m_pitch=4752)) > 0
    bp = tg.block_params(1, 64, 128, 2, 128, 512, dtype=tg.TG_BF16)
    bp.agg.m_pitch = 264
    assert tg.tg_workspace_size(tg.TG_WS_BLOCK, bp) == 0
    dp = _agg(m=512, m_pitch=264)
    assert tg.tg_workspace_size(tg.TG_WS_DECODE, dp) == 0


def test_backward_far_scan_workspace(lib):
    """WANGO's far older pairs through the scans need their per-strip sums, 2 directions x
    ceil(m_h / n_s) strips (n_s in 512, 384, 256) x B * T * d_qk floats, plus 3 x B * H * nblk * d_h floats of
    block sums; the pair path needs neither.  With no block beyond the window's band
    (T = 300, W = 200: 3 blocks, band 2) the two are the same."""
    kw = dict(B=2, T=1500, H=2, d_qk=128, m=4096, window=64)
    scan = tg.tg_workspace_size(tg.TG_WS_WANGO_BWD, _agg(flags=tg.TG_FLAG_BWD_FAR_SCAN, **kw))
    pairs = tg.tg_workspace_size(tg.TG_WS_WANGO_BWD, _agg(flags=tg.TG_FLAG_BWD_FAR_PAIRS, **kw))
    nblk = -(-1500 // 128)
    fits = [s for s in (-(-2048 // ns) for ns in (512, 384, 256))
            if 0 <= scan - pairs - (2 * s * 2 * 1500 * 128 * 4 + 3 * 2 * 2 * nblk * 64 * 4) <= 512]
    assert fits, scan - pairs
    # the library's own choice is one of the two
    auto = tg.tg_workspace_size(tg.TG_WS_WANGO_BWD, _agg(**kw))
    assert auto in (scan, pairs)
    kw = dict(B=2, T=300, H=2, d_qk=128, m=512, window=200)
    assert tg.tg_workspace_size(tg.TG_WS_WANGO_BWD, _agg(flags=tg.TG_FLAG_BWD_FAR_SCAN, **kw)) == \
        tg.tg_workspace_size(tg.TG_WS_WANGO_BWD, _agg(flags=tg.TG_FLAG_BWD_FAR_PAIRS, **kw))


def test_backward_far_path_choice(lib):
    """The library's own choice for WANGO's far older pairs (W = 256, the 70M-tier gate
    width): pair by pair where the band covers most of the sequence (B = 8, T = 2,048:
    42 far tiles per head against a scan chain of 13 steps on 6 waves), the running-sum
    scans at long context (T >= 4,096), which is linear in T.  Read from the workspace
    size, which carries the scans' per-strip sums only when they run."""
    def path(B, T):
        kw = dict(B=B, T=T, H=2, d_qk=128, m=28480, window=256)
        auto = tg.tg_workspace_size(tg.TG_WS_WANGO_BWD, _agg(**kw))
        scan = tg.tg_workspace_size(tg.TG_WS_WANGO_BWD, _agg(flags=tg.TG_FLAG_BWD_FAR_SCAN, **kw))
        pairs = tg.tg_workspace_size(tg.TG_WS_WANGO_BWD, _agg(flags=tg.TG_FLAG_BWD_FAR_PAIRS, **kw))
        assert scan > pairs
        return "scan" if auto == scan else "pairs" if auto == pairs else None
    assert path(8, 2048) == "pairs"
    assert path(1, 2048) == "pairs"
    for B, T in ((1, 4096), (8, 4096), (1, 8192), (1, 16384)):
        assert path(B, T) == "scan", (B, T)
    # a window that leaves no block beyond its band: both are the pair path
    kw = dict(B=1, T=512, H=2, d_qk=128, m=2048, window=512)
    assert tg.tg_workspace_size(tg.TG_WS_WANGO_BWD, _agg(flags=tg.TG_FLAG_BWD_FAR_SCAN, **kw)) == \
        tg.tg_workspace_size(tg.TG_WS_WANGO_BWD, _agg(**kw))
