"""tango_aggregate_noalloc: the aggregation entry point for callers that cannot
allocate device memory (runtimes that forbid cudaMalloc once running, code confined to
a pool it does not own).  It uses the library's fixed device scratch array instead of
a caller workspace; its results must equal tango_aggregate's on the same inputs.

This file is collected last on purpose, so that a run stopping at the first failure
has already run every other test.  It passes alone in a fresh process and after the
other tests.
"""
import ctypes

import pytest
import torch

import cross_token_gated_gb300 as tg
from cross_token_gated_gb300 import synth

def rel(a, b):
    a, b = a.double().cpu(), b.double().cpu()
    return float((a - b).abs().max() / b.abs().max().clamp_min(1e-30))


def test_noalloc_rejects_oversized_problem_on_host(lib):
    """Needing more scratch than the fixed array holds is refused before any launch."""
    p = tg.agg_params(8, 8192, 2, 128, 1024, dtype=tg.TG_BF16)   # 2 x 16 MiB of q/k copies
    assert tg.tg_workspace_size(tg.TG_WS_TANGO, p) > tg.TG_NOALLOC_SCRATCH_BYTES
    st = tg.load().tango_aggregate_noalloc(ctypes.byref(p), 256, 256, 256, 256, 256, None)
    assert st == tg.TG_ERR_WORKSPACE
    assert tg.load().tango_aggregate_noalloc(None, 256, 256, 256, 256, 256, None) == tg.TG_ERR_INVALID_ARG


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_noalloc_matches_tango_aggregate_twice(dtype):
    """Two calls in a row on different inputs, the second smaller than the first so that
    a stale part of the scratch left by the first would show: each equals
    tango_aggregate's output bit for bit (the same kernels run on the same inputs, and
    their summation order does not depend on where the scratch lives)."""
    H = 2
    for call, (B, T, dqk, m, seed) in enumerate([(2, 300, 128, 1040, 21), (1, 700, 64, 512, 22)]):
        q, k, g, v = (t.cuda() for t in synth.agg_inputs(B, T, dqk, m, seed=seed, dtype=dtype))
        ref = torch.empty_like(g)
        tg.tango_aggregate(q, k, g, v, ref, H=H)
        got = torch.full_like(g, float("nan"))
        tg.tango_aggregate_noalloc(q, k, g, v, got, H=H)
        st, word = tg.tg_check_device_error()
        assert st == tg.TG_OK, (call, st, hex(word))
        assert torch.isfinite(got.float()).all(), call
        assert torch.equal(got, ref), (call, rel(got, ref))
