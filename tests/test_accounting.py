"""Pins of the work accounting against the figures printed in "TANGO: Token-Aggregated
Nonlinear Gating Operators ..." (tests/golden/paper_figures.json, each with its citation)."""
import json
import os

import pytest

from cross_token_gated_gb300 import accounting as acc

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "paper_figures.json")))


def printed(x, digits):
    """Round to the number of significant digits the page prints."""
    from math import floor, log10
    return round(x, -int(floor(log10(abs(x)))) + digits - 1)


def test_block_params_table1():
    f = GOLD["block_params"]
    assert acc.paper_block_params(f["d"], f["F"], f["H"]) == f["value"]


def test_embedding_params():
    f = GOLD["embedding_params"]
    assert f["d"] * f["vocab"] == f["value"]


@pytest.mark.parametrize("key", ["macs_tango_T8192", "macs_tango_T256"])
def test_tango_macs_exact_to_printed_digits(key):
    f = GOLD[key]
    macs = acc.paper_macs_tango(f["T"], f["d"], f["F"], f["vocab"], f["R"])
    assert printed(macs, f["printed_digits"]) == pytest.approx(f["value"], rel=1e-12)


@pytest.mark.parametrize("key", ["macs_wango_T8192", "macs_wango_T256"])
def test_wango_macs_estimate_close(key):
    """The pages' WANGO accounting is not fully stated; the estimate lands within 0.2 %."""
    f = GOLD[key]
    est = acc.paper_macs_wango_estimate(f["T"], f["d"], f["F"], f["vocab"], f["W"], f["H"], f["R"])
    assert abs(est / f["value"] - 1) < 2e-3


def test_build_units_at_70m_shapes():
    # TANGO aggregation, B=8, T=2048, dqk=128, m=28480: causal pairs x (dqk + m) x 2
    assert acc.causal_pairs(2048) == 2_098_176
    assert acc.tango_agg_flops(8, 2048, 128, 28480) == 2 * 8 * 2_098_176 * 28608
    assert acc.agg_bytes(8, 2048, 128, 28480) == 16384 * (256 + 85440) * 2
    # window pairs reduce to causal pairs when W >= T
    assert acc.window_pairs(100, 100) == acc.causal_pairs(100)
    assert acc.window_pairs(100, 7) == sum(min(i + 1, 7) for i in range(100))
    # WANGO with W >= T has no older prefix: same flops as TANGO
    assert acc.wango_agg_flops(2, 64, 32, 256, 2, 64) == acc.tango_agg_flops(2, 64, 32, 256)
