"""The seeded input generators: the recipe both the CUDA path and the oracle rely on.

They must give the same values for the same seed, the stated shapes and scales, and bf16
rounded to nearest-even; the oracle view of a bf16 tensor must carry its exact bits."""
import numpy as np
import pytest
import torch

from cross_token_gated_gb300 import synth


def test_same_seed_same_values_other_seed_other_values():
    a = synth.agg_inputs(2, 5, 8, 16, seed=4)
    b = synth.agg_inputs(2, 5, 8, 16, seed=4)
    c = synth.agg_inputs(2, 5, 8, 16, seed=5)
    for x, y, z in zip(a, b, c):
        assert torch.equal(x, y)
        assert not torch.equal(x, z)


def test_shapes_dtypes_and_draw_order():
    q, k, g, v = synth.agg_inputs(2, 3, 8, 12, seed=1, dtype="f32")
    assert [t.shape for t in (q, k, g, v)] == [(2, 3, 8), (2, 3, 8), (2, 3, 12), (2, 3, 12)]
    assert all(t.dtype == torch.float32 for t in (q, k, g, v))
    # q, k, g, v are consecutive draws of one generator, in that order
    rng = np.random.default_rng(1)
    for t, n in ((q, 48), (k, 48), (g, 72), (v, 72)):
        ref = rng.standard_normal(size=n, dtype=np.float32)
        assert np.array_equal(t.numpy().ravel(), ref)


def test_block_weight_scales_follow_fan_in():
    d, dqk, m = 256, 128, 1024
    h, w = synth.block_inputs(4, 64, d, dqk, m, seed=2, dtype="f32")
    assert h.shape == (4, 64, d) and abs(float(h.std()) - 1.0) < 0.02
    for name, fan_in in (("Wq", d), ("Wk", d), ("Wg", d), ("Wv", d), ("Wo", m)):
        std = float(w[name].std())
        assert abs(std * fan_in ** 0.5 - 1.0) < 0.03, (name, std)
    assert torch.equal(w["gamma"], torch.ones(d))
    assert w["Wg"].shape == (m, d) and w["Wo"].shape == (d, m)


def test_bf16_rounding_is_to_nearest_even():
    one = 1.0
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: ties go to the even mantissa (1.0);
    # 1 + 3 * 2^-8 lies halfway between 1 + 2^-7 and 1 + 2^-6: ties go to 1 + 2^-6
    x = np.array([one + 2.0 ** -8, one + 3 * 2.0 ** -8, one + 2.0 ** -8 + 2.0 ** -12], dtype=np.float32)
    got = synth.cast(x, "bf16").float().numpy()
    assert got.tolist() == [1.0, 1.0 + 2.0 ** -6, 1.0 + 2.0 ** -7]


def test_oracle_view_keeps_the_exact_bits():
    q, *_ = synth.agg_inputs(1, 4, 8, 8, seed=9, dtype="bf16")
    bits = synth.oracle_view(q)
    assert bits.dtype == np.uint16 and bits.shape == (1, 4, 8)
    widened = (bits.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(widened, q.float().numpy())
    f = synth.agg_inputs(1, 4, 8, 8, seed=9, dtype="f32")[0]
    assert synth.oracle_view(f).dtype == np.float32


def test_model_inputs_range_and_embedding_scale():
    ids, E = synth.model_inputs(8, 256, 64, 1000, seed=3, dtype="f32")
    assert ids.dtype == torch.int64 and ids.shape == (8, 256)
    assert int(ids.min()) >= 0 and int(ids.max()) < 1000
    assert abs(float(E.std()) - 0.02) < 0.001 and E.shape == (1000, 64)


@pytest.mark.parametrize("extra", [(), (0, 5, 99, 5)])
def test_random_rows_sorted_unique_in_range(extra):
    rows = synth.random_rows(2, 50, 30, seed=7, extra=extra)
    assert np.all(np.diff(rows) > 0)
    assert rows.min() >= 0 and rows.max() < 100
    assert set(extra) <= set(rows.tolist())
