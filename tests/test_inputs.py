"""Checks of the seeded input generator (shapes, distributions, rounding)."""
import numpy as np

from gated_delta_rule_49_gb300 import inputs


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, 1.0 + 2**-9, -2.5, 3.0e-3], np.float32)
    r = inputs.round_to_bf16(x)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: ties go to the even mantissa (1.0)
    assert r[0] == 1.0 and r[1] == 1.0 and r[2] == np.float32(1.0 + 2**-6)
    assert r[3] == 1.0 and r[4] == -2.5
    assert abs(r[5] - 3.0e-3) <= 3.0e-3 * 2**-8
    b = inputs.bf16_bits(r)
    np.testing.assert_array_equal(inputs.bf16_from_bits(b), r)


def test_tiny_workload_shapes_and_norms():
    p = inputs.make_tiny()
    assert p.q.shape == (1, 256, 1, 32) and p.v.shape == (1, 256, 1, 32)
    assert p.S0 is None and p.dtype == "fp32"
    np.testing.assert_allclose(np.linalg.norm(p.k, axis=-1), 1.0, atol=1e-6)
    assert np.all((p.alpha > 0) & (p.alpha < 1)) and np.all((p.beta > 0) & (p.beta < 1))
    p2 = inputs.make_tiny()
    np.testing.assert_array_equal(p.q, p2.q)  # seeded


def test_prefill_decay_horizons_span_the_pages_range():
    # per-head horizons -1/mean(log alpha) from ~10 to ~1000s of tokens
    p = inputs.make_prefill(B=2, T=512)
    hor = -1.0 / np.log(p.alpha.astype(np.float64)).mean(axis=(0, 1))
    assert hor.min() < 15 and hor.max() > 300
    assert np.all(inputs.round_to_bf16(p.q) == p.q)
    np.testing.assert_allclose(np.linalg.norm(p.q, axis=-1), 1.0, atol=1e-2)


def test_pruned_uses_same_draws_renormalised():
    full = inputs.make_prefill(B=1, T=64, H=4)
    pr = inputs.make_prefill(B=1, T=64, H=4, pruned_K=64)
    idx = pr.meta["kept_channels"]
    assert pr.k.shape[-1] == 64 and idx.shape == (4, 64)
    np.testing.assert_array_equal(pr.v, full.v)
    np.testing.assert_array_equal(pr.alpha, full.alpha)
    np.testing.assert_allclose(np.linalg.norm(pr.k, axis=-1), 1.0, atol=1e-2)
    # same direction as the kept channels of the full-width draw
    h = 2
    a = full.k[0, :, h][:, idx[h]].astype(np.float64)
    b = pr.k[0, :, h].astype(np.float64)
    cos = (a * b).sum(-1) / np.linalg.norm(a, axis=-1) / np.linalg.norm(b, axis=-1)
    assert cos.min() > 0.999


def test_long_workload_key_cone():
    p = inputs.make_long(T=2048)
    m = np.linalg.norm(p.k.astype(np.float64).mean(axis=1), axis=-1)[0]
    assert np.all((m > 0.88) & (m < 0.92)), m
    assert p.alpha.min() >= 0.9995 - 1e-7 and p.alpha.max() <= 0.9999 + 1e-7


def test_decode_initial_state_low_stable_rank():
    import oracle
    p = inputs.make_decode(B=2, H=2, steps=4)
    assert p.S0.shape == (2, 2, 128, 128)
    er = oracle.stable_rank(p.S0)[2]
    assert np.all((er > 1.0) & (er < 3.0)), er
    pp = inputs.make_decode(B=2, H=2, steps=4, pruned_K=64)
    assert pp.S0.shape == (2, 2, 128, 64) and pp.k.shape[-1] == 64
