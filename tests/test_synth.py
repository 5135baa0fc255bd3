"""Seeded input generator: determinism, layouts and the bf16 rounding (no GPU)."""
import numpy as np

import synth


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-9, -2.5, 3.0e38, 1e-40], dtype=np.float32)
    b = synth.f32_to_bf16_bits(x)
    y = synth.bf16_bits_to_f32(b)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: even mantissa -> 1.0
    assert y[0] == 1.0 and y[1] == 1.0 and y[2] == np.float32(1.0 + 2**-7) and y[3] == -2.5
    # exact for values already representable
    z = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(y))
    assert np.array_equal(z, y)
    # nearest: |x - y| <= half an ulp of bf16
    r = np.random.default_rng(0).normal(size=10000).astype(np.float32)
    rb = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(r))
    assert np.all(np.abs(rb - r) <= np.abs(r) * 2.0**-8)


def test_deterministic_and_shapes():
    a = synth.make_prefill("gdn4k", seed=0, B=1, T=70, H=2)
    b = synth.make_prefill("gdn4k", seed=0, B=1, T=70, H=2)
    c = synth.make_prefill("gdn4k", seed=1, B=1, T=70, H=2)
    for name in ("q", "k", "v", "alpha", "eta"):
        assert np.array_equal(getattr(a, name), getattr(b, name))
        assert not np.array_equal(getattr(a, name), getattr(c, name))
    assert a.q.shape == (1, 70, 2, 128) and a.q.dtype == np.uint16
    assert a.alpha.shape == (1, 70, 2) and a.alpha.dtype == np.float32
    assert np.all((a.alpha > 0) & (a.alpha < 1)) and np.all((a.eta > 0) & (a.eta < 1))
    kd = synth.make_prefill("kda8k", seed=0, B=1, T=16, H=1)
    assert kd.alpha.shape == (1, 16, 1, 128)
    t = synth.make_prefill("tiny")
    assert t.q.dtype == np.float32 and t.q.shape == (1, 64, 1, 16) and t.S0 is None


def test_gate_distribution_matches_recipe():
    a = synth.make_prefill("gdn4k", seed=0, B=2, T=4096, H=4).alpha.astype(np.float64)
    # alpha = exp(-softplus(x)), x ~ N(-4, 1): E[-log alpha] = E[softplus(x)] ~= 0.030
    m = float(np.mean(-np.log(a)))
    assert 0.025 < m < 0.035, m


def test_decode_inputs():
    d = synth.make_decode(seed=0, B=2, H=3, steps=5)
    assert d.q.shape == (5, 2, 3, 128) and d.S.shape == (2, 3, 128, 128)
    assert abs(float(np.std(d.S)) - 0.02) < 0.002
