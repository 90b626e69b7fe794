"""Pins of oracle.gated_rmsnorm (CPU): properties the gate's definition fixes, checked
without retyping its formula."""
import numpy as np

import oracle


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_open_gate_gives_unit_rms_rows():
    o = _rand((5, 7, 64), 1)
    y = oracle.gated_rmsnorm(o, np.full(o.shape, 60.0), eps=0.0)   # sigmoid(60) == 1 in fp64
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, rtol=1e-12)
    # the direction of each row is o's
    cos = np.sum(y * o, axis=-1) / np.linalg.norm(y, axis=-1) / np.linalg.norm(o, axis=-1)
    np.testing.assert_allclose(cos, 1.0, rtol=1e-12)


def test_zero_logit_halves_and_closed_gate_vanishes():
    o, w = _rand((3, 32), 2), _rand(32, 3)
    full = oracle.gated_rmsnorm(o, np.full(o.shape, 60.0), w)
    np.testing.assert_allclose(oracle.gated_rmsnorm(o, np.zeros(o.shape), w), 0.5 * full, rtol=1e-12)
    with np.errstate(over="ignore"):   # exp(800) overflows to inf: the gate is exactly 0
        assert np.all(np.abs(oracle.gated_rmsnorm(o, np.full(o.shape, -800.0), w)) < 1e-300)


def test_scale_invariance_and_weight_linearity():
    o, z, w = _rand((4, 16), 4), _rand((4, 16), 5), _rand(16, 6)
    base = oracle.gated_rmsnorm(o, z, w, eps=0.0)
    np.testing.assert_allclose(oracle.gated_rmsnorm(37.5 * o, z, w, eps=0.0), base, rtol=1e-12)
    np.testing.assert_allclose(oracle.gated_rmsnorm(o, z, 3.0 * w, eps=0.0), 3.0 * base, rtol=1e-12)
    np.testing.assert_allclose(oracle.gated_rmsnorm(o, z, None), oracle.gated_rmsnorm(o, z, np.ones(16)),
                               rtol=0, atol=0)


def test_gate_is_the_logistic_function_channel_by_channel():
    """Each channel's factor is in (0, 1), increasing in its own logit, and
    sigmoid(z) + sigmoid(-z) == 1."""
    o = np.ones((1, 8))
    z = np.linspace(-4, 4, 8)[None]
    a, b = oracle.gated_rmsnorm(o, z, eps=0.0), oracle.gated_rmsnorm(o, -z, eps=0.0)
    assert np.all((a > 0) & (a < 1)) and np.all(np.diff(a[0]) > 0)
    np.testing.assert_allclose(a + b, 1.0, rtol=1e-14)


def test_eps_enters_as_the_stated_floor():
    """A zero row stays zero; a row with mean square m is scaled by 1 / sqrt(m + eps)."""
    y = oracle.gated_rmsnorm(np.zeros((1, 8)), np.full((1, 8), 60.0), eps=1e-6)
    assert np.all(y == 0.0)
    o = np.full((1, 4), 2.0)   # mean square 4
    y = oracle.gated_rmsnorm(o, np.full((1, 4), 60.0), eps=5.0)   # 2 / sqrt(9)
    np.testing.assert_allclose(y, 2.0 / 3.0, rtol=1e-14)
