"""Pins of the oracle's q/k L2 normalisation (``oracle.l2norm_rows``, ``oracle.round_bf16``).

The method reads q and k after L2 normalisation ("はじめての自然言語処理 -- Kimi K3",
section 3.1, the associative-memory read-out paragraph).  These checks tie the oracle's
version to values worked out by hand, to a library conversion, and to the exact-overwrite
property of the recurrence, so that a dropped square root, a missing eps, the wrong axis, a
wrong rounding or a normalisation applied after the recurrence reads k fails one of them.
"""
import numpy as np
import pytest
import torch

import oracle


def test_round_bf16_hand_values():
    # bf16 spacing on [0.5, 1) is 2^-8: 0.6 = 153.6 steps -> 154, 0.8 = 204.8 -> 205
    assert oracle.round_bf16(np.array([0.6]))[0] == 154 * 2.0 ** -8
    assert oracle.round_bf16(np.array([0.8]))[0] == 205 * 2.0 ** -8
    assert oracle.round_bf16(np.array([-0.6]))[0] == -154 * 2.0 ** -8
    # halfway cases on [1, 2) (spacing 2^-7) go to the even neighbour
    assert oracle.round_bf16(np.array([1 + 2.0 ** -8]))[0] == 1.0
    assert oracle.round_bf16(np.array([1 + 3 * 2.0 ** -8]))[0] == 1 + 2.0 ** -6
    # subnormal range: steps of 2^-133, halfway to even; below half a step -> 0
    assert oracle.round_bf16(np.array([3 * 2.0 ** -134]))[0] == 2.0 ** -132
    assert oracle.round_bf16(np.array([2.0 ** -140]))[0] == 0.0
    assert oracle.round_bf16(np.array([2.0 ** -130]))[0] == 2.0 ** -130


def test_round_bf16_matches_torch_on_float32_values():
    # from float32 values torch's conversion rounds once, to nearest even
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(20000) * np.exp(rng.uniform(-30, 30, 20000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    assert np.array_equal(oracle.round_bf16(x.astype(np.float64)), ref)


def test_l2norm_closed_forms():
    y = oracle.l2norm_rows(np.array([[3.0, 4.0, 0.0, 0.0]]), 0.0)
    assert y[0, 0] == 0.6 and y[0, 1] == 0.8 and y[0, 2] == 0.0
    # eps enters under the root: (1, 0) with eps = 3 -> 1 / sqrt(4)
    assert oracle.l2norm_rows(np.array([[1.0, 0.0]]), 3.0)[0, 0] == 0.5
    # a zero row stays zero, also with eps = 0
    z = oracle.l2norm_rows(np.zeros((2, 8)), 0.0)
    assert np.array_equal(z, np.zeros((2, 8)))
    # rounded to bf16 after normalising
    assert np.array_equal(oracle.l2norm_rows(np.array([[3.0, 4.0]]), 0.0, "bf16"),
                          np.array([[154 * 2.0 ** -8, 205 * 2.0 ** -8]]))


def test_l2norm_unit_rows_and_axis():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((3, 7, 2, 64)) * rng.uniform(0.1, 30, (3, 7, 2, 1))
    y = oracle.l2norm_rows(x, 0.0)
    assert np.max(np.abs(np.sum(y * y, axis=-1) - 1.0)) < 1e-14
    # each row is a positive multiple of its input row
    ratio = y / x
    assert np.max(np.abs(ratio - ratio[..., :1])) < 1e-12 * np.max(np.abs(ratio))
    assert np.all(ratio > 0)


def test_l2norm_scale_invariance_exact():
    # doubling a row is exact, and so are sqrt(4 s) = 2 sqrt(s) and the quotient
    rng = np.random.default_rng(7)
    x = rng.standard_normal((50, 128))
    assert np.array_equal(oracle.l2norm_rows(2.0 * x, 0.0), oracle.l2norm_rows(x, 0.0))
    assert np.array_equal(oracle.l2norm_rows(0.25 * x, 0.0, "bf16"), oracle.l2norm_rows(x, 0.0, "bf16"))


@pytest.mark.parametrize("io", ["f64", "bf16"])
def test_normalised_keys_overwrite_exactly(io):
    # g = 0, beta = 1 and keys that are scaled unit vectors: once normalised they are the unit
    # vectors themselves, and each write replaces that row of S by v exactly (the delta rule's
    # overwrite); rows no key touches keep S0.  With the scale left in, the row would be
    # written with c^2-weighted corrections instead.
    rng = np.random.default_rng(11)
    dk, dv, T = 8, 5, 4
    slots = [2, 5, 2, 7]
    scale = [3.0, 0.5, 12.0, 2.0 ** -6]
    k = np.zeros((1, T, 1, dk))
    for t in range(T):
        k[0, t, 0, slots[t]] = scale[t]
    q = rng.standard_normal((1, T, 1, dk))
    v = rng.standard_normal((1, T, 1, dv))
    g = np.zeros((1, T, 1, dk))
    beta = np.ones((1, T, 1))
    s0 = rng.standard_normal((1, 1, dk, dv))
    kn = oracle.l2norm_rows(k, 1e-300 if io == "f64" else 0.0, io)
    qn = oracle.l2norm_rows(q, 0.0, io)
    _, sT = oracle.forward(qn, kn, v, g, beta, s0)
    last = {s: t for t, s in enumerate(slots)}
    for i in range(dk):
        want = v[0, last[i], 0] if i in last else s0[0, 0, i]
        assert np.max(np.abs(sT[0, 0, i] - want)) < 1e-12, i
