"""The chunkwise algebra the kernels implement equals the token-by-token oracle.

The oracle is pinned on its own (test_oracle_pins.py); this file checks that
the chunk form with 16-token sub-tile factoring (tests/chunk_algebra.py) is the
same function, at the edge lengths the kernels must handle and at the decay
bound (every g at -5, so every sub-tile reaches cumulative log decay -80).
"""
import numpy as np
import pytest

import oracle
from tests.chunk_algebra import chunk_forward_fp64
from tests.helpers import rand_inputs, rel_max_err


@pytest.mark.parametrize("L", [1, 15, 16, 17, 63, 64, 65, 127, 200])
def test_chunk_form_matches_oracle(L):
    rng = np.random.default_rng(100 + L)
    dk, dv = 16, 12
    q, k, v, g, b = rand_inputs(rng, L, dk, dv)
    S0 = 0.1 * rng.standard_normal((1, 1, dk, dv))
    ro, rs = oracle.forward(q, k, v, g, b, S0)
    co, cs = chunk_forward_fp64(q[0, :, 0], k[0, :, 0], v[0, :, 0], g[0, :, 0], b[0, :, 0], S0[0, 0])
    assert rel_max_err(co, ro[0, :, 0]) < 1e-12
    assert rel_max_err(cs, rs[0, 0]) < 1e-12


def test_chunk_form_at_the_decay_bound():
    rng = np.random.default_rng(7)
    L, dk, dv = 192, 32, 8
    q, k, v, g, b = rand_inputs(rng, L, dk, dv)
    g[:] = -5.0
    ro, rs = oracle.forward(q, k, v, g, b, None)
    co, cs = chunk_forward_fp64(q[0, :, 0], k[0, :, 0], v[0, :, 0], g[0, :, 0], b[0, :, 0],
                                np.zeros((dk, dv)))
    assert rel_max_err(co, ro[0, :, 0]) < 1e-12
    assert rel_max_err(cs, rs[0, 0]) < 1e-12


def test_sub_tile_factors_stay_in_bf16_range():
    """With g in [-5, 0], every factor the sub-tile split forms lies in [e^-80, e^80]."""
    bf16_max = (2 - 2 ** -7) * 2.0 ** 127
    g = np.full((64, 4), -5.0)
    gam = np.cumsum(g, axis=0)
    ref = np.zeros((4, 4)); ref[1:] = gam[15:63:16]
    x = np.exp(gam - ref[np.arange(64) // 16])
    assert x.min() >= np.exp(-80) * (1 - 1e-12) and x.max() <= 1.0
    assert (1 / x).max() <= np.exp(80) * (1 + 1e-12) < bf16_max
