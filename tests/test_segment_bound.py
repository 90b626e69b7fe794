"""CPU pins of the bound the sequence split relies on.

A segment of a sequence may start from a zero state at an earlier token w when the transitions
between w and its first token shrink every state enough: for one token,
    || (I - beta k k^T) Diag(e^g) ||_2  <=  max_i e^{g_i} * max(1, |1 - beta |k|^2|)
(Diag(e^g) has norm max_i e^{g_i}; I - beta k k^T is symmetric with eigenvalues 1 and
1 - beta |k|^2), and the norm of a product is at most the product of the norms.  So the state
reached from a zero start at w differs from the true state by the true state at w carried
through those transitions, whose norm is at most that product times ||S_w||.  Checked here in
fp64: the one-token bound, the product bound on explicit transition matrices, and, through the
oracle, the difference between a full run and a run started from zero at w, with keys that are
and are not unit vectors and with decays that do and do not reach the bound.
"""
import numpy as np
import pytest

import oracle
from tests.helpers import rand_inputs


def token_bound(g, beta, k):
    return np.exp(g.max()) * max(1.0, abs(1.0 - beta * float(k @ k)))


def transition(g, beta, k):
    return (np.eye(k.size) - beta * np.outer(k, k)) @ np.diag(np.exp(g))


@pytest.mark.parametrize("seed", range(6))
def test_one_token_norm_bound(seed):
    rng = np.random.default_rng(seed)
    for _ in range(200):
        d = int(rng.integers(1, 9))
        k = rng.standard_normal(d) * rng.uniform(0.1, 2.0)
        g = -5.0 * rng.uniform(0, 1, d) * (rng.uniform() < 0.8)
        beta = rng.uniform(0, 1.5)
        n = np.linalg.norm(transition(g, beta, k), 2)
        assert n <= token_bound(g, beta, k) * (1 + 1e-12)


def test_the_bound_is_attained():
    # a unit key along the slowest channel with beta = 0 gives exactly max_i e^{g_i}, and
    # beta |k|^2 = 3 stretches the key direction by exactly 2
    g = np.array([-1.0, -3.0, -0.25])
    k = np.array([0.0, 0.0, 1.0])
    assert np.isclose(np.linalg.norm(transition(g, 0.0, k), 2), np.exp(-0.25))
    k = np.array([1.0, 0.0, 0.0]) * np.sqrt(3.0)
    g = np.zeros(3)
    assert np.isclose(np.linalg.norm(transition(g, 1.0, k), 2), 2.0)


@pytest.mark.parametrize("seed", range(4))
def test_product_bound_on_explicit_transitions(seed):
    rng = np.random.default_rng(100 + seed)
    d, T = 6, 30
    k = rng.standard_normal((T, d)) * rng.uniform(0.3, 1.6, (T, 1))
    g = -5.0 * rng.uniform(0, 1, (T, d))
    beta = rng.uniform(0, 1.2, T)
    phi = np.eye(d)
    bound = 1.0
    for t in range(T):
        phi = transition(g[t], beta[t], k[t]) @ phi
        bound *= token_bound(g[t], beta[t], k[t])
        assert np.linalg.norm(phi, 2) <= bound * (1 + 1e-10)


@pytest.mark.parametrize("normalised", [True, False])
@pytest.mark.parametrize("decay", ["bound", "sigmoid", "one_channel_still"])
def test_zero_start_differs_by_at_most_the_bound(normalised, decay):
    rng = np.random.default_rng(7)
    T, d, w = 90, 8, 37
    q, k, v, g, b = rand_inputs(rng, T, d, d)
    if not normalised:
        k = k * rng.uniform(0.5, 1.5, (1, T, 1, 1))
    if decay == "bound":
        g = np.full_like(g, -5.0)
    elif decay == "one_channel_still":
        g[..., 3] = 0.0
    S0 = rng.standard_normal((1, 1, d, d))
    # the true state at w, and at T from the start
    _, Sw = oracle.forward(q[:, :w], k[:, :w], v[:, :w], g[:, :w], b[:, :w], S0)
    out, ST = oracle.forward(q, k, v, g, b, S0)
    # from a zero state at w
    out_w, ST_w = oracle.forward(q[:, w:], k[:, w:], v[:, w:], g[:, w:], b[:, w:], None)
    bound = np.prod([token_bound(g[0, t, 0], b[0, t, 0], k[0, t, 0]) for t in range(w, T)])
    diff = np.linalg.norm(ST[0, 0] - ST_w[0, 0])
    rnd = 1e-13 * np.linalg.norm(ST[0, 0])   # the two fp64 runs round differently
    assert diff <= bound * np.linalg.norm(Sw[0, 0]) * (1 + 1e-9) + rnd
    if decay == "bound":
        assert bound < 2.0 ** -160      # 53 tokens at g = -5: far past the horizon
    if decay == "one_channel_still" and normalised:
        assert bound == 1.0              # no horizon: a segment would start at the sequence start
    # the outputs after w obey the same bound token by token (each o_t = S_t^T q_t)
    for t in range(w, T, 7):
        bt = np.prod([token_bound(g[0, s, 0], b[0, s, 0], k[0, s, 0]) for s in range(w, t + 1)])
        do = np.linalg.norm(out[0, t, 0] - out_w[0, t - w, 0])
        rnd = 1e-13 * max(1.0, np.linalg.norm(out[0, t, 0]))
        assert do <= bt * np.linalg.norm(Sw[0, 0], 2) * np.linalg.norm(q[0, t, 0]) * (1 + 1e-9) + rnd


def warm_start_rule(g, beta, k, c_lo, C=64, horizon_log2=160.0, max_chunks=16):
    """The chunk boundary a segment whose first stored chunk is c_lo starts from: the latest
    one at most max_chunks chunks earlier where the summed per-token log2 bounds reach
    -horizon_log2, else 0 (the sequence start, with the initial state)."""
    acc = 0.0
    for c in range(c_lo - 1, max(0, c_lo - max_chunks) - 1, -1):
        for t in range(c * C, (c + 1) * C):
            acc += np.log2(token_bound(g[t], beta[t], k[t]))
        if acc <= -horizon_log2:
            return c
    return 0


@pytest.mark.parametrize("decay", ["bound", "sigmoid", "one_channel_still"])
@pytest.mark.parametrize("P", [2, 3, 5])
def test_segmented_runs_equal_the_full_run(decay, P):
    # the segment scheme the tensor-core kernel uses, run with the oracle in fp64: segment p
    # stores chunks [p nc / P, (p+1) nc / P) and runs from warm_start_rule's boundary
    rng = np.random.default_rng(11)
    C, nc, d = 64, 13, 8
    T = nc * C - 20                      # a ragged last chunk
    q, k, v, g, b = rand_inputs(rng, T, d, d)
    if decay == "bound":
        g = np.full_like(g, -5.0)
    elif decay == "one_channel_still":
        g[..., 2] = 0.0
    S0 = rng.standard_normal((1, 1, d, d))
    out, ST = oracle.forward(q, k, v, g, b, S0)
    seg_out = np.full_like(out, np.nan)
    for p in range(P):
        c_lo, c_hi = p * nc // P, (p + 1) * nc // P
        if c_lo == c_hi:
            continue
        c_run = warm_start_rule(g[0, :, 0], b[0, :, 0], k[0, :, 0], c_lo) if c_lo > 0 else 0
        t0, t1 = c_run * C, min(c_hi * C, T)
        o_p, s_p = oracle.forward(q[:, t0:t1], k[:, t0:t1], v[:, t0:t1], g[:, t0:t1], b[:, t0:t1],
                                  S0 if c_run == 0 else None)
        seg_out[:, c_lo * C:t1] = o_p[:, c_lo * C - t0:]
        if p == P - 1:
            seg_state = s_p
        if decay == "bound" and c_lo > 0:
            assert c_run == c_lo - 1      # one chunk of g = -5 is 461 below the log2 horizon
        if decay == "one_channel_still" and c_lo > 0:
            assert c_run == 0             # no horizon: from the start, with S0
    assert not np.isnan(seg_out).any()
    scale = np.sqrt(np.mean(out ** 2))
    assert np.abs(seg_out - out).max() <= 1e-12 * scale
    assert np.abs(seg_state - ST).max() <= 1e-12 * np.sqrt(np.mean(ST ** 2))
