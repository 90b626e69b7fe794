"""Pins of the fp64 oracle against things other than itself.

Each check follows the KDA description in "はじめての自然言語処理 -- Kimi K3"
(ogis-ri.co.jp), section 3.1:
  * brute force -- the folded one-line form, report equation (1):
    S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T, built
    as explicit dense transition matrices and multiplied out;
  * exact rational arithmetic on a tiny case (sympy);
  * closed forms: beta = 0 is pure per-channel decay; g = 0, beta = 1 with
    orthonormal keys overwrites each stored association exactly ("beta = 1
    replaces the value for that key"); g = 0 with orthonormal keys reads out
    o = sum_i beta_i (q . k_i) v_i (the associative-memory read paragraph);
    the scalar dk = dv = 1 recurrence;
  * invariants: any split point gives the same result when the state is carried,
    packed sequences equal separate runs, (V, S_0) -> (O, S_T) is linear;
  * the decay bound numbers of the lower-bound paragraph (g >= -5, 16-token
    tiles within [-80, 0], e^80 below the bf16 maximum);
  * planted mistakes (mutated copies of the oracle source) must fail the pins.
"""
import ctypes
import math
import os
import re
import subprocess

import numpy as np
import pytest

import oracle
from tests.helpers import rand_inputs, rel_max_err

ORACLE_SRC = os.path.join(os.path.dirname(oracle.__file__), "kda_oracle.c")


# ----------------------------------------------------------------------------- brute force
def brute_force(q, k, v, g, beta, S0):
    """One (sequence, head): explicit transition products, no recurrence loop state."""
    T, dk = q.shape
    dv = v.shape[1]
    M = [(np.eye(dk) - beta[t] * np.outer(k[t], k[t])) @ np.diag(np.exp(g[t]))
         for t in range(T)]

    def prod(hi, lo):  # M_hi M_{hi-1} ... M_lo  (identity when hi < lo)
        P = np.eye(dk)
        for s in range(lo, hi + 1):
            P = M[s] @ P
        return P

    outs, S = [], None
    for t in range(T):
        S = prod(t, 0) @ S0
        for s in range(t + 1):
            S = S + prod(t, s + 1) @ (beta[s] * np.outer(k[s], v[s]))
        outs.append(S.T @ q[t])
    return np.array(outs), S


@pytest.mark.parametrize("T,dk,dv,seed", [(1, 3, 5, 0), (7, 4, 3, 1), (24, 5, 6, 2),
                                          (40, 8, 8, 3), (64, 6, 2, 4)])
def test_brute_force(T, dk, dv, seed):
    rng = np.random.default_rng(seed)
    q, k, v, g, b = rand_inputs(rng, T, dk, dv)
    S0 = 0.3 * rng.standard_normal((1, 1, dk, dv))
    out, sT = oracle.forward(q, k, v, g, b, S0)
    ro, rs = brute_force(q[0, :, 0], k[0, :, 0], v[0, :, 0], g[0, :, 0], b[0, :, 0], S0[0, 0])
    assert rel_max_err(out[0, :, 0], ro) < 1e-12
    assert rel_max_err(sT[0, 0], rs) < 1e-12


def test_exact_rational_tiny():
    """d_k = 2, d_v = 3, T = 3 in exact rationals (alpha given as rationals, g = ln alpha)."""
    sp = pytest.importorskip("sympy")
    R = sp.Rational
    alpha = [[R(1, 2), R(3, 4)], [R(9, 10), R(1, 5)], [R(2, 3), R(7, 8)]]
    kk = [[R(3, 5), R(4, 5)], [R(1, 1), R(0)], [R(-5, 13), R(12, 13)]]
    qq = [[R(0), R(1)], [R(8, 17), R(-15, 17)], [R(1, 2), R(1, 3)]]
    vv = [[R(1), R(-2), R(3)], [R(1, 2), R(0), R(-1, 4)], [R(2), R(5, 7), R(1)]]
    bb = [R(1, 3), R(3, 4), R(1, 2)]
    S = sp.Matrix([[R(1, 10), R(0), R(-1, 5)], [R(0), R(3, 10), R(1, 7)]])
    outs = []
    for t in range(3):
        kt = sp.Matrix(kk[t]); qt = sp.Matrix(qq[t]); vt = sp.Matrix(vv[t])
        S = (sp.eye(2) - bb[t] * kt * kt.T) * sp.diag(*alpha[t]) * S + bb[t] * kt * vt.T
        outs.append(list(S.T * qt))
    S0 = np.array([[0.1, 0.0, -0.2], [0.0, 0.3, 1 / 7]]).reshape(1, 1, 2, 3)
    f = lambda a: np.array(a, dtype=np.float64)
    q = f([[float(x) for x in r] for r in qq]).reshape(1, 3, 1, 2)
    k = f([[float(x) for x in r] for r in kk]).reshape(1, 3, 1, 2)
    v = f([[float(x) for x in r] for r in vv]).reshape(1, 3, 1, 3)
    g = f([[math.log(float(x)) for x in r] for r in alpha]).reshape(1, 3, 1, 2)
    b = f([float(x) for x in bb]).reshape(1, 3, 1)
    out, sT = oracle.forward(q, k, v, g, b, S0)
    exp_out = f([[float(x) for x in r] for r in outs])
    exp_S = f(S.tolist())
    np.testing.assert_allclose(out[0, :, 0], exp_out, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(sT[0, 0], exp_S, rtol=1e-13, atol=1e-14)


# ----------------------------------------------------------------------------- closed forms
def test_beta_zero_is_pure_decay():
    rng = np.random.default_rng(5)
    T, dk, dv = 50, 7, 4
    q, k, v, g, b = rand_inputs(rng, T, dk, dv, beta=0.0)
    S0 = rng.standard_normal((1, 1, dk, dv))
    out, sT = oracle.forward(q, k, v, g, b, S0)
    cum = np.cumsum(g[0, :, 0], axis=0)                     # [T, dk]
    St = np.exp(cum)[:, :, None] * S0[0, 0][None]          # [T, dk, dv]
    ref_o = np.einsum("tij,ti->tj", St, q[0, :, 0])
    assert rel_max_err(out[0, :, 0], ref_o) < 1e-13
    assert rel_max_err(sT[0, 0], St[-1]) < 1e-13


def test_unit_beta_overwrites_orthonormal_keys():
    rng = np.random.default_rng(6)
    dk, dv = 8, 5
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    key_ids = [0, 1, 2, 1, 3, 0, 4]           # repeated keys: the last write must win
    T = len(key_ids)
    k = np.stack([Qm[:, i] for i in key_ids]).reshape(1, T, 1, dk)
    q = rng.standard_normal((1, T, 1, dk))
    v = rng.standard_normal((1, T, 1, dv))
    g = np.zeros((1, T, 1, dk))
    b = np.ones((1, T, 1))
    S0 = rng.standard_normal((1, 1, dk, dv))
    _, sT = oracle.forward(q, k, v, g, b, S0)
    S = sT[0, 0]
    last = {i: t for t, i in enumerate(key_ids)}
    for i, t in last.items():
        np.testing.assert_allclose(S.T @ Qm[:, i], v[0, t, 0], rtol=0, atol=1e-13)
    for i in range(5, dk):                     # directions no key touched keep S_0
        np.testing.assert_allclose(S.T @ Qm[:, i], S0[0, 0].T @ Qm[:, i], rtol=0, atol=1e-13)


def test_associative_read_without_decay():
    rng = np.random.default_rng(7)
    dk, dv, T = 9, 4, 6
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    k = Qm[:, :T].T.reshape(1, T, 1, dk)
    q = rng.standard_normal((1, T, 1, dk))
    v = rng.standard_normal((1, T, 1, dv))
    b = rng.uniform(0.1, 0.9, size=(1, T, 1))
    out, _ = oracle.forward(q, k, v, np.zeros((1, T, 1, dk)), b, None)
    for t in range(T):
        ref = sum(b[0, i, 0] * (q[0, t, 0] @ k[0, i, 0]) * v[0, i, 0] for i in range(t + 1))
        np.testing.assert_allclose(out[0, t, 0], ref, rtol=1e-13, atol=1e-13)


def test_scalar_recurrence():
    rng = np.random.default_rng(8)
    T = 200
    q, k, v = (rng.standard_normal(T) for _ in range(3))
    g = rng.uniform(-5, 0, T)
    b = rng.uniform(0, 1, T)
    s, ref = 0.7, []
    for t in range(T):
        s = (1 - b[t] * k[t] ** 2) * math.exp(g[t]) * s + b[t] * k[t] * v[t]
        ref.append(s * q[t])
    r4 = lambda a: a.reshape(1, T, 1, 1)
    out, sT = oracle.forward(r4(q), r4(k), r4(v), r4(g), b.reshape(1, T, 1),
                             np.full((1, 1, 1, 1), 0.7))
    np.testing.assert_allclose(out[0, :, 0, 0], ref, rtol=1e-12, atol=1e-14)
    assert abs(sT[0, 0, 0, 0] - s) < 1e-13


# ----------------------------------------------------------------------------- invariants
def test_split_invariance_every_point():
    rng = np.random.default_rng(9)
    T, dk, dv = 37, 6, 5
    q, k, v, g, b = rand_inputs(rng, T, dk, dv, H=2)
    S0 = rng.standard_normal((1, 2, dk, dv))
    out, sT = oracle.forward(q, k, v, g, b, S0)
    for t0 in range(0, T + 1):
        o1, s1 = oracle.forward(q[:, :t0], k[:, :t0], v[:, :t0], g[:, :t0], b[:, :t0], S0)
        o2, s2 = oracle.forward(q[:, t0:], k[:, t0:], v[:, t0:], g[:, t0:], b[:, t0:], s1)
        np.testing.assert_allclose(np.concatenate([o1, o2], axis=1), out, rtol=0, atol=1e-13)
        np.testing.assert_allclose(s2, sT, rtol=0, atol=1e-13)


def test_packed_equals_separate():
    rng = np.random.default_rng(10)
    lens = [1, 17, 64, 5, 130]
    dk, dv, H = 5, 3, 2
    parts = [rand_inputs(rng, L, dk, dv, H=H) for L in lens]
    S0 = rng.standard_normal((len(lens), H, dk, dv))
    cat = [np.concatenate([p[i] for p in parts], axis=1) for i in range(5)]
    cu = np.concatenate([[0], np.cumsum(lens)])
    out, sT = oracle.forward(*cat, S0, cu)
    for n, p in enumerate(parts):
        o, s = oracle.forward(*p, S0[n:n + 1])
        np.testing.assert_array_equal(out[:, cu[n]:cu[n + 1]], o)
        np.testing.assert_array_equal(sT[n], s[0])


def test_linear_in_values_and_state():
    rng = np.random.default_rng(11)
    T, dk, dv = 30, 6, 4
    q, k, v1, g, b = rand_inputs(rng, T, dk, dv)
    v2 = rng.standard_normal(v1.shape)
    s1 = rng.standard_normal((1, 1, dk, dv))
    s2 = rng.standard_normal((1, 1, dk, dv))
    a, c = 0.7, -1.3
    o1, t1 = oracle.forward(q, k, v1, g, b, s1)
    o2, t2 = oracle.forward(q, k, v2, g, b, s2)
    o3, t3 = oracle.forward(q, k, a * v1 + c * v2, g, b, a * s1 + c * s2)
    np.testing.assert_allclose(o3, a * o1 + c * o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(t3, a * t1 + c * t2, rtol=0, atol=1e-12)


def test_state_size_does_not_grow_with_length():
    rng = np.random.default_rng(12)
    for T in (1, 10, 300):
        q, k, v, g, b = rand_inputs(rng, T, 4, 3)
        _, sT = oracle.forward(q, k, v, g, b, None)
        assert sT.shape == (1, 1, 4, 3)


def test_decode_step_equals_one_token_forward():
    rng = np.random.default_rng(13)
    N, H, dk, dv = 5, 3, 6, 4
    q, k, v, g, b = rand_inputs(rng, 1, dk, dv, H=H, B=N)   # [N, 1, H, d]
    pool = rng.standard_normal((N + 2, H, dk, dv))
    idx = np.array([3, 0, 6, 2, 5])
    ref_pool = pool.copy()
    out = oracle.decode_step(q[:, 0], k[:, 0], v[:, 0], g[:, 0], b[:, 0], pool, idx)
    for n in range(N):
        o, s = oracle.forward(q[n:n + 1], k[n:n + 1], v[n:n + 1], g[n:n + 1], b[n:n + 1],
                              ref_pool[idx[n]][None])
        np.testing.assert_array_equal(out[n], o[0, 0])
        np.testing.assert_array_equal(pool[idx[n]], s[0])
    untouched = [i for i in range(N + 2) if i not in idx]
    np.testing.assert_array_equal(pool[untouched], ref_pool[untouched])


# ----------------------------------------------------------------------------- decay bound
def test_decay_bound_numbers():
    """g >= -5 per step => alpha >= e^-5 ~= 0.0067; 16 steps => log decay >= -80;
    e^80 ~= 5.5e34 stays below the bf16 maximum ~= 3.39e38."""
    bf16_max = (2 - 2 ** -7) * 2.0 ** 127
    assert abs(bf16_max - 3.3895e38) / 3.3895e38 < 1e-4
    assert math.exp(80) < bf16_max
    assert abs(math.exp(80) - 5.54e34) / 5.54e34 < 1e-2
    assert abs(math.exp(-5) - 0.0067) < 1e-4
    torch = pytest.importorskip("torch")
    from linear_attention_fwd_gb300 import inputs
    d = inputs.make_prefill(batch=1, seqlen=256, heads=2, dk=16, dv=16,
                            dtype=torch.bfloat16, g_mode="near_bound", seed=3)
    g = d["g"].double().numpy()
    assert np.all(g == -5.0)            # -5 + 0.01 U(0,1) rounds to -5 in bf16
    tiles = g.reshape(1, 16, 16, 2, 16).sum(axis=2)
    assert tiles.min() >= -80.0 and np.exp(-tiles.min()) < bf16_max
    d = inputs.make_prefill(batch=1, seqlen=256, heads=2, dk=16, dv=16,
                            dtype=torch.bfloat16, g_mode="sigmoid", seed=4)
    g = d["g"].double().numpy()
    assert g.min() >= -5.0 and g.max() <= 0.0


def test_decay_across_the_bound_closed_form():
    """One writing token after a sub-tile at the bound: with every key the same unit vector
    and only token 15 writing (beta = 1, v = 100), o_r = 100 e^{gamma_r - gamma_15} for
    r >= 15 and the state ends at 100 e^{gamma_63 - gamma_15} in that key's row.  Tokens
    0-15 decay by -5 each (the sub-tile reaches -80) and later ones by -0.25, so the values
    reach e^-12 of the write: the oracle carries them in full (they are far above fp64's
    range limits)."""
    T, d = 64, 4
    q = np.zeros((1, T, 1, d)); q[..., 0] = 1.0
    k = q.copy()
    v = np.zeros((1, T, 1, d)); v[0, 15] = 100.0
    g = np.full((1, T, 1, d), -0.25); g[0, :16] = -5.0
    b = np.zeros((1, T, 1)); b[0, 15] = 1.0
    o, s = oracle.forward(q, k, v, g, b)
    r = np.arange(T)
    ref = np.where(r >= 15, 100.0 * np.exp(-0.25 * np.maximum(r - 15, 0)), 0.0)
    np.testing.assert_allclose(o[0, :, 0, 1], ref, rtol=1e-13, atol=0)
    np.testing.assert_allclose(s[0, 0, 0, :], 100.0 * math.exp(-12.0), rtol=1e-13)
    assert np.count_nonzero(s[0, 0, 1:, :]) == 0


# ----------------------------------------------------------------------------- planted mistakes
def _mutants():
    src = open(ORACLE_SRC).read()
    forget = re.search(r"    /\* forget.*?\n    }\n", src, re.S).group(0)
    read = re.search(r"    /\* read with the current key.*?e\[j\] = v\[j\] - e\[j\];\n", src, re.S).group(0)
    write = re.search(r"    /\* write the correction.*?\n    }\n", src, re.S).group(0)
    out = re.search(r"    /\* read-out with the updated state.*?o\[j\] \+= S\[i \* dv \+ j\] \* q\[i\];\n", src, re.S).group(0)
    body = forget + read + write + out
    assert body in src
    return {
        "decay_after_read": src.replace(body, read + forget + write + out),
        "readout_before_write": src.replace(body, forget + read + out + write),
        "no_beta_on_write": src.replace("const double bk = beta * k[i];", "const double bk = k[i];"),
        "delta_sign": src.replace("e[j] = v[j] - e[j];", "e[j] = e[j] - v[j];"),
        "decay_on_value_axis": src.replace("S[i * dv + j] *= a;", "S[i * dv + j] *= exp(g[j]);"),
        "query_for_key": src.replace("e[j] += S[i * dv + j] * k[i];", "e[j] += S[i * dv + j] * q[i];"),
    }


def _run_lib(path, q, k, v, g, b, S0):
    lib = ctypes.CDLL(path)
    d = ctypes.POINTER(ctypes.c_double)
    p64 = ctypes.POINTER(ctypes.c_int64)
    i64 = ctypes.c_int64
    lib.kda_oracle_forward.argtypes = [d, d, d, d, d, d, p64, i64, i64, i64, i64, d, d, i64, i64]
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    cu = np.arange(B + 1, dtype=np.int64) * T
    arrs = [np.ascontiguousarray(x, dtype=np.float64) for x in (q, k, v, g, b, S0)]
    out = np.zeros((B, T, H, dv)); sT = np.zeros((B, H, dk, dv))
    P = lambda a: a.ctypes.data_as(d)
    lib.kda_oracle_forward(*[P(a) for a in arrs], cu.ctypes.data_as(p64), B, H, dk, dv,
                           P(out), P(sT), 0, B * H)
    return out, sT


@pytest.mark.parametrize("name", ["decay_after_read", "readout_before_write", "no_beta_on_write",
                                  "delta_sign", "decay_on_value_axis", "query_for_key"])
def test_planted_mistake_is_caught(name, tmp_path):
    src = _mutants()[name]
    c = tmp_path / "mut.c"
    c.write_text(src)
    so = tmp_path / "mut.so"
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-std=c99", str(c), "-o", str(so), "-lm"])
    rng = np.random.default_rng(14)
    T, d = 12, 5
    q, k, v, g, b = rand_inputs(rng, T, d, d)
    S0 = 0.5 * rng.standard_normal((1, 1, d, d))
    out, sT = _run_lib(str(so), q, k, v, g, b, S0)
    ro, rs = brute_force(q[0, :, 0], k[0, :, 0], v[0, :, 0], g[0, :, 0], b[0, :, 0], S0[0, 0])
    err = max(rel_max_err(out[0, :, 0], ro), rel_max_err(sT[0, 0], rs))
    assert err > 1e-3, f"mutant {name} slipped through the brute-force pin (err {err})"
    # and the unmutated oracle passes the same check
    out, sT = oracle.forward(q, k, v, g, b, S0)
    assert max(rel_max_err(out[0, :, 0], ro), rel_max_err(sT[0, 0], rs)) < 1e-12
