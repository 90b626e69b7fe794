"""The hand-worked fixtures in tests/golden/ against the oracle (CPU) and the CUDA path (GPU).

``kda_hand_worked.json`` holds a three-token, two-channel KDA recurrence and two rows of the
output gate, each value derived by hand from the update and read-out of
"はじめての自然言語処理 -- Kimi K3" (ogis-ri.co.jp), section 3.1, with the arithmetic written
beside it.  The oracle must reproduce them to fp64 rounding; the fp32 kernels must reproduce the
recurrence embedded in 64 and 128 channels (zero padding, no decay on the padded channels,
which then stay zero) to fp32 rounding.
"""
import json
import os
import subprocess

import numpy as np
import pytest

import oracle
from tests.test_oracle_pins import _mutants, _run_lib

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "kda_hand_worked.json")


@pytest.fixture(scope="module")
def fx():
    with open(GOLDEN, encoding="utf-8") as f:
        return json.load(f)


def _rec(fx):
    r = fx["recurrence"]
    a = {k: np.asarray(r[k], dtype=np.float64)
         for k in ("q", "k", "v", "g", "beta", "initial_state", "out", "final_state")}
    return a


def test_oracle_forward_matches_the_hand_worked_recurrence(fx):
    a = _rec(fx)
    out, sT = oracle.forward(a["q"][None, :, None], a["k"][None, :, None], a["v"][None, :, None],
                             a["g"][None, :, None], a["beta"][None, :, None],
                             a["initial_state"][None, None])
    np.testing.assert_allclose(out[0, :, 0], a["out"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(sT[0, 0], a["final_state"], rtol=0, atol=1e-13)


def test_oracle_decode_steps_match_the_hand_worked_recurrence(fx):
    a = _rec(fx)
    state = np.ascontiguousarray(a["initial_state"][None, None])
    for t in range(3):
        o = oracle.decode_step(a["q"][None, t, None], a["k"][None, t, None], a["v"][None, t, None],
                               a["g"][None, t, None], a["beta"][None, t, None], state)
        np.testing.assert_allclose(o[0, 0], a["out"][t], rtol=0, atol=1e-13)
    np.testing.assert_allclose(state[0, 0], a["final_state"], rtol=0, atol=1e-13)


def test_oracle_packed_copies_match_the_hand_worked_recurrence(fx):
    # the same sequence twice in one packed batch, each copy from its own initial state
    a = _rec(fx)
    cat = lambda x: np.concatenate([x, x])[None, :, None]
    s0 = np.stack([a["initial_state"], a["initial_state"]])[:, None]
    out, sT = oracle.forward(cat(a["q"]), cat(a["k"]), cat(a["v"]), cat(a["g"]), cat(a["beta"]),
                             s0, np.array([0, 3, 6]))
    np.testing.assert_allclose(out[0, :, 0], np.concatenate([a["out"], a["out"]]), rtol=0, atol=1e-13)
    for n in range(2):
        np.testing.assert_allclose(sT[n, 0], a["final_state"], rtol=0, atol=1e-13)


def test_oracle_gate_matches_the_hand_worked_rows(fx):
    gt = fx["gate"]
    y = oracle.gated_rmsnorm(np.asarray(gt["o"]), np.asarray(gt["z"]), np.asarray(gt["weight"]),
                             eps=0.0)
    np.testing.assert_allclose(y, np.asarray(gt["y"]), rtol=0, atol=1e-14)


def _embedded(a, d):
    """The two-channel example inside d channels: zero q, k, v, S0 and g on channels >= 2."""
    import torch
    T = a["q"].shape[0]
    out = {}
    for name in ("q", "k", "g"):
        x = np.zeros((1, T, 1, d))
        x[0, :, 0, :2] = a[name]
        out[name] = torch.tensor(x, dtype=torch.float32, device="cuda")
    v = np.zeros((1, T, 1, d))
    v[0, :, 0, :2] = a["v"]
    out["v"] = torch.tensor(v, dtype=torch.float32, device="cuda")
    out["beta"] = torch.tensor(a["beta"][None, :, None], dtype=torch.float32, device="cuda")
    s0 = np.zeros((1, 1, d, d))
    s0[0, 0, :2, :2] = a["initial_state"]
    out["s0"] = torch.tensor(s0, dtype=torch.float32, device="cuda")
    return out


@pytest.mark.gpu
@pytest.mark.parametrize("d", [64, 128])
def test_kernels_reproduce_the_hand_worked_recurrence(fx, d, cuda_device):
    import torch
    from linear_attention_fwd_gb300 import build, kda
    build.build()
    a = _rec(fx)
    e = _embedded(a, d)
    out, sT = kda.kda_chunk_fwd(e["q"], e["k"], e["v"], e["g"], e["beta"], e["s0"].clone())
    torch.cuda.synchronize()
    o = out.double().cpu().numpy()[0, :, 0]
    s = sT.double().cpu().numpy()[0, 0]
    np.testing.assert_allclose(o[:, :2], a["out"], rtol=0, atol=2e-6)
    np.testing.assert_allclose(s[:2, :2], a["final_state"], rtol=0, atol=2e-6)
    assert np.all(o[:, 2:] == 0.0) and np.all(s[2:, :] == 0.0) and np.all(s[:, 2:] == 0.0)

    state = e["s0"].clone()
    for t in range(3):
        ot = kda.kda_recurrent_step(e["q"][:, t], e["k"][:, t], e["v"][:, t], e["g"][:, t],
                                    e["beta"][:, t], state)
        torch.cuda.synchronize()
        np.testing.assert_allclose(ot.double().cpu().numpy()[0, 0, :2], a["out"][t], rtol=0, atol=2e-6)
    np.testing.assert_allclose(state.double().cpu().numpy()[0, 0, :2, :2], a["final_state"],
                               rtol=0, atol=2e-6)


@pytest.mark.parametrize("name", ["decay_after_read", "readout_before_write", "no_beta_on_write",
                                  "delta_sign", "decay_on_value_axis", "query_for_key"])
def test_planted_mistake_misses_the_hand_worked_values(fx, name, tmp_path):
    # the hand-worked values alone catch each planted mistake in the oracle source
    c = tmp_path / "mut.c"
    c.write_text(_mutants()[name])
    so = tmp_path / "mut.so"
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-std=c99", str(c), "-o", str(so), "-lm"])
    a = _rec(fx)
    out, sT = _run_lib(str(so), a["q"][None, :, None], a["k"][None, :, None], a["v"][None, :, None],
                       a["g"][None, :, None], a["beta"][None, :, None], a["initial_state"][None, None])
    err = max(np.abs(out[0, :, 0] - a["out"]).max(), np.abs(sT[0, 0] - a["final_state"]).max())
    assert err > 1e-2, f"mutant {name} reproduces the hand-worked values (err {err})"
