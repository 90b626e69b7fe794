"""GPU tests of kda_recurrent_steps (several decode tokens per row: speculative-decoding
verify and replay) through the C ABI.

The multi-token kernel keeps the fp32 state on chip between tokens; T single steps store
and reload it in fp32 (exactly), with the same arithmetic per token.  So a T-token call must
equal T calls of kda_recurrent_step bit for bit; against the fp64 oracle (the token
recurrence over the row's accepted prefix, from the row's state) the usual bars apply.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_fwd_gb300 import inputs
from tests.helpers import rel_max_err
from tests.parity import TOL, excess_err, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K(cuda_device):
    from linear_attention_fwd_gb300 import build, kda
    build.build()
    return kda


def _draft(T, N, H, d, dtype, seed):
    """Inputs of T draft tokens for N rows, laid out [N, T, H, d] (and [N, T, H] for beta)."""
    ins = inputs.make_decode_inputs(steps=T, rows=N, heads=H, dk=d, dv=d, dtype=dtype,
                                    device="cuda", seed=seed)
    return {kk: ins[kk].transpose(0, 1).contiguous() for kk in ins}


def _single_steps(K, a, state, idx, m):
    """Row n runs its first m[n] tokens through kda_recurrent_step; returns the outputs."""
    N, T = a["q"].shape[:2]
    outs = torch.zeros((N, T) + tuple(a["v"].shape[2:]), dtype=a["q"].dtype, device="cuda")
    for t in range(T):
        rows = [n for n in range(N) if m[n] > t]
        if not rows:
            continue
        sel = torch.tensor(rows, device="cuda")
        sl = {kk: a[kk][sel, t].contiguous() for kk in a}
        sub_idx = idx[sel].contiguous() if idx is not None else sel.to(torch.int32)
        o = K.kda_recurrent_step(sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"], state, sub_idx)
        outs[sel, t] = o
    return outs


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float32, 64), (torch.float32, 128)])
def test_steps_equal_single_steps_bit_for_bit(K, dtype, d):
    N, T, H, P = 5, 4, 3, 7
    a = _draft(T, N, H, d, dtype, seed=31)
    idx = torch.tensor([3, 0, 6, 1, 4], dtype=torch.int32, device="cuda")
    m = [4, 2, 0, 1, 3]
    num = torch.tensor(m, dtype=torch.int32, device="cuda")
    s_multi = inputs.make_decode_state(num_slots=P, heads=H, dk=d, dv=d, device="cuda", seed=32)
    s_single = s_multi.clone()
    o_multi = K.kda_recurrent_steps(a["q"], a["k"], a["v"], a["g"], a["beta"], s_multi, idx, num)
    o_single = _single_steps(K, a, s_single, idx, m)
    torch.cuda.synchronize()
    torch.testing.assert_close(s_multi, s_single, rtol=0, atol=0)
    torch.testing.assert_close(o_multi, o_single, rtol=0, atol=0)
    for n in range(N):   # tokens past the row's count are not written
        assert torch.all(o_multi[n, m[n]:] == 0)


@pytest.mark.parametrize("T", [8, 11, 17])
def test_steps_past_one_staging_group(K, T):
    """More draft tokens than the kernel stages at once (8): the groups chain through the
    on-chip state exactly like single steps, including a ragged last group."""
    dtype, d, N, H, P = torch.bfloat16, 128, 4, 2, 5
    a = _draft(T, N, H, d, dtype, seed=61 + T)
    idx = torch.tensor([2, 4, 0, 1], dtype=torch.int32, device="cuda")
    m = [T, T - 3, 9 if T > 9 else T, 1]
    num = torch.tensor(m, dtype=torch.int32, device="cuda")
    s_multi = inputs.make_decode_state(num_slots=P, heads=H, dk=d, dv=d, device="cuda", seed=62)
    s_single = s_multi.clone()
    o_multi = K.kda_recurrent_steps(a["q"], a["k"], a["v"], a["g"], a["beta"], s_multi, idx, num)
    o_single = _single_steps(K, a, s_single, idx, m)
    torch.cuda.synchronize()
    torch.testing.assert_close(s_multi, s_single, rtol=0, atol=0)
    torch.testing.assert_close(o_multi, o_single, rtol=0, atol=0)


def test_verify_leaves_the_state_and_replay_matches_the_oracle(K):
    """Speculative decoding: verify all T draft tokens (state untouched), then replay each
    row's accepted prefix into the state (no outputs)."""
    dtype, d, N, T, H, P = torch.bfloat16, 128, 6, 5, 2, 6
    a = _draft(T, N, H, d, dtype, seed=41)
    state = inputs.make_decode_state(num_slots=P, heads=H, dk=d, dv=d, device="cuda", seed=42)
    saved = state.clone()
    o = K.kda_recurrent_steps(a["q"], a["k"], a["v"], a["g"], a["beta"], state,
                              update_state=False)
    torch.cuda.synchronize()
    torch.testing.assert_close(state, saved, rtol=0, atol=0)
    accepted = [5, 0, 3, 1, 5, 2]
    r = K.kda_recurrent_steps(a["q"], a["k"], a["v"], a["g"], a["beta"], state, None,
                              torch.tensor(accepted, dtype=torch.int32, device="cuda"),
                              want_out=False)
    torch.cuda.synchronize()
    assert r is None
    for n in range(N):
        for h in range(H):
            sl = lambda t: t[n, :, h][None, :, None]   # noqa: E731 -- [1, T, 1, d]
            ro, _ = oracle.forward(sl(a["q"]), sl(a["k"]), sl(a["v"]), sl(a["g"]),
                                   a["beta"][n, :, h][None, :, None], saved[n, h][None, None])
            assert excess_err(f64(o[n, :, h]), ro[0, :, 0], dtype) <= TOL[dtype]
            m = accepted[n]
            if m == 0:
                torch.testing.assert_close(state[n, h], saved[n, h], rtol=0, atol=0)
                continue
            cut = lambda t: t[n, :m, h][None, :, None]   # noqa: E731
            _, rs = oracle.forward(cut(a["q"]), cut(a["k"]), cut(a["v"]), cut(a["g"]),
                                   a["beta"][n, :m, h][None, :, None], saved[n, h][None, None])
            assert rel_max_err(f64(state[n, h]), rs[0, 0]) <= TOL[dtype]


def test_steps_skip_rows_outside_the_pool_and_validate(K):
    d, H, T = 64, 2, 3
    a = _draft(T, 3, H, d, torch.float32, seed=51)
    state = inputs.make_decode_state(num_slots=2, heads=H, dk=d, dv=d, device="cuda", seed=52)
    ref = state.clone()
    out = torch.full((3, T, H, d), 7.0, device="cuda")
    idx = torch.tensor([5, 1, -2], dtype=torch.int32, device="cuda")
    K.kda_recurrent_steps(a["q"], a["k"], a["v"], a["g"], a["beta"], state, idx, out=out)
    torch.cuda.synchronize()
    assert torch.all(out[0] == 7.0) and torch.all(out[2] == 7.0)
    torch.testing.assert_close(state[0], ref[0], rtol=0, atol=0)
    assert not torch.equal(state[1], ref[1])
    with pytest.raises(K.KdaError):   # misaligned q
        qb = torch.empty(a["q"].numel() + 1, device="cuda")[1:].view_as(a["q"])
        K.kda_recurrent_steps(qb, a["k"], a["v"], a["g"], a["beta"], state, idx, out=out)
