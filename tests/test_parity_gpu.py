"""GPU parity: libkda (through its C ABI) against the fp64 oracle.

Every case feeds both sides the same seeded inputs; the oracle gets the exact
rounded values the GPU saw.  Bars: max |err| / RMS(ref) <= 1e-4 (fp32 inputs)
and <= 2e-2 (bf16 inputs, fp32 state), for both the outputs and the final
states.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_fwd_gb300 import inputs
from tests.helpers import rel_max_err
from tests.parity import TOL, check_prefill, compare_prefill, excess_err, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K(cuda_device):
    from linear_attention_fwd_gb300 import build, kda
    build.build()
    return kda


def impls_for(K, dtype, d):
    """Kernels that can run this shape: always the SIMT kernel, plus the
    tensor-core kernel where the library selects it."""
    out = ["simt"]
    probe_q = torch.empty((1, 1, 1, d), dtype=dtype, device="cuda")
    probe_v = torch.empty((1, 1, 1, d), dtype=dtype, device="cuda")
    if K.kda_chunk_fwd_selected_impl(probe_q, probe_v) == "tc":
        out.append("tc")
    return out


def run(K, inp, impl="auto", with_state=True):
    return K.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                           inp.get("initial_state"), inp.get("cu_seqlens"),
                           output_final_state=with_state, impl=impl)


def check(res, dtype):
    check_prefill(res, dtype)


# --------------------------------------------------------------------------- small, exhaustive
def test_tiny_fp32_workload(K):
    """B=1 H=2 T=256 dk=dv=64 fp32 (the tiny fp32 workload), full parity."""
    inp = inputs.make_workload("tiny_fp32", device="cuda")
    out, sT = run(K, inp)
    check(compare_prefill(inp, out, sT), torch.float32)


@pytest.mark.parametrize("T", [1, 15, 16, 17, 63, 64, 65, 127, 300])
@pytest.mark.parametrize("dtype,d", [(torch.float32, 64), (torch.float32, 128),
                                     (torch.bfloat16, 128), (torch.bfloat16, 64)])
def test_dense_edge_lengths(K, T, dtype, d):
    for impl in impls_for(K, dtype, d):
        inp = inputs.make_prefill(batch=2, seqlen=T, heads=3, dk=d, dv=d, dtype=dtype,
                                  device="cuda", seed=1000 + T, init_state=True)
        out, sT = run(K, inp, impl)
        check(compare_prefill(inp, out, sT), dtype)


@pytest.mark.parametrize("dk,dv", [(64, 128), (128, 64)])
def test_rectangular_heads(K, dk, dv):
    inp = inputs.make_prefill(batch=1, seqlen=130, heads=2, dk=dk, dv=dv, dtype=torch.float32,
                              device="cuda", seed=5, init_state=True)
    out, sT = run(K, inp)
    check(compare_prefill(inp, out, sT), torch.float32)


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64)])
def test_narrow_heads_on_the_tensor_cores(K, dk, dv):
    # a 64-wide head runs on the tensor-core kernel at 128 channels, the missing ones read as
    # zeros by the TMA; outputs and states of the real channels only, against the oracle; dense
    # (balanced schedule, sequences split between CTAs) and packed, with initial states
    assert K.kda_chunk_fwd_selected_impl(torch.empty((1, 1, 1, dk), dtype=torch.bfloat16, device="cuda"),
                                         torch.empty((1, 1, 1, dv), dtype=torch.bfloat16, device="cuda")) == "tc"
    inp = inputs.make_prefill(batch=2, seqlen=2000, heads=3, dk=dk, dv=dv, dtype=torch.bfloat16,
                              device="cuda", seed=6, init_state=True)
    out, sT = run(K, inp, "tc")
    assert out.shape[-1] == dv and sT.shape[-2:] == (dk, dv)
    check(compare_prefill(inp, out, sT), torch.bfloat16)
    inp = inputs.make_prefill(batch=1, seqlen=0, heads=2, dk=dk, dv=dv, dtype=torch.bfloat16,
                              device="cuda", seed=7, init_state=True, lengths=[1, 64, 0, 130, 17, 65])
    out, sT = run(K, inp, "tc")
    check(compare_prefill(inp, out, sT), torch.bfloat16)
    torch.testing.assert_close(sT[2], inp["initial_state"][2], rtol=0, atol=0)


@pytest.mark.parametrize("dtype,d", [(torch.float32, 64), (torch.bfloat16, 128)])
def test_varlen_with_short_and_empty_sequences(K, dtype, d):
    lengths = [1, 64, 0, 130, 17, 1, 65]
    for impl in impls_for(K, dtype, d):
        inp = inputs.make_prefill(batch=1, seqlen=0, heads=2, dk=d, dv=d, dtype=dtype,
                                  device="cuda", seed=77, init_state=True, lengths=lengths)
        out, sT = run(K, inp, impl)
        check(compare_prefill(inp, out, sT), dtype)
        # the empty sequence's final state is its initial state
        torch.testing.assert_close(sT[2], inp["initial_state"][2], rtol=0, atol=0)


def test_more_packed_sequences_than_threads(K):
    # 600 packed sequences (more than the 512 threads that rank them longest first, so they run
    # in their given order), lengths 0..150 with empty and one-token members, on both kernels
    rng = np.random.default_rng(12)
    lengths = [int(x) for x in rng.integers(0, 151, 600)]
    lengths[:4] = [0, 1, 64, 65]
    for dtype, d in [(torch.bfloat16, 128), (torch.float32, 64)]:
        for impl in impls_for(K, dtype, d):
            inp = inputs.make_prefill(batch=1, seqlen=0, heads=2, dk=d, dv=d, dtype=dtype,
                                      device="cuda", seed=78, init_state=True, lengths=lengths)
            out, sT = run(K, inp, impl)
            check(compare_prefill(inp, out, sT), dtype)
            torch.testing.assert_close(sT[0], inp["initial_state"][0], rtol=0, atol=0)


def test_decay_bound_extreme(K):
    """Every g = -5 (every 16-token sub-tile reaches cumulative log decay -80)."""
    for dtype, d in [(torch.float32, 64), (torch.bfloat16, 128)]:
        for impl in impls_for(K, dtype, d):
            inp = inputs.make_prefill(batch=1, seqlen=512, heads=2, dk=d, dv=d, dtype=dtype,
                                      device="cuda", seed=9, g_mode="near_bound", init_state=True)
            if dtype == torch.bfloat16:      # -5 + 0.01 U(0,1) rounds to exactly -5 in bf16
                assert torch.all(inp["g"] == -5.0)
            else:
                assert inp["g"].min() >= -5.0 and inp["g"].max() <= -4.99
            out, sT = run(K, inp, impl)
            res = compare_prefill(inp, out, sT)
            check(res, dtype)
            assert torch.isfinite(out).all() and torch.isfinite(sT).all()


def test_inplace_resume_and_split_invariance(K):
    """final_state may alias initial_state; [0,T) == [0,t0) then [t0,T) resumed."""
    d, dtype = 128, torch.bfloat16
    inp = inputs.make_prefill(batch=2, seqlen=320, heads=2, dk=d, dv=d, dtype=dtype,
                              device="cuda", seed=31, init_state=True)
    _, full_S = run(K, inp)
    t0 = 130     # not a chunk multiple
    per_token = ("q", "k", "v", "g", "beta")
    first = {n: inp[n][:, :t0].contiguous() for n in per_token}
    second = {n: inp[n][:, t0:].contiguous() for n in per_token}
    state = inp["initial_state"].clone()
    o1, _ = K.kda_chunk_fwd(first["q"], first["k"], first["v"], first["g"], first["beta"],
                            state, None, final_state=state)
    o2, _ = K.kda_chunk_fwd(second["q"], second["k"], second["v"], second["g"], second["beta"],
                            state, None, final_state=state)
    # the resumed run is chunked differently (a boundary at 130, not 128), so it
    # agrees with the one-shot run to the kernel's precision, not bit for bit
    assert rel_max_err(f64(state), f64(full_S)) <= TOL[dtype]
    # and both halves agree with the oracle run over the whole sequence
    check(compare_prefill(inp, torch.cat([o1, o2], 1), state), dtype)


def test_empty_input_copies_state(K):
    inp = inputs.make_prefill(batch=2, seqlen=0, heads=2, dk=64, dv=64, dtype=torch.float32,
                              device="cuda", seed=3, init_state=True)
    out, sT = run(K, inp)
    assert out.numel() == 0
    torch.testing.assert_close(sT, inp["initial_state"], rtol=0, atol=0)
    inp["initial_state"] = None
    _, sT = run(K, inp)
    assert torch.count_nonzero(sT) == 0


def test_outputs_do_not_spill_past_buffers(K):
    """Canary padding around out and final_state stays untouched."""
    d, T, H, B = 128, 70, 2, 1
    inp = inputs.make_prefill(batch=B, seqlen=T, heads=H, dk=d, dv=d, dtype=torch.bfloat16,
                              device="cuda", seed=4)
    pad = 4096
    ob = torch.full((B * T * H * d + 2 * pad,), 7.0, dtype=torch.bfloat16, device="cuda")
    sb = torch.full((B * H * d * d + 2 * pad,), 7.0, dtype=torch.float32, device="cuda")
    out = ob[pad:pad + B * T * H * d].view(B, T, H, d)
    fs = sb[pad:pad + B * H * d * d].view(B, H, d, d)
    K.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], None, None,
                    out=out, final_state=fs)
    torch.cuda.synchronize()
    assert torch.all(ob[:pad] == 7.0) and torch.all(ob[-pad:] == 7.0)
    assert torch.all(sb[:pad] == 7.0) and torch.all(sb[-pad:] == 7.0)


# --------------------------------------------------------------------------- decode
@pytest.mark.parametrize("dtype,d", [(torch.float32, 64), (torch.float32, 128),
                                     (torch.bfloat16, 128), (torch.bfloat16, 64)])
def test_recurrent_step_multi_step(K, dtype, d):
    N, H, P, steps = 6, 3, 9, 5
    st = inputs.make_decode_state(num_slots=P, heads=H, dk=d, dv=d, device="cuda", seed=11)
    ins = inputs.make_decode_inputs(steps=steps, rows=N, heads=H, dk=d, dv=d, dtype=dtype,
                                    device="cuda", seed=12)
    idx = torch.tensor([4, 0, 8, 2, 7, 5], dtype=torch.int32, device="cuda")
    pool = f64(st).copy()
    for s in range(steps):
        a = {kk: ins[kk][s].contiguous() for kk in ins}
        o = K.kda_recurrent_step(a["q"], a["k"], a["v"], a["g"], a["beta"], st, idx)
        ro = oracle.decode_step(a["q"], a["k"], a["v"], a["g"], a["beta"], pool, idx.cpu())
        assert excess_err(f64(o), ro, dtype) <= TOL[dtype]
    assert rel_max_err(f64(st), pool) <= TOL[dtype]
    torch.testing.assert_close(st[[1, 3, 6]], inputs.make_decode_state(
        num_slots=P, heads=H, dk=d, dv=d, device="cuda", seed=11)[[1, 3, 6]], rtol=0, atol=0)


def test_recurrent_step_skips_rows_outside_the_pool(K):
    d, H = 128, 2
    st = inputs.make_decode_state(num_slots=3, heads=H, dk=d, dv=d, device="cuda", seed=1)
    ref = st.clone()
    ins = inputs.make_decode_inputs(steps=1, rows=3, heads=H, dk=d, dv=d, dtype=torch.bfloat16,
                                    device="cuda", seed=2)
    a = {kk: ins[kk][0].contiguous() for kk in ins}
    out = torch.full((3, H, d), 5.0, dtype=torch.bfloat16, device="cuda")
    idx = torch.tensor([-1, 1, 3], dtype=torch.int32, device="cuda")
    K.kda_recurrent_step(a["q"], a["k"], a["v"], a["g"], a["beta"], st, idx, out=out)
    torch.cuda.synchronize()
    assert torch.all(out[0] == 5.0) and torch.all(out[2] == 5.0)
    torch.testing.assert_close(st[[0, 2]], ref[[0, 2]], rtol=0, atol=0)
    assert not torch.equal(st[1], ref[1])


def test_recurrent_step_equals_chunk_fwd_one_token(K):
    """A decode step and a one-token prefill compute the same thing."""
    d, H, N = 128, 4, 5
    inp = inputs.make_prefill(batch=N, seqlen=1, heads=H, dk=d, dv=d, dtype=torch.float32,
                              device="cuda", seed=21, init_state=True)
    o1, s1 = run(K, inp, "simt")
    st = inp["initial_state"].clone()
    o2 = K.kda_recurrent_step(inp["q"][:, 0].contiguous(), inp["k"][:, 0].contiguous(),
                              inp["v"][:, 0].contiguous(), inp["g"][:, 0].contiguous(),
                              inp["beta"][:, 0].contiguous(), st)
    torch.testing.assert_close(o2, o1[:, 0], rtol=1e-5, atol=1e-5)
    torch.testing.assert_close(st, s1, rtol=1e-5, atol=1e-5)
