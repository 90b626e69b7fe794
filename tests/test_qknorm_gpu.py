"""GPU parity of the fused q/k L2 normalisation: kda_chunk_fwd_qknorm and
kda_recurrent_step_qknorm against the fp64 oracle.

The method reads q and k after L2 normalisation ("はじめての自然言語処理 -- Kimi K3",
section 3.1, the read-out paragraph).  The calls here get raw q and k (N(0, 1) entries,
norms near sqrt(dk)); the oracle normalises the same values in fp64 (the library keeps the
normalised rows in fp32, unrounded) and runs the recurrence on them.  Bars as for the plain
forward.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_fwd_gb300 import inputs
from tests.helpers import rel_max_err
from tests.parity import TOL, check_prefill, compare_prefill, excess_err, f64

pytestmark = pytest.mark.gpu

EPS = 1e-6


@pytest.fixture(scope="module")
def K(cuda_device):
    from linear_attention_fwd_gb300 import build, kda
    build.build()
    return kda


def normalised(inp, eps):
    """The inputs with q and k as the oracle's normalised rows (fp64)."""
    out = dict(inp)
    out["q"] = oracle.l2norm_rows(inp["q"], eps)
    out["k"] = oracle.l2norm_rows(inp["k"], eps)
    return out


def run(K, inp, eps=EPS):
    return K.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                           inp.get("initial_state"), inp.get("cu_seqlens"), qk_eps=eps)


@pytest.mark.parametrize("T", [1, 17, 64, 300])
@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.bfloat16, 64),
                                     (torch.float32, 64), (torch.float32, 128)])
def test_dense(K, T, dtype, d):
    inp = inputs.make_prefill(batch=2, seqlen=T, heads=3, dk=d, dv=d, dtype=dtype, device="cuda",
                              seed=4000 + T + d, init_state=True, raw_qk=True)
    out, sT = run(K, inp)
    check_prefill(compare_prefill(normalised(inp, EPS), out, sT), dtype)


def test_long_sequences_split_between_ctas(K):
    # two units of 96 chunks: the balanced schedule splits each between many CTAs, whose
    # pieces start from a warm-up over earlier chunks (the bound it uses sees normalised keys)
    inp = inputs.make_prefill(batch=1, seqlen=96 * 64 + 5, heads=2, dk=128, dv=128,
                              dtype=torch.bfloat16, device="cuda", seed=4101, raw_qk=True)
    out, sT = run(K, inp)
    check_prefill(compare_prefill(normalised(inp, EPS), out, sT), torch.bfloat16)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_packed_with_initial_states(K, dtype):
    inp = inputs.make_prefill(batch=1, seqlen=0, heads=2, dk=128, dv=128, dtype=dtype,
                              device="cuda", seed=4202, init_state=True, raw_qk=True,
                              lengths=[1, 63, 64, 65, 0, 200, 7])
    out, sT = run(K, inp)
    check_prefill(compare_prefill(normalised(inp, EPS), out, sT), dtype)


def test_inputs_in_memory_are_not_modified(K):
    inp = inputs.make_prefill(batch=2, seqlen=130, heads=2, dk=128, dv=128, dtype=torch.bfloat16,
                              device="cuda", seed=4303, raw_qk=True)
    q0, k0 = inp["q"].clone(), inp["k"].clone()
    run(K, inp)
    torch.cuda.synchronize()
    assert torch.equal(inp["q"], q0) and torch.equal(inp["k"], k0)


def test_zero_rows_stay_zero_with_eps_zero(K):
    # |x|^2 + eps = 0: the row stays zero rather than 0/0; nothing turns NaN
    inp = inputs.make_prefill(batch=1, seqlen=100, heads=2, dk=128, dv=128, dtype=torch.bfloat16,
                              device="cuda", seed=4404, raw_qk=True)
    inp["q"][0, 10] = 0
    inp["k"][0, 40:45] = 0
    out, sT = run(K, inp, eps=0.0)
    assert torch.isfinite(out.float()).all() and torch.isfinite(sT).all()
    check_prefill(compare_prefill(normalised(inp, 0.0), out, sT), torch.bfloat16)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_scale_invariance(K, dtype):
    # q and k scaled by 2^3 and 2^-5 (exact in both dtypes): with eps = 0 the normalised rows
    # are the same up to the approximate reciprocal square root, so the results agree far
    # inside the parity bar
    inp = inputs.make_prefill(batch=2, seqlen=150, heads=2, dk=128, dv=128, dtype=dtype,
                              device="cuda", seed=4505, raw_qk=True)
    o1, s1 = run(K, inp, eps=0.0)
    inp2 = dict(inp, q=inp["q"] * 8, k=inp["k"] / 32)
    o2, s2 = run(K, inp2, eps=0.0)
    assert rel_max_err(f64(s2), f64(s1)) < 1e-5
    assert excess_err(f64(o2), f64(o1), dtype) < 1e-3


def test_bad_eps_rejected(K):
    inp = inputs.make_prefill(batch=1, seqlen=8, heads=1, dk=128, dv=128, dtype=torch.bfloat16,
                              device="cuda", seed=1, raw_qk=True)
    for bad in (-1.0, float("nan"), float("inf")):
        with pytest.raises(K.KdaError) as e:
            run(K, inp, eps=bad)
        assert e.value.status == K.KDA_ERR_SHAPE


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float32, 64)])
def test_recurrent_step(K, dtype, d):
    N, H, P, steps = 5, 3, 7, 4
    st = inputs.make_decode_state(num_slots=P, heads=H, dk=d, dv=d, device="cuda", seed=41)
    ins = inputs.make_decode_inputs(steps=steps, rows=N, heads=H, dk=d, dv=d, dtype=dtype,
                                    device="cuda", seed=42, raw_qk=True)
    idx = torch.tensor([3, 0, 6, 2, 5], dtype=torch.int32, device="cuda")
    pool = f64(st).copy()
    for s in range(steps):
        a = {kk: ins[kk][s].contiguous() for kk in ins}
        o = K.kda_recurrent_step(a["q"], a["k"], a["v"], a["g"], a["beta"], st, idx, qk_eps=EPS)
        ro = oracle.decode_step(oracle.l2norm_rows(a["q"], EPS), oracle.l2norm_rows(a["k"], EPS),
                                a["v"], a["g"], a["beta"], pool, idx.cpu())
        assert excess_err(f64(o), ro, dtype) <= TOL[dtype]
    assert rel_max_err(f64(st), pool) <= TOL[dtype]


def test_recurrent_step_equals_one_token_prefill(K):
    d, H, N = 128, 2, 4
    inp = inputs.make_prefill(batch=N, seqlen=1, heads=H, dk=d, dv=d, dtype=torch.float32,
                              device="cuda", seed=4606, init_state=True, raw_qk=True)
    o1, s1 = run(K, inp)
    st = inp["initial_state"].clone()
    o2 = K.kda_recurrent_step(inp["q"][:, 0].contiguous(), inp["k"][:, 0].contiguous(),
                              inp["v"][:, 0].contiguous(), inp["g"][:, 0].contiguous(),
                              inp["beta"][:, 0].contiguous(), st, qk_eps=EPS)
    torch.testing.assert_close(o2, o1[:, 0], rtol=1e-5, atol=1e-5)
    torch.testing.assert_close(st, s1, rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float32, 64)])
def test_recurrent_steps_verify_and_replay(K, dtype, d):
    # several tokens per row with the normalisation: equal bit for bit to the same tokens run
    # one kda_recurrent_step_qknorm call at a time, and within the bars of the oracle; a verify
    # call (update_state off) leaves the state untouched
    N, T, H, P = 4, 5, 2, 6
    ins = inputs.make_decode_inputs(steps=T, rows=N, heads=H, dk=d, dv=d, dtype=dtype,
                                    device="cuda", seed=43, raw_qk=True)
    a = {kk: ins[kk].transpose(0, 1).contiguous() for kk in ins}
    idx = torch.tensor([5, 0, 3, 1], dtype=torch.int32, device="cuda")
    m = [5, 3, 0, 2]
    num = torch.tensor(m, dtype=torch.int32, device="cuda")
    s0 = inputs.make_decode_state(num_slots=P, heads=H, dk=d, dv=d, device="cuda", seed=44)
    s_ver = s0.clone()
    K.kda_recurrent_steps(a["q"], a["k"], a["v"], a["g"], a["beta"], s_ver, idx, num,
                          update_state=False, qk_eps=EPS)
    torch.cuda.synchronize()
    assert torch.equal(s_ver, s0)
    s_multi = s0.clone()
    o_multi = K.kda_recurrent_steps(a["q"], a["k"], a["v"], a["g"], a["beta"], s_multi, idx, num,
                                    qk_eps=EPS)
    s_single = s0.clone()
    pool = f64(s0).copy()
    for t in range(T):
        rows = [n for n in range(N) if m[n] > t]
        sel = torch.tensor(rows, device="cuda")
        sl = {kk: a[kk][sel, t].contiguous() for kk in a}
        o = K.kda_recurrent_step(sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"], s_single,
                                 idx[sel].contiguous(), qk_eps=EPS)
        assert torch.equal(o, o_multi[sel, t])
        ro = oracle.decode_step(oracle.l2norm_rows(sl["q"], EPS), oracle.l2norm_rows(sl["k"], EPS),
                                sl["v"], sl["g"], sl["beta"], pool, idx[sel].cpu())
        assert excess_err(f64(o), ro, dtype) <= TOL[dtype]
    torch.cuda.synchronize()
    assert torch.equal(s_multi, s_single)
    assert rel_max_err(f64(s_multi), pool) <= TOL[dtype]


def test_in_place_resume_and_many_packed_units(K):
    # the one-CTA-per-unit instantiation of the tensor-core kernel with the normalisation: an
    # in-place resume (the initial state buffer is also the final one), and more packed units
    # than twice the SMs (one CTA each, longest first)
    inp = inputs.make_prefill(batch=2, seqlen=300, heads=3, dk=128, dv=128, dtype=torch.bfloat16,
                              device="cuda", seed=4707, init_state=True, raw_qk=True)
    ref = normalised(inp, EPS)
    ref["initial_state"] = inp["initial_state"].clone()
    st = inp["initial_state"]
    out, sT = K.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], st, None,
                              final_state=st, qk_eps=EPS)
    check_prefill(compare_prefill(ref, out, sT), torch.bfloat16)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    nseq = sms + 8   # x 2 heads: more than twice the SMs
    lengths = [1 + (37 * i) % 150 for i in range(nseq)]
    inp = inputs.make_prefill(batch=1, seqlen=0, heads=2, dk=128, dv=128, dtype=torch.bfloat16,
                              device="cuda", seed=4708, init_state=True, raw_qk=True, lengths=lengths)
    out, sT = run(K, inp)
    check_prefill(compare_prefill(normalised(inp, EPS), out, sT), torch.bfloat16)
