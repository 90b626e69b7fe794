"""GPU parity of the two-pass chunk forward (kda_chunk_fwd_ws: the state-independent chunk
work for all chunks first, into a caller-owned workspace, then the state chain) against the
fp64 oracle, through the C ABI; and its agreement with the one-pass tensor-core kernel.

Cases: dense edge lengths (1 .. 300 tokens), packed sequences with empty and one-token members
and initial states, 600 packed sequences, every g = -5, in-place resume split off a chunk
boundary, v and the initial state scaled by 2^k, a chunk whose decay factors fall below the
fp32 normal range, a workspace written over garbage, and the full-size workloads on sampled
heads.  Bars as everywhere: 2e-2 of RMS on the outputs beyond their own bf16 rounding and on
the fp32 states.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from linear_attention_fwd_gb300 import inputs
from tests.helpers import rel_max_err
from tests.parity import TOL, check_prefill, compare_prefill, f64

pytestmark = pytest.mark.gpu
BF = torch.bfloat16


@pytest.fixture(scope="module")
def K(cuda_device):
    from linear_attention_fwd_gb300 import build, kda
    build.build()
    return kda


def run(K, inp, impl="two_pass", **kw):
    out, sT = K.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                              inp.get("initial_state"), inp.get("cu_seqlens"), impl=impl, **kw)
    torch.cuda.synchronize()
    return out, sT


@pytest.mark.parametrize("T", [1, 15, 16, 17, 63, 64, 65, 127, 300])
def test_dense_edge_lengths(K, T):
    inp = inputs.make_prefill(batch=2, seqlen=T, heads=3, dk=128, dv=128, dtype=BF,
                              device="cuda", seed=2000 + T, init_state=True)
    out, sT = run(K, inp)
    check_prefill(compare_prefill(inp, out, sT), BF)


def test_agrees_with_one_pass_kernel(K):
    inp = inputs.make_prefill(batch=2, seqlen=700, heads=4, dk=128, dv=128, dtype=BF,
                              device="cuda", seed=2101, init_state=True)
    o1, s1 = run(K, inp, impl="tc")
    o2, s2 = run(K, inp)
    assert rel_max_err(f64(o2), f64(o1)) <= TOL[BF]
    assert rel_max_err(f64(s2), f64(s1)) <= TOL[BF]


def test_varlen_with_short_and_empty_sequences(K):
    inp = inputs.make_prefill(batch=1, seqlen=0, heads=2, dk=128, dv=128, dtype=BF, device="cuda",
                              seed=2102, init_state=True, lengths=[1, 64, 0, 130, 17, 1, 65, 0])
    out, sT = run(K, inp)
    check_prefill(compare_prefill(inp, out, sT), BF)
    torch.testing.assert_close(sT[2], inp["initial_state"][2], rtol=0, atol=0)
    torch.testing.assert_close(sT[7], inp["initial_state"][7], rtol=0, atol=0)


def test_more_packed_sequences_than_threads(K):
    rng = np.random.default_rng(2103)
    lengths = [int(x) for x in rng.integers(0, 151, 600)]
    lengths[:4] = [0, 1, 64, 65]
    inp = inputs.make_prefill(batch=1, seqlen=0, heads=2, dk=128, dv=128, dtype=BF, device="cuda",
                              seed=2104, init_state=True, lengths=lengths)
    out, sT = run(K, inp)
    check_prefill(compare_prefill(inp, out, sT), BF)


def test_decay_bound_extreme(K):
    inp = inputs.make_prefill(batch=1, seqlen=512, heads=2, dk=128, dv=128, dtype=BF, device="cuda",
                              seed=2105, g_mode="near_bound", init_state=True)
    assert torch.all(inp["g"] == -5.0)
    out, sT = run(K, inp)
    check_prefill(compare_prefill(inp, out, sT), BF)


def test_inplace_resume(K):
    inp = inputs.make_prefill(batch=2, seqlen=320, heads=2, dk=128, dv=128, dtype=BF, device="cuda",
                              seed=2106, init_state=True)
    t0 = 130
    first = {n: inp[n][:, :t0].contiguous() for n in ("q", "k", "v", "g", "beta")}
    second = {n: inp[n][:, t0:].contiguous() for n in ("q", "k", "v", "g", "beta")}
    state = inp["initial_state"].clone()
    o1, _ = K.kda_chunk_fwd(first["q"], first["k"], first["v"], first["g"], first["beta"], state,
                            final_state=state, impl="two_pass")
    o2, _ = K.kda_chunk_fwd(second["q"], second["k"], second["v"], second["g"], second["beta"], state,
                            final_state=state, impl="two_pass")
    torch.cuda.synchronize()
    check_prefill(compare_prefill(inp, torch.cat([o1, o2], 1), state), BF)


@pytest.mark.parametrize("kv,ks", [(-24, -24), (20, 20), (20, 0), (0, -24)])
def test_input_scales(K, kv, ks):
    inp = inputs.make_prefill(batch=2, seqlen=300, heads=2, dk=128, dv=128, dtype=BF, device="cuda",
                              seed=2107, init_state=True)
    inp["v"] = (inp["v"].float() * 2.0 ** kv).to(BF)
    inp["initial_state"] = inp["initial_state"] * 2.0 ** ks
    out, sT = run(K, inp)
    assert torch.isfinite(out.float()).all() and torch.isfinite(sT).all()
    check_prefill(compare_prefill(inp, out, sT), BF)


def test_decay_factors_below_fp32_normal_range(K):
    T, H, d = 64, 1, 128
    e0 = torch.zeros(d, device="cuda")
    e0[0] = 1.0
    q = e0.expand(1, T, H, d).to(BF).contiguous()
    v = torch.zeros(1, T, H, d, device="cuda")
    v[0, 15] = 100.0
    g = torch.full((1, T, H, d), -0.25, device="cuda")
    g[0, :16] = -5.0
    beta = torch.zeros(1, T, H, device="cuda")
    beta[0, 15] = 1.0
    inp = dict(q=q, k=q.clone(), v=v.to(BF).contiguous(), g=g.to(BF).contiguous(),
               beta=beta.to(BF).contiguous(), initial_state=None)
    out, sT = run(K, inp)
    r = np.arange(T)
    ref = np.where(r >= 15, 100.0 * np.exp(-0.25 * np.maximum(r - 15, 0)), 0.0)
    got = f64(out)[0, :, 0, :]
    for j in (0, 37, 127):
        np.testing.assert_allclose(got[15:, j], ref[15:], rtol=2e-2)
    np.testing.assert_allclose(f64(sT)[0, 0, 0, :], 100.0 * math.exp(-12.0), rtol=2e-2)


def test_workspace_contents_do_not_matter(K):
    inp = inputs.make_prefill(batch=1, seqlen=200, heads=2, dk=128, dv=128, dtype=BF, device="cuda",
                              seed=2108, init_state=True)
    need = K.kda_chunk_fwd_workspace_bytes(inp["q"], inp["v"])
    ws = torch.full((need,), 0xAB, dtype=torch.uint8, device="cuda")
    o1, s1 = run(K, inp, workspace=ws)
    ws.fill_(0x7F)
    o2, s2 = run(K, inp, workspace=ws)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)
    with pytest.raises(K.KdaError) as e:
        run(K, inp, workspace=ws[:need - 1024])
    assert e.value.status == K.KDA_ERR_WORKSPACE


@pytest.mark.parametrize("name,heads", [("prefill_b4_h32_t8192", [0, 5, 13, 31]),
                                        ("long_h64_t65536", [0, 37, 63]),
                                        ("varlen_16seq_1m", [3, 30])])
def test_full_size(K, name, heads):
    inp = inputs.make_workload(name, device="cuda")
    out, sT = run(K, inp)
    assert torch.isfinite(out).all() and torch.isfinite(sT).all()
    res = compare_prefill(inp, out, sT, heads=heads)
    print(name, res)
    check_prefill(res, BF)
