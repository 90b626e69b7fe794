"""GPU parity over the magnitudes of v and the initial state, and at decay factors below the
fp32 normal range.

The method is linear in (V, S_0) for fixed (q, k, g, beta): nothing in it bounds the size of
the values or of the state, so a bf16 v and an fp32 S_0 may sit anywhere in their formats'
ranges.  The tensor-core kernel carries fp16 copies of S, Z and U; these tests check that it
meets the same bars at every scale 2^k of v and S_0 (k from -24, where fp16 alone would be
subnormal, to 20, where it would overflow), together and apart, and that for a common scale
its results are exactly 2^k times those at k = 0 (a power of two commutes with rounding).
The decode kernel (fp32 state) runs the same sweep.

The last test builds one 64-token chunk whose first 16-token sub-tile reaches the decay bound
(g = -5, cumulative -80) and whose later tokens decay by 0.25 each.  Keys of that sub-tile are
then scaled by e^80 inside the kernel while the factors that carry them to the last sub-tile
(e^-88) and to the chunk end (e^-92) lie below 2^-126; the true products (e^-8.25 and e^-12)
must survive.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from linear_attention_fwd_gb300 import inputs
from tests.helpers import rel_max_err
from tests.parity import TOL, check_prefill, compare_prefill, excess_err, f64

pytestmark = pytest.mark.gpu

SCALES = [(-24, -24), (-12, -12), (0, 0), (12, 12), (20, 20), (20, 0), (0, 20), (-24, 0), (0, -24)]


@pytest.fixture(scope="module")
def K(cuda_device):
    from linear_attention_fwd_gb300 import build, kda
    build.build()
    return kda


def scaled_prefill(kv, ks, seed=41):
    inp = inputs.make_prefill(batch=2, seqlen=300, heads=2, dk=128, dv=128, dtype=torch.bfloat16,
                              device="cuda", seed=seed, init_state=True)
    inp["v"] = (inp["v"].float() * 2.0 ** kv).to(torch.bfloat16)   # exact: a power of two
    inp["initial_state"] = inp["initial_state"] * 2.0 ** ks
    return inp


def run(K, inp, impl):
    out, sT = K.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                              inp["initial_state"], inp.get("cu_seqlens"), impl=impl)
    torch.cuda.synchronize()
    return out, sT


@pytest.mark.parametrize("kv,ks", SCALES)
def test_chunk_tc_scale_sweep(K, kv, ks):
    inp = scaled_prefill(kv, ks)
    out, sT = run(K, inp, "tc")
    assert torch.isfinite(out.float()).all() and torch.isfinite(sT).all()
    res = compare_prefill(inp, out, sT)
    check_prefill(res, torch.bfloat16)


@pytest.mark.parametrize("k", [-24, -12, 12, 20])
def test_chunk_tc_scales_exactly(K, k):
    """A common scale 2^k of v and S_0 scales outputs and final states by exactly 2^k."""
    base = scaled_prefill(0, 0)
    o0, s0 = run(K, base, "tc")
    inp = scaled_prefill(k, k)
    o1, s1 = run(K, inp, "tc")
    assert torch.equal(o1, (o0.float() * 2.0 ** k).to(torch.bfloat16))
    assert torch.equal(s1, s0 * 2.0 ** k)


@pytest.mark.parametrize("kv,ks", [(-24, -24), (20, 20), (20, 0), (0, -24)])
def test_chunk_simt_scale_sweep(K, kv, ks):
    inp = scaled_prefill(kv, ks, seed=42)
    out, sT = run(K, inp, "simt")
    check_prefill(compare_prefill(inp, out, sT), torch.bfloat16)


@pytest.mark.parametrize("kv,ks", SCALES)
def test_recurrent_step_scale_sweep(K, kv, ks):
    N, H, d, steps = 4, 2, 128, 3
    st = inputs.make_decode_state(num_slots=N, heads=H, dk=d, dv=d, device="cuda", seed=43) * 2.0 ** ks
    ins = inputs.make_decode_inputs(steps=steps, rows=N, heads=H, dk=d, dv=d, dtype=torch.bfloat16,
                                    device="cuda", seed=44)
    pool = f64(st).copy()
    for s in range(steps):
        a = {kk: ins[kk][s].contiguous() for kk in ins}
        a["v"] = (a["v"].float() * 2.0 ** kv).to(torch.bfloat16)
        o = K.kda_recurrent_step(a["q"], a["k"], a["v"], a["g"], a["beta"], st)
        ro = oracle.decode_step(a["q"], a["k"], a["v"], a["g"], a["beta"], pool)
        assert excess_err(f64(o), ro, torch.bfloat16) <= TOL[torch.bfloat16]
    assert rel_max_err(f64(st), pool) <= TOL[torch.bfloat16]


def test_decay_factors_below_fp32_normal_range(K):
    T, H, d = 64, 1, 128
    dev = "cuda"
    e0 = torch.zeros(d, device=dev)
    e0[0] = 1.0
    q = e0.expand(1, T, H, d).to(torch.bfloat16).contiguous()
    k = q.clone()
    v = torch.zeros(1, T, H, d, device=dev)
    v[0, 15] = 100.0
    g = torch.full((1, T, H, d), -0.25, device=dev)
    g[0, :16] = -5.0
    beta = torch.zeros(1, T, H, device=dev)
    beta[0, 15] = 1.0
    inp = dict(q=q, k=k, v=v.to(torch.bfloat16).contiguous(), g=g.to(torch.bfloat16).contiguous(),
               beta=beta.to(torch.bfloat16).contiguous(), initial_state=None)
    out, sT = run(K, inp, "tc")
    # closed form (every key the same unit vector, only token 15 writes): for r >= 15,
    # o_r = 100 e^{gamma_r - gamma_15} in every value channel; the final state holds
    # 100 e^{gamma_63 - gamma_15} = 100 e^-12 in its first row
    r = np.arange(T)
    ref = np.where(r >= 15, 100.0 * np.exp(-0.25 * np.maximum(r - 15, 0)), 0.0)
    got = f64(out)[0, :, 0, :]
    for j in (0, 37, 127):
        np.testing.assert_allclose(got[48:, j], ref[48:], rtol=2e-2)   # the e^-88 pair (3, 0)
        np.testing.assert_allclose(got[15:48, j], ref[15:48], rtol=2e-2)
    s_ref = 100.0 * math.exp(-12.0)
    np.testing.assert_allclose(f64(sT)[0, 0, 0, :], s_ref, rtol=2e-2)
    assert np.count_nonzero(f64(sT)[0, 0, 1:, :]) == 0
    # and the oracle agrees with the closed form, and the kernel with the oracle
    ro, rs = oracle.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"])
    np.testing.assert_allclose(ro[0, :, 0, 0], ref, rtol=1e-12, atol=1e-300)
    res = compare_prefill(inp, out, sT)
    check_prefill(res, torch.bfloat16)
