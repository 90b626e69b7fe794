"""GPU parity on the degenerate cases of the method, for both chunk kernels (tensor-core bf16
d=128, SIMT fp32 d=64 and d=128) and the decode kernel.

* beta = 0: nothing is written, the state only decays: S_t = Diag(exp sum_{s<=t} g_s) S_0 and
  o_t = S_t^T q_t, checked against that closed form directly (not through the oracle).
* g = 0: no decay anywhere (every sub-tile factor is 1), against the oracle.
* beta = 1 with each key repeated on the next token: A has entries up to 1 next to its diagonal
  (the second write mostly replaces the first), against the oracle.
* q = 0 gives outputs that are exactly zero; v = 0 with S_0 = 0 gives outputs and states that
  are exactly zero.
"""
import numpy as np
import pytest
import torch

from linear_attention_fwd_gb300 import inputs
from tests.helpers import rel_max_err
from tests.parity import TOL, check_prefill, compare_prefill, excess_err, f64

pytestmark = pytest.mark.gpu

KERNELS = [("tc", torch.bfloat16, 128), ("simt", torch.float32, 64), ("simt", torch.float32, 128)]


@pytest.fixture(scope="module")
def K(cuda_device):
    from linear_attention_fwd_gb300 import build, kda
    build.build()
    return kda


def make(dtype, d, T=300, B=2, H=2, seed=401, **kw):
    return inputs.make_prefill(batch=B, seqlen=T, heads=H, dk=d, dv=d, dtype=dtype,
                               device="cuda", seed=seed, init_state=True, **kw)


def run(K, inp, impl):
    out, sT = K.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                              inp["initial_state"], inp.get("cu_seqlens"), impl=impl)
    torch.cuda.synchronize()
    return out, sT


@pytest.mark.parametrize("impl,dtype,d", KERNELS)
def test_beta_zero_is_pure_decay(K, impl, dtype, d):
    inp = make(dtype, d, seed=402)
    inp["beta"] = torch.zeros_like(inp["beta"])
    out, sT = run(K, inp, impl)
    q, g, s0 = f64(inp["q"]), f64(inp["g"]), f64(inp["initial_state"])
    cg = np.cumsum(g, axis=1)                                  # [B, T, H, dk]
    ref = np.einsum("bthi,bhij->bthj", q * np.exp(cg), s0)     # o_t = (Diag(e^cg) S0)^T q_t
    ref_s = np.exp(cg[:, -1])[..., None] * s0                  # [B, H, dk, dv]
    assert rel_max_err(f64(sT), ref_s) <= TOL[dtype]
    if dtype == torch.bfloat16:
        assert excess_err(f64(out), ref, dtype) <= TOL[dtype]
    else:
        assert rel_max_err(f64(out), ref) <= TOL[dtype]


@pytest.mark.parametrize("impl,dtype,d", KERNELS)
def test_no_decay(K, impl, dtype, d):
    inp = make(dtype, d, T=700, seed=403, g_mode="zero")
    out, sT = run(K, inp, impl)
    check_prefill(compare_prefill(inp, out, sT), dtype)


@pytest.mark.parametrize("impl,dtype,d", KERNELS)
def test_repeated_keys_with_unit_beta(K, impl, dtype, d):
    inp = make(dtype, d, T=260, seed=404)
    k = inp["k"].clone()
    k[:, 1::2] = k[:, 0::2][:, : k[:, 1::2].shape[1]]           # token 2m+1 repeats token 2m's key
    inp["k"] = k
    inp["beta"] = torch.ones_like(inp["beta"])
    out, sT = run(K, inp, impl)
    check_prefill(compare_prefill(inp, out, sT), dtype)


@pytest.mark.parametrize("impl,dtype,d", KERNELS)
def test_zero_query_and_zero_values(K, impl, dtype, d):
    inp = make(dtype, d, T=200, seed=405)
    inp["q"] = torch.zeros_like(inp["q"])
    out, _ = run(K, inp, impl)
    assert torch.count_nonzero(out) == 0
    inp = make(dtype, d, T=200, seed=406)
    inp["v"] = torch.zeros_like(inp["v"])
    inp["initial_state"] = torch.zeros_like(inp["initial_state"])
    out, sT = run(K, inp, impl)
    assert torch.count_nonzero(out) == 0 and torch.count_nonzero(sT) == 0


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float32, 64)])
def test_decode_beta_zero_is_pure_decay(K, dtype, d):
    st = inputs.make_decode_state(num_slots=8, heads=2, dk=d, dv=d, device="cuda", seed=407)
    di = inputs.make_decode_inputs(steps=1, rows=8, heads=2, dk=d, dv=d, dtype=dtype,
                                   device="cuda", seed=408)
    s0 = f64(st).copy()
    beta = torch.zeros_like(di["beta"][0])
    out = K.kda_recurrent_step(di["q"][0], di["k"][0], di["v"][0], di["g"][0], beta, st)
    torch.cuda.synchronize()
    ref_s = np.exp(f64(di["g"][0]))[..., None] * s0
    ref_o = np.einsum("nhi,nhij->nhj", f64(di["q"][0]), ref_s)
    assert rel_max_err(f64(st), ref_s) <= TOL[dtype]
    if dtype == torch.bfloat16:
        assert excess_err(f64(out), ref_o, dtype) <= TOL[dtype]
    else:
        assert rel_max_err(f64(out), ref_o) <= TOL[dtype]
