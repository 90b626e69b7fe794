"""GPU parity of kda_chunk_fwd_gated (the KDA output gate fused into the output store)
against the oracle: oracle.gated_rmsnorm applied to the oracle's own fp64 forward outputs.
Covers the tensor-core kernel (bf16, d=128: fused into its output staging) and the SIMT
kernel plus the separate gate pass (fp32; bf16 d=64).

The bar (derived from the arithmetic; the forward's own bar is TOL * RMS(o) over the
stored-output rounding).  The gate normalises each row of o to unit RMS, so an error d in o
reaches y = o * rstd * w * sigmoid(z) as d * rstd * |w sigmoid| * (1 + |o_j| * rstd) to first
order (the second term is rstd's own change) -- large for the rare rows whose read-out is small.
So, elementwise, with eps_o = TOL * RMS(o) (+ the bf16 rounding of o for bf16 outputs, which
the forward's bar allows on top):
    |y - y_ref| <= eps_o * rstd_row * |w sigmoid(z)| * (1 + |o_j| rstd_row)
                   (+ for bf16: the rounding of y_ref and one ulp of y),
and, so that a systematic error cannot hide under that bound, the 99th percentile of
|y - y_ref| stays within TOL * RMS(y_ref).  On the rows where the normalisation does not
amplify (RMS(o_row) >= RMS(o): it multiplies an error in o by at most 1 / RMS(o)), the
forward's flat bar is held as well: the error beyond y's own storage rounding (and, for bf16,
beyond the rounding of o itself, half an ulp of |y| relative, which the separate gate pass
after the SIMT kernel reads back) stays within TOL * RMS(y_ref).  (Rows between 0.1 RMS(o)
and RMS(o) are amplified up to tenfold; on the bf16 tensor-core kernel their flat error
measured 0.023, above the bar, which is why the threshold is where it is; the value at 0.1 is
printed.)
"""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_fwd_gb300 import inputs
from tests.parity import TOL, f64, oracle_prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K(cuda_device):
    from linear_attention_fwd_gb300 import build, kda
    build.build()
    return kda


def _gate_inputs(inp, seed, with_weight=True):
    gen = torch.Generator(device="cuda").manual_seed(seed)
    v = inp["v"]
    z = (2.0 * torch.randn(v.shape, generator=gen, device="cuda")).to(v.dtype)
    w = (1.0 + 0.25 * torch.randn(v.shape[-1], generator=gen, device="cuda")) if with_weight else None
    return z, w


def _check(K, inp, heads, eps=1e-6, seed=0, with_weight=True):
    dtype = inp["q"].dtype
    z, w = _gate_inputs(inp, seed, with_weight)
    y, fs = K.kda_chunk_fwd_gated(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], z, w, eps,
                                  inp["initial_state"], inp["cu_seqlens"])
    # the plain call compared bit for bit runs the kernel the gated call runs (the library keeps
    # the gate on the SIMT kernel at d=64)
    impl = "tc" if (dtype == torch.bfloat16 and inp["q"].shape[-1] == 128) else "simt"
    _, fs_plain = K.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                  inp["initial_state"], inp["cu_seqlens"], impl=impl)
    torch.cuda.synchronize()
    torch.testing.assert_close(fs, fs_plain, rtol=0, atol=0)   # the gate touches only the outputs
    ro, _, heads = oracle_prefill(inp, heads)
    zz = f64(z[:, :, heads])
    ww = np.ones(ro.shape[-1]) if w is None else f64(w)
    ry = oracle.gated_rmsnorm(ro, zz, ww, eps)
    gy = f64(y[:, :, heads])
    tol = TOL[dtype]
    rms_o = np.sqrt(np.mean(ro ** 2))
    rstd = (1.0 / np.sqrt(np.mean(ro ** 2, axis=-1) + eps))[..., None]
    gain = np.abs(ww / (1.0 + np.exp(-zz)))
    eps_o = tol * rms_o + (2.0 ** -8 * np.abs(ro) if dtype == torch.bfloat16 else 0.0)
    bound = eps_o * rstd * gain * (1.0 + np.abs(ro) * rstd)
    if dtype == torch.bfloat16:
        stor = torch.from_numpy(np.ascontiguousarray(ry)).to(torch.bfloat16).double().numpy()
        bound = bound + np.abs(stor - ry) + np.abs(ry) * 2.0 ** -8
    err = np.abs(gy - ry)
    assert np.all(err <= bound), float(np.max(err / bound))
    rms_y = np.sqrt(np.mean(ry ** 2))
    assert np.quantile(err, 0.99) <= tol * rms_y
    row_rms = np.sqrt(np.mean(ro ** 2, axis=-1))
    stor_y = np.abs(torch.from_numpy(np.ascontiguousarray(ry)).to(dtype).double().numpy() - ry)
    if dtype == torch.bfloat16:
        stor_y = stor_y + 2.0 ** -9 * np.abs(ry)
    flat = {th: float(np.max((err - stor_y)[row_rms >= th * rms_o])) / rms_y for th in (0.1, 1.0)}
    print(f"gate flat error beyond storage, rows with RMS(o_row) >= 0.1 / 1 RMS(o): "
          f"{flat[0.1]:.4f} / {flat[1.0]:.4f}")
    assert flat[1.0] <= tol, flat


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float32, 64),
                                     (torch.float32, 128), (torch.bfloat16, 64)])
def test_gated_dense(K, dtype, d):
    inp = inputs.make_prefill(batch=2, seqlen=200, heads=3, dk=d, dv=d, dtype=dtype, device="cuda",
                              seed=71, init_state=True)
    _check(K, inp, heads=None, seed=72)


def test_gated_varlen_tc_without_weight(K):
    inp = inputs.make_prefill(batch=1, seqlen=0, heads=4, dk=128, dv=128, dtype=torch.bfloat16,
                              device="cuda", seed=73, init_state=True, lengths=[130, 1, 64, 257])
    _check(K, inp, heads=None, seed=74, with_weight=False, eps=1e-5)


def test_gated_full_size_sampled_heads(K):
    inp = inputs.make_workload("prefill_b4_h32_t8192", device="cuda")
    _check(K, inp, heads=[0, 17], seed=75)


def test_gated_validation(K):
    inp = inputs.make_prefill(batch=1, seqlen=64, heads=2, dk=128, dv=128, dtype=torch.bfloat16,
                              device="cuda", seed=76)
    z, w = _gate_inputs(inp, 77)
    with pytest.raises(K.KdaError):
        K.kda_chunk_fwd_gated(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], z, w, -1.0)
    with pytest.raises(K.KdaError):
        K.kda_chunk_fwd_gated(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], z, w, float("nan"))
