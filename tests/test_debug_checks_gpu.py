"""The debug build's device-side input checks (libkda_debug.so, build.build(debug=True)).

The log decay's bound g in [-5, 0] ("はじめての自然言語処理 -- Kimi K3", section 3.1: g = -5
sigmoid(x)) and the packed offsets' order live in device memory, so the host cannot check
them. The debug build checks them on the device before each call and reports a failure through
kda_device_status as KDA_ERR_INPUT, without trapping. Checked here: a g of -6, of +0.25 and
NaN in one element each (chunk forward, both kernels, and decode); offsets that do not start at
0, that decrease, or that end before seqlen; clean inputs give KDA_OK and the same results as
the release library. The fixture switches the binding back to the release library afterwards.
"""
import pytest
import torch

from linear_attention_fwd_gb300 import inputs

pytestmark = pytest.mark.gpu
BF = torch.bfloat16


@pytest.fixture(scope="module")
def K(cuda_device):
    from linear_attention_fwd_gb300 import build, kda
    release = build.build()
    kda.use_library(release)
    assert kda.kda_debug_checks() == 0
    inp = inputs.make_prefill(batch=2, seqlen=300, heads=2, dk=128, dv=128, dtype=BF, device="cuda",
                              seed=501, init_state=True)
    ref = kda.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["initial_state"])
    torch.cuda.synchronize()
    kda.use_library(build.build(debug=True))
    assert kda.kda_debug_checks() == 3
    kda.ref = (inp, ref)
    yield kda
    kda.use_library(release)


def fwd(K, inp, g=None, cu=None, impl="auto"):
    out, sT = K.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"] if g is None else g, inp["beta"],
                              inp.get("initial_state"), inp.get("cu_seqlens") if cu is None else cu,
                              impl=impl)
    return out, sT


def test_clean_inputs_pass_and_match_the_release_build(K):
    inp, (ro, rs) = K.ref
    assert K.kda_device_status() == K.KDA_OK
    out, sT = fwd(K, inp)
    assert K.kda_device_status() == K.KDA_OK
    assert torch.equal(out, ro) and torch.equal(sT, rs)


@pytest.mark.parametrize("impl", ["tc", "simt"])
@pytest.mark.parametrize("bad", [-6.0, 0.25, float("nan")])
def test_decay_outside_the_bound_is_reported(K, impl, bad):
    inp, _ = K.ref
    if impl == "simt":
        inp = {k: (v.float() if v is not None and v.dtype == BF else v) for k, v in inp.items()}
    g = inp["g"].clone()
    g[1, 123, 1, 7] = bad
    fwd(K, inp, g=g, impl=impl)
    assert K.kda_device_status() == K.KDA_ERR_INPUT
    fwd(K, inp, impl=impl)
    assert K.kda_device_status() == K.KDA_OK   # read, cleared, and clean again


def test_decode_decay_outside_the_bound_is_reported(K):
    state = inputs.make_decode_state(num_slots=8, heads=2, dk=128, dv=128, device="cuda", seed=502)
    step = inputs.make_decode_inputs(steps=1, rows=8, heads=2, dk=128, dv=128, dtype=BF, device="cuda",
                                     seed=503)
    args = [step[n][0] for n in ("q", "k", "v", "g", "beta")]
    K.kda_recurrent_step(*args, state)
    assert K.kda_device_status() == K.KDA_OK
    args[3] = args[3].clone()
    args[3][5, 1, 100] = -5.5
    K.kda_recurrent_step(*args, state)
    assert K.kda_device_status() == K.KDA_ERR_INPUT


@pytest.mark.parametrize("offsets,ok", [([0, 100, 300, 600], True), ([0, 300, 100, 600], False),
                                        ([5, 100, 300, 600], False), ([0, 100, 300, 590], False)])
def test_packed_offsets(K, offsets, ok):
    inp = inputs.make_prefill(batch=1, seqlen=0, heads=2, dk=128, dv=128, dtype=BF, device="cuda",
                              seed=504, init_state=True, lengths=[100, 200, 300])
    cu = torch.tensor(offsets, dtype=torch.int32, device="cuda")
    fwd(K, inp, cu=cu)
    assert K.kda_device_status() == (K.KDA_OK if ok else K.KDA_ERR_INPUT)
