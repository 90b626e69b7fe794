"""GPU parity of the segmented tensor-core launch against the oracle.

With P segments, CTA p stores the outputs of chunks [p nc / P, (p+1) nc / P) of its sequence and
starts from a zero state at the latest chunk boundary (at most 16 chunks earlier) past which the
bound prod_t max_i e^{g_t,i} max(1, |1 - beta_t |k_t|^2|) on the transitions has fallen to
2^-160, else at the start of the sequence with its initial state.  Checked here: the decay
bound (one chunk of warm-up), the standard decay distribution (several chunks), keys that are
not unit vectors (transitions that can stretch the state), a decay-free channel (no horizon:
every segment runs from the start and the result equals one CTA per unit bit for bit), packed
sequences with empty and one-token members, empty segments, the library's own choice on a long
sequence, the bounded-wait expiry path under segments, and the in-place rejection.
"""
import numpy as np
import pytest
import torch

from linear_attention_fwd_gb300 import inputs
from tests.parity import check_prefill, compare_prefill, f64

pytestmark = pytest.mark.gpu
BF = torch.bfloat16


@pytest.fixture(scope="module")
def K(cuda_device):
    from linear_attention_fwd_gb300 import build, kda
    build.build()
    return kda


def run(K, inp, **kw):
    out, sT = K.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                              inp.get("initial_state"), inp.get("cu_seqlens"), impl="tc", **kw)
    torch.cuda.synchronize()
    return out, sT


def rel_diff(a, b):
    a, b = f64(a), f64(b)
    return float(np.abs(a - b).max() / np.sqrt(np.mean(b * b)))


@pytest.mark.parametrize("P", [2, 3, 5, 8])
def test_segments_at_the_decay_bound(K, P):
    # every g is -5 in bf16: one warm-up chunk reaches the 2^-160 horizon
    inp = inputs.make_prefill(batch=1, seqlen=2000, heads=2, dk=128, dv=128, dtype=BF,
                              device="cuda", seed=301, g_mode="near_bound", init_state=True)
    out, sT = run(K, inp, segments=P)
    check_prefill(compare_prefill(inp, out, sT), BF)
    out1, sT1 = run(K, inp, segments=1)
    assert rel_diff(sT, sT1) <= 1e-3   # (bf16 outputs may differ by an ulp: both meet the bar)


@pytest.mark.parametrize("P", [2, 4])
def test_segments_with_the_standard_decay(K, P):
    # g = -5 sigmoid(N(0,1)): the largest channel decays slowly, so the warm-up spans chunks
    inp = inputs.make_prefill(batch=2, seqlen=3000, heads=2, dk=128, dv=128, dtype=BF,
                              device="cuda", seed=302, init_state=True)
    out, sT = run(K, inp, segments=P)
    check_prefill(compare_prefill(inp, out, sT), BF)


def test_segments_with_keys_that_stretch_the_state(K):
    # |k| = 1.7 and beta = 1: I - beta k k^T stretches the k direction by |1 - 2.89| = 1.89,
    # which the bound counts (log2 1.89 per token against -7.2 of decay)
    inp = inputs.make_prefill(batch=1, seqlen=1500, heads=2, dk=128, dv=128, dtype=BF,
                              device="cuda", seed=303, g_mode="near_bound", init_state=True)
    inp["k"] = (f64(inp["k"]) * 1.7)
    inp["k"] = torch.tensor(inp["k"], dtype=BF, device="cuda")
    inp["beta"] = torch.ones_like(inp["beta"])
    out, sT = run(K, inp, segments=4)
    check_prefill(compare_prefill(inp, out, sT), BF)


def test_no_horizon_runs_every_segment_from_the_start(K):
    # one channel never decays: the bound never falls, so each segment starts at token 0 with
    # the initial state and computes exactly what one CTA per unit computes
    inp = inputs.make_prefill(batch=1, seqlen=1200, heads=2, dk=128, dv=128, dtype=BF,
                              device="cuda", seed=304, g_mode="near_bound", init_state=True)
    inp["g"][..., 5] = 0
    out1, sT1 = run(K, inp, segments=1)
    for P in (2, 3, 7):
        out, sT = run(K, inp, segments=P)
        assert torch.equal(out, out1) and torch.equal(sT, sT1)
    check_prefill(compare_prefill(inp, out1, sT1), BF)


def test_packed_sequences_with_segments(K):
    lengths = [1, 64, 0, 130, 2000, 1100, 65]
    inp = inputs.make_prefill(batch=1, seqlen=0, heads=3, dk=128, dv=128, dtype=BF,
                              device="cuda", seed=305, g_mode="near_bound", init_state=True,
                              lengths=lengths)
    for P in (3, 6):
        out, sT = run(K, inp, segments=P)
        check_prefill(compare_prefill(inp, out, sT), BF)


def test_empty_segments(K):
    # 2 chunks over 5 segments: segments 0, 1 and 3 store nothing and return at once
    inp = inputs.make_prefill(batch=2, seqlen=100, heads=2, dk=128, dv=128, dtype=BF,
                              device="cuda", seed=306, g_mode="near_bound", init_state=True)
    out, sT = run(K, inp, segments=5)
    check_prefill(compare_prefill(inp, out, sT), BF)


def test_library_choice_on_a_long_sequence(K):
    # 4 units on a GPU with more SMs: the default call splits each sequence
    inp = inputs.make_prefill(batch=1, seqlen=8192, heads=4, dk=128, dv=128, dtype=BF,
                              device="cuda", seed=307, init_state=True)
    out, sT = K.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                              inp["initial_state"])
    torch.cuda.synchronize()
    check_prefill(compare_prefill(inp, out, sT), BF)
    out1, sT1 = run(K, inp, segments=1)
    assert rel_diff(sT, sT1) <= 1e-3   # (bf16 outputs may differ by an ulp: both meet the bar)


def test_expired_waits_under_segments(K):
    # 1 unit and 64 chunks: the library picks 4 segments; with a bound of zero polls every
    # segment stops at its first wait, every segment's outputs and the final state are NaN
    inp = inputs.make_prefill(batch=1, seqlen=4096, heads=1, dk=128, dv=128, dtype=BF,
                              device="cuda", seed=308, init_state=True)
    out, sT = run(K, inp, wait_polls=0)
    assert torch.isnan(sT).all() and torch.isnan(out.float()).all()
    assert K.kda_device_status() == K.KDA_ERR_TIMEOUT   # reported to the host, and cleared
    out, sT = run(K, inp)
    assert K.kda_device_status() == K.KDA_OK
    check_prefill(compare_prefill(inp, out, sT), BF)


def test_in_place_state_is_rejected_with_segments(K):
    inp = inputs.make_prefill(batch=1, seqlen=256, heads=1, dk=128, dv=128, dtype=BF,
                              device="cuda", seed=309, init_state=True)
    s = inp["initial_state"]
    with pytest.raises(K.KdaError):
        K.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], s, final_state=s,
                        impl="tc", segments=2)
    with pytest.raises(K.KdaError):
        K.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], s, impl="tc",
                        segments=65)
