"""kda_chunk_fwd_noalloc -- the two-pass forward in the library's fixed per-device scratch area
-- against the existing entry point with a caller workspace (kda_chunk_fwd_ws): two calls in a
row on different inputs, each within the forward's bar (TOL * RMS of the existing entry
point's result), with no device allocation by the caller's allocator during the call; a call
whose workspace would exceed the area is rejected before anything is written.

The file sorts last so that it also runs after every other GPU test in the same process (the
area is set up by whichever call comes first on the device); it passes alone as well.
"""
import pytest
import torch

from linear_attention_fwd_gb300 import inputs
from tests.parity import TOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K(cuda_device):
    from linear_attention_fwd_gb300 import build, kda
    build.build()
    return kda


def _rel(x, ref):
    x, ref = x.double(), ref.double()
    rms = ref.pow(2).mean().sqrt().item()
    return (x - ref).abs().max().item() / rms


def _with_workspace(K, inp):
    return K.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                           inp["initial_state"], inp["cu_seqlens"], impl="two_pass")


def _noalloc(K, inp):
    q, v = inp["q"], inp["v"]
    n = q.shape[0] if inp["cu_seqlens"] is None else inp["cu_seqlens"].numel() - 1
    out = torch.full_like(v, float("nan"))
    fs = torch.full((n, q.shape[2], q.shape[3], v.shape[3]), float("nan"), device=q.device)
    torch.cuda.synchronize()
    before = torch.cuda.memory_stats(q.device).get("allocation.all.allocated", 0)
    K.kda_chunk_fwd_noalloc(q, inp["k"], v, inp["g"], inp["beta"], inp["initial_state"],
                            inp["cu_seqlens"], out, fs)
    torch.cuda.synchronize()
    after = torch.cuda.memory_stats(q.device).get("allocation.all.allocated", 0)
    assert after == before, "the call went through the caller's allocator"
    return out, fs


def test_two_calls_in_a_row_match_the_workspace_entry_point(K):
    cases = [
        inputs.make_prefill(batch=2, seqlen=300, heads=4, dk=128, dv=128, dtype=torch.bfloat16,
                            device="cuda", seed=91, init_state=True),
        inputs.make_prefill(batch=1, seqlen=0, heads=3, dk=128, dv=128, dtype=torch.bfloat16,
                            device="cuda", seed=92, init_state=True, lengths=[200, 1, 64, 129]),
    ]
    tol = TOL[torch.bfloat16]
    for inp in cases:
        need = K.kda_chunk_fwd_workspace_bytes(inp["q"], inp["v"], inp["cu_seqlens"])
        assert 0 < need <= K.NOALLOC_SCRATCH_BYTES
        ro, rf = _with_workspace(K, inp)
        o, f = _noalloc(K, inp)
        assert torch.isfinite(o).all() and torch.isfinite(f).all()
        eo, ef = _rel(o, ro), _rel(f, rf)
        print(f"noalloc vs workspace entry point: output {eo:.2e}, final state {ef:.2e}")
        assert eo <= tol and ef <= tol


def test_rejects_a_call_beyond_the_scratch_area(K):
    # B=1, T=8192, H=32: 129 chunk slots per head of 24 KB, about 101 MB > 64 MiB
    inp = inputs.make_prefill(batch=1, seqlen=8192, heads=32, dk=128, dv=128,
                              dtype=torch.bfloat16, device="cuda", seed=93)
    assert K.kda_chunk_fwd_workspace_bytes(inp["q"], inp["v"]) > K.NOALLOC_SCRATCH_BYTES
    out = torch.full_like(inp["v"], float("nan"))
    fs = torch.full((1, 32, 128, 128), float("nan"), device="cuda")
    with pytest.raises(K.KdaError) as e:
        K.kda_chunk_fwd_noalloc(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], None, None,
                                out, fs)
    assert e.value.status == K.KDA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.isnan(out).all() and torch.isnan(fs).all()   # nothing ran
