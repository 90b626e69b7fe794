"""GPU tests of kda_chunk_fwd_checkpointed (recurrent-state checkpoints inside each sequence,
for prefix caching) through the C ABI, on both chunk kernels (fp32 and bf16 d=64: the SIMT
kernel, which the library keeps for checkpoints at d=64; bf16 d=128: the tensor-core kernel).

Pins: a checkpoint is the final state of the same computation on the prefix, which the oracle
computes independently (its token recurrence over the first (k+1)*interval tokens); and, for
the same kernel, the checkpoint equals the final state of a call on that prefix bit for bit
(a chunk's arithmetic never depends on later tokens).
"""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_fwd_gb300 import inputs
from tests.helpers import rel_max_err
from tests.parity import TOL, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K(cuda_device):
    from linear_attention_fwd_gb300 import build, kda
    build.build()
    return kda


CASES = [(torch.float32, 64), (torch.bfloat16, 64), (torch.bfloat16, 128)]


def _prefix(inp, n, cu, L):
    """Inputs of the first L tokens of sequence n as a one-sequence dense batch."""
    if cu is None:
        sl = lambda t: t[n:n + 1, :L]   # noqa: E731
    else:
        b = int(cu[n])
        sl = lambda t: t[:, b:b + L]    # noqa: E731
    return {kk: sl(inp[kk]).contiguous() for kk in ("q", "k", "v", "g", "beta")}


@pytest.mark.parametrize("dtype,d", CASES)
@pytest.mark.parametrize("varlen", [False, True])
def test_checkpoints_match_prefix_states(K, dtype, d, varlen):
    H, interval = 3, 128
    lengths = [449, 64, 320, 1] if varlen else None
    inp = inputs.make_prefill(batch=2, seqlen=385, heads=H, dk=d, dv=d, dtype=dtype, device="cuda",
                              seed=61, init_state=True, lengths=lengths)
    cu = inp["cu_seqlens"]
    out, fs, ck, off = K.kda_chunk_fwd_checkpointed(inp["q"], inp["k"], inp["v"], inp["g"],
                                                    inp["beta"], inp["initial_state"], cu,
                                                    interval=interval)
    torch.cuda.synchronize()
    # the plain calls compared bit for bit run the kernel the checkpointed call runs
    impl = "tc" if (dtype == torch.bfloat16 and d == 128) else "simt"
    ref_out, ref_fs = K.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                      inp["initial_state"], cu, impl=impl)
    torch.testing.assert_close(out, ref_out, rtol=0, atol=0)   # checkpoints change nothing else
    torch.testing.assert_close(fs, ref_fs, rtol=0, atol=0)
    offs = off.cpu().numpy()
    cuh = None if cu is None else cu.cpu().numpy()
    lens = [385, 385] if cu is None else lengths
    for n, L in enumerate(lens):
        count = offs[n + 1] - offs[n]
        assert count == max(0, (L - 1) // interval)
        for kth in range(count):
            P = (kth + 1) * interval
            pre = _prefix(inp, n, cuh, P)
            s0 = inp["initial_state"][n:n + 1].contiguous()
            _, gpu_fs = K.kda_chunk_fwd(pre["q"], pre["k"], pre["v"], pre["g"], pre["beta"], s0, impl=impl)
            torch.cuda.synchronize()
            torch.testing.assert_close(ck[offs[n] + kth], gpu_fs[0], rtol=0, atol=0)
            _, rs = oracle.forward(pre["q"], pre["k"], pre["v"], pre["g"], pre["beta"], s0)
            assert rel_max_err(f64(ck[offs[n] + kth]), rs[0]) <= TOL[dtype]


def test_checkpoint_validation(K):
    inp = inputs.make_prefill(batch=1, seqlen=256, heads=2, dk=128, dv=128, dtype=torch.bfloat16,
                              device="cuda", seed=62)
    with pytest.raises(K.KdaError):   # interval not a multiple of the chunk
        K.kda_chunk_fwd_checkpointed(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                     interval=100)
    # slots outside a sequence's range are never written
    off = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    ck = torch.full((2, 2, 128, 128), 3.0, device="cuda")
    K.kda_chunk_fwd_checkpointed(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], interval=64,
                                 checkpoints=ck, offsets=off)
    torch.cuda.synchronize()
    assert torch.all(ck[1] == 3.0) and not torch.all(ck[0] == 3.0)
