"""GPU test of the tensor-core kernel's bounded waits, without a GPU fault: with a bound of
zero polls every wait gives up at once, so each (sequence, head) unit stops at its first
chunk, lets its copies in flight land, and reports through a NaN final state and through
kda_device_status (KDA_ERR_TIMEOUT, also when no final state is requested); the context stays
usable, the next call with the normal bound matches the oracle and the status is clean again.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_fwd_gb300 import inputs
from tests.helpers import rel_max_err
from tests.parity import TOL, excess_err, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K(cuda_device):
    from linear_attention_fwd_gb300 import build, kda
    build.build()
    return kda


def test_expired_waits_mark_the_state_and_leave_the_context_usable(K):
    inp = inputs.make_prefill(batch=2, seqlen=200, heads=3, dk=128, dv=128, dtype=torch.bfloat16,
                              device="cuda", seed=71, init_state=True)
    args = (inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["initial_state"])
    assert K.kda_device_status() == K.KDA_OK          # nothing pending from earlier calls
    _, fs = K.kda_chunk_fwd(*args, impl="tc", wait_polls=0)
    torch.cuda.synchronize()   # raises if the expiry path faulted
    assert torch.isnan(fs).all()
    assert K.kda_device_status() == K.KDA_ERR_TIMEOUT
    assert K.kda_device_status() == K.KDA_OK          # read and cleared
    # no final state requested: the status is the only signal, and it is there
    _, none = K.kda_chunk_fwd(*args, impl="tc", wait_polls=0, output_final_state=False)
    assert none is None
    assert K.kda_device_status() == K.KDA_ERR_TIMEOUT
    out, fs = K.kda_chunk_fwd(*args, impl="tc")
    torch.cuda.synchronize()
    assert K.kda_device_status() == K.KDA_OK
    ro, rs = oracle.forward(*args)
    assert excess_err(f64(out), ro, torch.bfloat16) <= TOL[torch.bfloat16]
    assert rel_max_err(f64(fs), rs) <= TOL[torch.bfloat16]
    assert np.isfinite(f64(fs)).all()
