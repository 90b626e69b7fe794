"""Seeded synthetic inputs for the KDA workloads.

This module only draws random numbers and applies the caller-side preparation
that precedes the operator (L2-normalised q and k, g = -5*sigmoid(x),
beta = sigmoid(x)); it holds none of the recurrence's arithmetic.  Both the
CUDA path and the fp64 oracle are fed from it, the oracle with the exact
(rounded) values the GPU sees.

Distributions follow the KDA description in "はじめての自然言語処理 -- Kimi K3"
section 3.1: q and k are used after L2 normalisation, beta is a sigmoid in
(0, 1), and the log decay is -5*sigmoid(.) so that g lies in (-5, 0).

Draw order inside one workload is fixed: q, k, v, g source, beta source,
initial state.  Everything comes from one ``torch.Generator`` on ``device``
seeded with ``seed``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

SEED_BASE = 20260


@dataclass(frozen=True)
class Workload:
    """One synthetic workload.  ``kind`` is 'prefill' or 'decode'."""
    name: str
    kind: str
    heads: int
    dk: int
    dv: int
    dtype: torch.dtype
    batch: int = 1
    seqlen: int = 0
    num_seqs: int = 0          # varlen: number of packed sequences (batch == 1)
    total_tokens: int = 0      # varlen: sum of the lengths
    g_mode: str = "sigmoid"    # 'sigmoid': -5*sigmoid(N(0,1)); 'near_bound': -5 + 0.01*U(0,1)
    init_state: bool = False   # initial/decode state ~ N(0, 0.02^2)
    decode_steps: int = 0
    seed: int = SEED_BASE
    note: str = ""
    extra: dict = field(default_factory=dict)


WORKLOADS = {
    "tiny_fp32": Workload(
        "tiny_fp32", "prefill", heads=2, dk=64, dv=64, dtype=torch.float32,
        batch=1, seqlen=256, seed=SEED_BASE + 0,
        note="B=1 H=2 T=256 dk=dv=64 fp32, zero initial state"),
    "prefill_b4_h32_t8192": Workload(
        "prefill_b4_h32_t8192", "prefill", heads=32, dk=128, dv=128,
        dtype=torch.bfloat16, batch=4, seqlen=8192, seed=SEED_BASE + 1,
        note="B=4 H=32 T=8192 d=128 bf16, zero initial state"),
    "long_h64_t65536": Workload(
        "long_h64_t65536", "prefill", heads=64, dk=128, dv=128,
        dtype=torch.bfloat16, batch=1, seqlen=65536, g_mode="near_bound",
        seed=SEED_BASE + 2,
        note="B=1 H=64 T=65536 d=128 bf16, g = -5 + 0.01*U(0,1) (every 16-token tile at -80)"),
    "varlen_16seq_1m": Workload(
        "varlen_16seq_1m", "prefill", heads=32, dk=128, dv=128,
        dtype=torch.bfloat16, batch=1, num_seqs=16, total_tokens=1 << 20,
        init_state=True, seed=SEED_BASE + 3,
        note="16 packed sequences, log-uniform lengths in [1K,128K], 2^20 tokens, "
             "H=32 d=128 bf16, initial state N(0,0.02^2)"),
    "prefill_b4_h96_t8192": Workload(
        "prefill_b4_h96_t8192", "prefill", heads=96, dk=128, dv=128,
        dtype=torch.bfloat16, batch=4, seqlen=8192, seed=SEED_BASE + 5,
        note="B=4 H=96 T=8192 d=128 bf16 (96 KDA heads per layer), zero initial state"),
    "decode_n256_h64": Workload(
        "decode_n256_h64", "decode", heads=64, dk=128, dv=128,
        dtype=torch.bfloat16, batch=256, init_state=True, decode_steps=1000,
        seed=SEED_BASE + 4,
        note="256 rows x 1 token, H=64 d=128, fp32 state N(0,0.02^2) in place, 1000 steps"),
}


def varlen_lengths(num_seqs: int, total: int, lo: int, hi: int, seed: int) -> list[int]:
    """Log-uniform lengths in [lo, hi], rescaled to sum exactly to ``total``.

    Draw l_i = exp(U(ln lo, ln hi)); repeatedly rescale to the target sum,
    round and clamp to [lo, hi]; the integer residual goes to the longest
    sequences that still have room.
    """
    if not (num_seqs * lo <= total <= num_seqs * hi):
        raise ValueError("total is not reachable within [lo, hi]")
    rng = np.random.default_rng(seed)
    x = np.exp(rng.uniform(math.log(lo), math.log(hi), size=num_seqs))
    for _ in range(64):
        x = np.clip(x * (total / x.sum()), lo, hi)
    n = np.clip(np.rint(x).astype(np.int64), lo, hi)
    resid = int(total - n.sum())
    order = np.argsort(-n, kind="stable")
    while resid != 0:
        moved = False
        for i in order:
            if resid > 0 and n[i] < hi:
                n[i] += 1; resid -= 1; moved = True
            elif resid < 0 and n[i] > lo:
                n[i] -= 1; resid += 1; moved = True
            if resid == 0:
                break
        if not moved:
            raise RuntimeError("cannot place the residual")
    assert int(n.sum()) == total
    return [int(a) for a in n]


def _l2n(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-6)


def _draw_g(gen, shape, mode, device):
    if mode == "sigmoid":
        return -5.0 * torch.sigmoid(torch.randn(shape, generator=gen, device=device))
    if mode == "near_bound":
        return -5.0 + 0.01 * torch.rand(shape, generator=gen, device=device)
    if mode == "zero":
        return torch.zeros(shape, device=device)
    raise ValueError(mode)


def make_prefill(*, batch: int, seqlen: int, heads: int, dk: int, dv: int,
                 dtype: torch.dtype, device="cpu", seed: int = SEED_BASE,
                 g_mode: str = "sigmoid", init_state: bool = False,
                 lengths: list[int] | None = None, raw_qk: bool = False) -> dict:
    """Inputs for one prefill / resume call.

    Dense when ``lengths`` is None ([batch, seqlen, heads, d]); otherwise packed
    ([1, sum(lengths), heads, d]) with int32 ``cu_seqlens``.  The initial state,
    when requested, is fp32 [N, heads, dk, dv] ~ N(0, 0.02^2).  ``raw_qk``: q and k
    are left as drawn, N(0, 1) entries (for calls that normalise them themselves).
    """
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    if lengths is not None:
        batch, seqlen, n_seq = 1, int(sum(lengths)), len(lengths)
    else:
        n_seq = batch
    shp_k = (batch, seqlen, heads, dk)
    shp_v = (batch, seqlen, heads, dv)
    nrm = (lambda x: x) if raw_qk else _l2n
    q = nrm(torch.randn(shp_k, generator=gen, device=device)).to(dtype)
    k = nrm(torch.randn(shp_k, generator=gen, device=device)).to(dtype)
    v = torch.randn(shp_v, generator=gen, device=device).to(dtype)
    g = _draw_g(gen, shp_k, g_mode, device).to(dtype)
    beta = torch.sigmoid(torch.randn((batch, seqlen, heads), generator=gen,
                                     device=device)).to(dtype)
    s0 = None
    if init_state:
        s0 = 0.02 * torch.randn((n_seq, heads, dk, dv), generator=gen, device=device)
    cu = None
    if lengths is not None:
        cu = torch.tensor([0] + list(np.cumsum(lengths)), dtype=torch.int32, device=device)
    return dict(q=q, k=k, v=v, g=g, beta=beta, initial_state=s0, cu_seqlens=cu)


def make_decode_state(*, num_slots: int, heads: int, dk: int, dv: int, device="cpu",
                      seed: int = SEED_BASE) -> torch.Tensor:
    """fp32 recurrent state pool [num_slots, heads, dk, dv] ~ N(0, 0.02^2)."""
    gen = torch.Generator(device=torch.device(device))
    gen.manual_seed(seed)
    return 0.02 * torch.randn((num_slots, heads, dk, dv), generator=gen, device=device)


def make_decode_inputs(*, steps: int, rows: int, heads: int, dk: int, dv: int,
                       dtype: torch.dtype, device="cpu", seed: int = SEED_BASE + 1,
                       g_mode: str = "sigmoid", raw_qk: bool = False) -> dict:
    """Per-step decode inputs [steps, rows, heads, d] (beta: [steps, rows, heads]); ``raw_qk``
    as in ``make_prefill``."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    nrm = (lambda x: x) if raw_qk else _l2n
    q = nrm(torch.randn((steps, rows, heads, dk), generator=gen, device=device)).to(dtype)
    k = nrm(torch.randn((steps, rows, heads, dk), generator=gen, device=device)).to(dtype)
    v = torch.randn((steps, rows, heads, dv), generator=gen, device=device).to(dtype)
    g = _draw_g(gen, (steps, rows, heads, dk), g_mode, device).to(dtype)
    beta = torch.sigmoid(torch.randn((steps, rows, heads), generator=gen,
                                     device=device)).to(dtype)
    return dict(q=q, k=k, v=v, g=g, beta=beta)


def make_workload(name: str, device="cpu", *, decode_steps: int | None = None) -> dict:
    """Inputs of one named workload (see ``WORKLOADS``)."""
    w = WORKLOADS[name]
    if w.kind == "prefill":
        lengths = None
        if w.num_seqs:
            lengths = varlen_lengths(w.num_seqs, w.total_tokens, 1024, 131072, w.seed)
        return make_prefill(batch=w.batch, seqlen=w.seqlen, heads=w.heads, dk=w.dk,
                            dv=w.dv, dtype=w.dtype, device=device, seed=w.seed,
                            g_mode=w.g_mode, init_state=w.init_state, lengths=lengths)
    steps = w.decode_steps if decode_steps is None else decode_steps
    state = make_decode_state(num_slots=w.batch, heads=w.heads, dk=w.dk, dv=w.dv,
                              device=device, seed=w.seed)
    inp = make_decode_inputs(steps=steps, rows=w.batch, heads=w.heads, dk=w.dk,
                             dv=w.dv, dtype=w.dtype, device=device, seed=w.seed + 1000)
    inp["state"] = state
    return inp
