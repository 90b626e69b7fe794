"""fp64 CPU oracle for Kimi Delta Attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package.  The product path (``linear_attention_fwd_gb300``)
never imports it, and this package imports nothing from the product path.

What it computes (``kda_oracle.c`` holds the arithmetic; this file only
marshals arrays and splits (sequence, head) units over threads):

* ``forward``: the token-by-token gated delta rule of "はじめての自然言語処理 --
  Kimi K3" section 3.1 (KDA): per token, forget with Diag(exp g_t), read
  vhat = S^T k_t, e = v_t - vhat, write S += beta_t k_t e^T, read out
  o_t = S_t^T q_t.  Dense batches and packed variable-length sequences
  (``cu_seqlens``) with an optional initial state; returns the outputs and the
  final states.
* ``decode_step``: the same single token step applied in place to a pool of
  states, row n using slot ``state_indices[n]`` (identity when None).
* ``l2norm_rows``: the L2 normalisation q and k go through before the recurrence
  reads them (same section, the associative-memory read-out paragraph: with
  normalised q and k, q . k is a cosine), x / sqrt(|x|^2 + eps) per row in
  float64, optionally rounded to an io dtype (``round_bf16`` for bf16); a row
  with |x|^2 + eps = 0 stays zero.
* ``gated_rmsnorm``: the output gate of the same page's KDA paragraph (the
  read-out is normalised to unit RMS over its value channels, scaled by a
  per-channel weight, and multiplied channel-wise by a sigmoid gate in (0, 1)):
  y = o / sqrt(mean_j o_j^2 + eps) * w * sigmoid(z), in numpy float64.

Inputs may be any float dtype (the exact values the GPU sees); they are widened
to float64.  Pinned against brute force, closed forms and invariants in
``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile kda_oracle.c into a shared library beside it (gcc -O2, no fast-math)."""
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-std=c99",
                               "-fno-fast-math", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            d = ctypes.POINTER(ctypes.c_double)
            i64 = ctypes.c_int64
            p64 = ctypes.POINTER(ctypes.c_int64)
            lib.kda_oracle_forward.restype = ctypes.c_int
            lib.kda_oracle_forward.argtypes = [d, d, d, d, d, d, p64, i64, i64, i64,
                                               i64, d, d, i64, i64]
            lib.kda_oracle_decode_step.restype = ctypes.c_int
            lib.kda_oracle_decode_step.argtypes = [d, d, d, d, d, d, p64, i64, i64,
                                                   i64, i64, d, i64, i64]
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # a torch tensor: take its exact values
        import torch
        x = x.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    if a.dtype == np.int64:
        return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _run_units(fn, n_units: int, threads: int | None, units=None):
    """Call fn(u0, u1) over unit ranges; ctypes drops the GIL so threads run in parallel."""
    if units is not None:
        todo = [(int(u), int(u) + 1) for u in units]
    else:
        threads = threads or default_threads()
        step = max(1, (n_units + threads * 4 - 1) // (threads * 4))
        todo = [(u, min(u + step, n_units)) for u in range(0, n_units, step)]
    threads = threads or default_threads()
    if threads == 1 or len(todo) == 1:
        for a, b in todo:
            if fn(a, b) != 0:
                raise MemoryError("oracle scratch allocation failed")
        return
    with ThreadPoolExecutor(max_workers=threads) as ex:
        for rc in ex.map(lambda ab: fn(*ab), todo):
            if rc != 0:
                raise MemoryError("oracle scratch allocation failed")


def forward(q, k, v, g, beta, initial_state=None, cu_seqlens=None, *,
            threads: int | None = None, units=None):
    """Token-by-token KDA forward in fp64.

    Dense: q, k, g are [B, T, H, dk], v is [B, T, H, dv], beta is [B, T, H].
    Varlen: the same with B == 1 and ``cu_seqlens`` ([N+1] offsets into T).
    ``initial_state``: [N, H, dk, dv] or None (zeros).
    ``units``: optional iterable of (sequence*H + head) units to compute; the
    outputs of the other units are left as NaN (sampled parity at full size).
    Returns (out [B, T, H, dv] float64, final_state [N, H, dk, dv] float64).
    """
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if cu_seqlens is None:
        N = B
        cu = np.arange(N + 1, dtype=np.int64) * T
    else:
        if B != 1:
            raise ValueError("packed sequences need B == 1")
        cu = np.ascontiguousarray(np.asarray(
            cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens, dtype=np.int64))
        N = cu.shape[0] - 1
        if cu[0] != 0 or cu[-1] != T or np.any(np.diff(cu) < 0):
            raise ValueError("cu_seqlens must rise from 0 to the token count")
    s0 = None if initial_state is None else _f64(initial_state)
    if s0 is not None and s0.shape != (N, H, dk, dv):
        raise ValueError(f"initial_state must be {(N, H, dk, dv)}, got {s0.shape}")
    out = np.full((B, T, H, dv), np.nan if units is not None else 0.0)
    sT = np.full((N, H, dk, dv), np.nan if units is not None else 0.0)
    lib = _load()
    args = [_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(s0), _ptr(cu),
            N, H, dk, dv, _ptr(out), _ptr(sT)]
    _run_units(lambda a, b: lib.kda_oracle_forward(*args, a, b), N * H, threads, units)
    return out, sT


def decode_step(q, k, v, g, beta, state, state_indices=None, *,
                threads: int | None = None, units=None):
    """One recurrent KDA token step per row, in place on ``state`` (float64 ndarray).

    q, k, g: [N, H, dk]; v: [N, H, dv]; beta: [N, H]; state: [P, H, dk, dv]
    float64, modified in place; state_indices: [N] slots or None (identity).
    Returns out [N, H, dv] float64.
    """
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    if not (isinstance(state, np.ndarray) and state.dtype == np.float64
            and state.flags.c_contiguous):
        raise TypeError("state must be a C-contiguous float64 ndarray (updated in place)")
    N, H, dk = q.shape
    dv = v.shape[-1]
    idx = None
    if state_indices is not None:
        idx = np.ascontiguousarray(np.asarray(
            state_indices.cpu() if hasattr(state_indices, "cpu") else state_indices,
            dtype=np.int64))
        if idx.shape != (N,) or np.any(idx < 0) or np.any(idx >= state.shape[0]):
            raise ValueError("state_indices out of range")
        if len(np.unique(idx)) != N:
            raise ValueError("state_indices must not repeat a slot")
    elif state.shape[0] < N:
        raise ValueError("state pool smaller than the number of rows")
    out = np.zeros((N, H, dv))
    lib = _load()
    args = [_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state), _ptr(idx),
            N, H, dk, dv, _ptr(out)]
    _run_units(lambda a, b: lib.kda_oracle_decode_step(*args, a, b), N * H, threads, units)
    return out


def gated_rmsnorm(o, gate, weight=None, eps: float = 1e-6) -> np.ndarray:
    """The KDA output gate: RMSNorm over the last (value-channel) axis, then the channel-wise
    sigmoid gate ("はじめての自然言語処理 -- Kimi K3", the paragraph after the decay bound:
    the gate multiplies each channel by a value in (0, 1) made from the token's input, and
    the RMSNorm before it evens out the magnitude of what is read from S).

    o: [..., dv] (any float dtype, e.g. ``forward``'s float64 output); gate: [..., dv] logits
    z; weight: [dv] or None (ones).  Returns float64 o / sqrt(mean(o^2) + eps) * w * sigmoid(z).
    """
    o = _f64(o)
    z = _f64(gate)
    w = np.ones(o.shape[-1]) if weight is None else _f64(weight)
    rstd = 1.0 / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps)
    return o * rstd * w / (1.0 + np.exp(-z))


def round_bf16(x) -> np.ndarray:
    """float64 values rounded to the nearest bfloat16 (ties to even), returned as float64.

    bfloat16 keeps 8 significant bits and float32's exponent range: a normal value
    m 2^e (0.5 <= |m| < 1) becomes rint(m 2^8) 2^(e-8), with numpy's rint rounding
    halfway cases to even; below 2^-126 the spacing is the subnormal step 2^-133.
    Finite inputs of magnitude below bfloat16's largest finite value only.
    """
    x = _f64(x)
    m, e = np.frexp(x)
    normal = np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)
    sub = np.rint(np.ldexp(x, 133)) * 2.0 ** -133
    return np.where(np.abs(x) < 2.0 ** -126, sub, normal)


def l2norm_rows(x, eps: float, io_dtype: str = "f64") -> np.ndarray:
    """x / sqrt(sum(x^2) + eps) over the last axis, in float64 ("はじめての自然言語処理 --
    Kimi K3", section 3.1, the read-out paragraph: q and k are used after L2
    normalisation).  A row with sum(x^2) + eps = 0 stays zero.  io_dtype "bf16" or "f32"
    rounds the result to that type (what a caller storing its normalised q and k passes
    on); "f64" leaves it unrounded.
    """
    x = _f64(x)
    den = np.sum(x * x, axis=-1, keepdims=True) + eps
    y = np.where(den > 0.0, x / np.sqrt(np.where(den > 0.0, den, 1.0)), 0.0)
    if io_dtype == "bf16":
        return round_bf16(y)
    if io_dtype == "f32":
        return y.astype(np.float32).astype(np.float64)
    if io_dtype != "f64":
        raise ValueError(f"io_dtype {io_dtype!r}")
    return y
