"""ctypes binding of libkda (include/kda.h): argument marshalling only.

Every computation runs in libkda's CUDA kernels; this module only checks
tensor metadata, fills ``kda_dims_t`` and passes device pointers and the
current CUDA stream.  There is no fallback: if ``libkda.so`` has not been built
the first call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkda.so")
DEBUG_LIB_PATH = os.path.join(_HERE, "libkda_debug.so")   # build.build(debug=True): device input checks

KDA_OK, KDA_ERR_NULL, KDA_ERR_SHAPE, KDA_ERR_UNSUPPORTED = 0, 1, 2, 3
KDA_ERR_ALIGN, KDA_ERR_WORKSPACE, KDA_ERR_CUDA, KDA_ERR_TIMEOUT, KDA_ERR_INPUT = 4, 5, 6, 7, 8
KDA_F32, KDA_BF16 = 0, 1
IMPLS = {"auto": 0, "simt": 1, "tc": 2}
IMPL_NAMES = {v: k for k, v in IMPLS.items()}

# every symbol include/kda.h declares
EXPORTED = ("kda_chunk_fwd", "kda_chunk_fwd_with", "kda_chunk_fwd_bounded", "kda_chunk_fwd_segmented",
            "kda_chunk_fwd_checkpointed", "kda_chunk_fwd_auto_ctas",
            "kda_chunk_fwd_gated", "kda_chunk_fwd_selected_impl", "kda_recurrent_step",
            "kda_recurrent_steps", "kda_device_status", "kda_chunk_fwd_ws",
            "kda_chunk_fwd_workspace_bytes", "kda_chunk_fwd_noalloc", "kda_debug_checks",
            "kda_chunk_fwd_qknorm", "kda_recurrent_step_qknorm", "kda_recurrent_steps_qknorm",
            "kda_status_string")


class KdaDims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("seqlen", ctypes.c_int32),
                ("num_seqs", ctypes.c_int32), ("heads", ctypes.c_int32),
                ("dk", ctypes.c_int32), ("dv", ctypes.c_int32), ("dtype", ctypes.c_int32)]


class KdaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {kda_status_string(status)} (status {status})")


_lib = None


def lib() -> ctypes.CDLL:
    """Load libkda.so (built in-tree by ``linear_attention_fwd_gb300.build``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        vp, dp = ctypes.c_void_p, ctypes.POINTER(KdaDims)
        L.kda_chunk_fwd.restype = ctypes.c_int
        L.kda_chunk_fwd.argtypes = [vp] * 9 + [dp, vp]
        L.kda_chunk_fwd_with.restype = ctypes.c_int
        L.kda_chunk_fwd_with.argtypes = [ctypes.c_int] + [vp] * 9 + [dp, vp]
        L.kda_chunk_fwd_bounded.restype = ctypes.c_int
        L.kda_chunk_fwd_bounded.argtypes = [ctypes.c_int] + [vp] * 9 + [ctypes.c_uint32, dp, vp]
        L.kda_chunk_fwd_segmented.restype = ctypes.c_int
        L.kda_chunk_fwd_segmented.argtypes = [ctypes.c_int] + [vp] * 9 + [ctypes.c_int32, dp, vp]
        L.kda_chunk_fwd_checkpointed.restype = ctypes.c_int
        L.kda_chunk_fwd_checkpointed.argtypes = [vp] * 11 + [ctypes.c_int32, dp, vp]
        L.kda_chunk_fwd_gated.restype = ctypes.c_int
        L.kda_chunk_fwd_gated.argtypes = [vp] * 7 + [ctypes.c_float] + [vp] * 4 + [dp, vp]
        L.kda_chunk_fwd_auto_ctas.restype = ctypes.c_int
        L.kda_chunk_fwd_auto_ctas.argtypes = [dp, ctypes.c_int, ctypes.c_int]
        L.kda_chunk_fwd_selected_impl.restype = ctypes.c_int
        L.kda_chunk_fwd_selected_impl.argtypes = [dp]
        L.kda_recurrent_step.restype = ctypes.c_int
        L.kda_recurrent_step.argtypes = [vp] * 8 + [dp, vp]
        L.kda_chunk_fwd_qknorm.restype = ctypes.c_int
        L.kda_chunk_fwd_qknorm.argtypes = [vp] * 5 + [ctypes.c_float] + [vp] * 4 + [dp, vp]
        L.kda_recurrent_step_qknorm.restype = ctypes.c_int
        L.kda_recurrent_step_qknorm.argtypes = [vp] * 5 + [ctypes.c_float] + [vp] * 3 + [dp, vp]
        L.kda_recurrent_steps_qknorm.restype = ctypes.c_int
        L.kda_recurrent_steps_qknorm.argtypes = [vp] * 5 + [ctypes.c_float] + [vp] * 4 + [ctypes.c_int, dp, vp]
        L.kda_recurrent_steps.restype = ctypes.c_int
        L.kda_recurrent_steps.argtypes = [vp] * 9 + [ctypes.c_int, dp, vp]
        L.kda_chunk_fwd_ws.restype = ctypes.c_int
        L.kda_chunk_fwd_ws.argtypes = [vp] * 10 + [ctypes.c_size_t, dp, vp]
        L.kda_chunk_fwd_workspace_bytes.restype = ctypes.c_size_t
        L.kda_chunk_fwd_workspace_bytes.argtypes = [dp]
        L.kda_chunk_fwd_noalloc.restype = ctypes.c_int
        L.kda_chunk_fwd_noalloc.argtypes = [vp] * 9 + [dp, vp]
        L.kda_device_status.restype = ctypes.c_int
        L.kda_device_status.argtypes = [vp]
        L.kda_debug_checks.restype = ctypes.c_int
        L.kda_debug_checks.argtypes = []
        L.kda_status_string.restype = ctypes.c_char_p
        L.kda_status_string.argtypes = [ctypes.c_int]
        _lib = L
    return _lib


def kda_status_string(status: int) -> str:
    return lib().kda_status_string(int(status)).decode()


def use_library(path: str) -> None:
    """Load libkda from `path` for the calls that follow (LIB_PATH, or DEBUG_LIB_PATH for the
    build with device-side input checks)."""
    global _lib, LIB_PATH
    LIB_PATH = path
    _lib = None
    lib()


def kda_debug_checks() -> int:
    """Bit mask of the device-side input checks the loaded library runs (0: release build)."""
    return int(lib().kda_debug_checks())


def kda_device_status(stream=None) -> int:
    """Wait for `stream` (default: the current one) and return the device's status code:
    KDA_ERR_TIMEOUT when a bounded device wait gave up since the last call, else KDA_OK
    (the count is cleared)."""
    st = torch.cuda.current_stream() if stream is None else stream
    return int(lib().kda_device_status(ctypes.c_void_p(st.cuda_stream)))


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return KDA_F32
    if t == torch.bfloat16:
        return KDA_BF16
    raise TypeError(f"unsupported dtype {t} (fp32 or bf16)")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check_dev(name, t, device, dtype=None):
    if t is None:
        return
    if not t.is_cuda or t.device != device:
        raise ValueError(f"{name} must be on {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def chunk_dims(q, v, cu_seqlens=None) -> KdaDims:
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    n = B if cu_seqlens is None else cu_seqlens.numel() - 1
    return KdaDims(B, T, n, H, dk, dv, _dtype_code(q.dtype))


def kda_chunk_fwd_workspace_bytes(q, v, cu_seqlens=None) -> int:
    """Bytes of device workspace the two-pass path needs for these shapes (0: one-pass)."""
    dims = chunk_dims(q, v, cu_seqlens)
    return int(lib().kda_chunk_fwd_workspace_bytes(ctypes.byref(dims)))


# KDA_NOALLOC_SCRATCH_BYTES: the fixed scratch area kda_chunk_fwd_noalloc runs in, per device
NOALLOC_SCRATCH_BYTES = 64 << 20


def kda_chunk_fwd_noalloc(q, k, v, g, beta, initial_state, cu_seqlens, out, final_state,
                          stream=None):
    """kda_chunk_fwd_noalloc: the two-pass forward in the library's own fixed scratch area.

    Every tensor is the caller's (out and final_state included; final_state may be None): the
    call allocates no device memory.  The first call with a device current sets the scratch
    area up on it; calls that overlap in time on one device race on that area."""
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("out", out)):
        _check_dev(name, t, dev, q.dtype)
    _check_dev("initial_state", initial_state, dev, torch.float32)
    _check_dev("cu_seqlens", cu_seqlens, dev, torch.int32)
    _check_dev("final_state", final_state, dev, torch.float32)
    if k.shape != q.shape or g.shape != q.shape or v.shape[:3] != q.shape[:3] \
            or beta.shape != q.shape[:3] or out.shape != v.shape:
        raise ValueError("inconsistent q/k/v/g/beta/out shapes")
    dims = chunk_dims(q, v, cu_seqlens)
    st = lib().kda_chunk_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                     _ptr(initial_state), _ptr(cu_seqlens), _ptr(out),
                                     _ptr(final_state), ctypes.byref(dims), _stream_handle(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_chunk_fwd_noalloc")
    return out, final_state


def kda_chunk_fwd(q, k, v, g, beta, initial_state=None, cu_seqlens=None, *, out=None,
                  final_state=None, output_final_state: bool = True, impl: str = "auto",
                  stream=None, wait_polls: int | None = None, segments: int | None = None,
                  workspace=None, qk_eps: float | None = None):
    """Chunkwise KDA forward (prefill / prefix-cache resume) through libkda.

    q, k, g: [B, T, H, dk]; v: [B, T, H, dv]; beta: [B, T, H] (all fp32 or all
    bf16, CUDA, contiguous).  initial_state: fp32 [N, H, dk, dv] or None.
    cu_seqlens: int32 [N+1] (packed sequences, B == 1) or None.
    Returns (out [B, T, H, dv], final_state [N, H, dk, dv] fp32 or None).
    wait_polls: bound on each device wait of the tensor-core kernel (kda_chunk_fwd_bounded);
    a unit whose wait gives up gets a NaN final state.
    segments: CTAs per (sequence, head) on the tensor-core kernel (kda_chunk_fwd_segmented;
    0 = the library's choice, which is also what the default call does).
    impl="two_pass": kda_chunk_fwd_ws, the state-independent chunk work for all chunks first,
    then the state chain; `workspace` is a uint8 CUDA tensor of at least
    kda_chunk_fwd_workspace_bytes bytes (allocated here, by the caller's allocator, when None).
    qk_eps: when given, kda_chunk_fwd_qknorm: q and k rows are L2-normalised first,
    x / sqrt(|x|^2 + qk_eps) in fp32 (impl="auto" only).
    """
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta)):
        _check_dev(name, t, dev, q.dtype)
    _check_dev("initial_state", initial_state, dev, torch.float32)
    _check_dev("cu_seqlens", cu_seqlens, dev, torch.int32)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or g.shape != q.shape or v.shape[:3] != q.shape[:3] \
            or beta.shape != q.shape[:3]:
        raise ValueError("inconsistent q/k/v/g/beta shapes")
    dims = chunk_dims(q, v, cu_seqlens)
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=q.dtype, device=dev)
    _check_dev("out", out, dev, q.dtype)
    if final_state is None and output_final_state:
        final_state = torch.empty((dims.num_seqs, H, dk, dv), dtype=torch.float32, device=dev)
    _check_dev("final_state", final_state, dev, torch.float32)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(initial_state),
            _ptr(cu_seqlens), _ptr(out), _ptr(final_state))
    if wait_polls is not None and segments is not None:
        raise ValueError("wait_polls and segments select different entry points")
    if qk_eps is not None:
        if impl != "auto" or wait_polls is not None or segments is not None:
            raise ValueError("qk_eps selects kda_chunk_fwd_qknorm, which takes impl='auto' only")
        st = lib().kda_chunk_fwd_qknorm(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                        ctypes.c_float(qk_eps), _ptr(initial_state),
                                        _ptr(cu_seqlens), _ptr(out), _ptr(final_state),
                                        ctypes.byref(dims), _stream_handle(stream))
        if st != KDA_OK:
            raise KdaError(st, "kda_chunk_fwd_qknorm")
        return out, final_state
    if impl == "two_pass":
        if wait_polls is not None or segments is not None:
            raise ValueError("the two-pass path takes neither wait_polls nor segments")
        need = int(lib().kda_chunk_fwd_workspace_bytes(ctypes.byref(dims)))
        if workspace is None:
            workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
        _check_dev("workspace", workspace, dev, torch.uint8)
        st = lib().kda_chunk_fwd_ws(*args, _ptr(workspace), ctypes.c_size_t(workspace.numel()),
                                    ctypes.byref(dims), _stream_handle(stream))
        if st != KDA_OK:
            raise KdaError(st, "kda_chunk_fwd_ws")
        return out, final_state
    if segments is not None:
        st = lib().kda_chunk_fwd_segmented(IMPLS[impl], *args, ctypes.c_int32(int(segments)),
                                           ctypes.byref(dims), _stream_handle(stream))
    elif wait_polls is None:
        st = lib().kda_chunk_fwd_with(IMPLS[impl], *args, ctypes.byref(dims), _stream_handle(stream))
    else:
        st = lib().kda_chunk_fwd_bounded(IMPLS[impl], *args, ctypes.c_uint32(int(wait_polls)),
                                         ctypes.byref(dims), _stream_handle(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_chunk_fwd")
    return out, final_state


def kda_chunk_fwd_segmented(q, k, v, g, beta, initial_state=None, cu_seqlens=None, *,
                            segments: int = 0, **kw):
    """kda_chunk_fwd with an explicit number of CTAs per (sequence, head) (tensor-core kernel)."""
    return kda_chunk_fwd(q, k, v, g, beta, initial_state, cu_seqlens, segments=segments, **kw)


def kda_chunk_fwd_auto_ctas(dims: KdaDims, packed: bool, sms: int) -> int:
    """CTAs kda_chunk_fwd launches for the tensor-core kernel on `sms` SMs (0: not that kernel)."""
    return int(lib().kda_chunk_fwd_auto_ctas(ctypes.byref(dims), int(bool(packed)), int(sms)))


def kda_chunk_fwd_selected_impl(q, v, cu_seqlens=None) -> str:
    code = lib().kda_chunk_fwd_selected_impl(ctypes.byref(chunk_dims(q, v, cu_seqlens)))
    return IMPL_NAMES.get(code, "invalid")


def kda_recurrent_step(q, k, v, g, beta, state, state_indices=None, *, out=None, stream=None,
                       qk_eps: float | None = None):
    """One decode token per row through libkda; ``state`` is updated in place.

    q, k, g: [N, H, dk]; v: [N, H, dv]; beta: [N, H]; state: fp32 [P, H, dk, dv];
    state_indices: int32 [N] or None.  Returns out [N, H, dv].
    qk_eps: when given, kda_recurrent_step_qknorm (q and k L2-normalised first).
    """
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta)):
        _check_dev(name, t, dev, q.dtype)
    _check_dev("state", state, dev, torch.float32)
    _check_dev("state_indices", state_indices, dev, torch.int32)
    N, H, dk = q.shape
    dv = v.shape[-1]
    if state.shape[1:] != (H, dk, dv):
        raise ValueError("state must be [P, H, dk, dv]")
    dims = KdaDims(N, 1, state.shape[0], H, dk, dv, _dtype_code(q.dtype))
    if out is None:
        out = torch.empty((N, H, dv), dtype=q.dtype, device=dev)
    _check_dev("out", out, dev, q.dtype)
    if qk_eps is None:
        st = lib().kda_recurrent_step(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state),
                                      _ptr(state_indices), _ptr(out), ctypes.byref(dims),
                                      _stream_handle(stream))
    else:
        st = lib().kda_recurrent_step_qknorm(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                             ctypes.c_float(qk_eps), _ptr(state),
                                             _ptr(state_indices), _ptr(out), ctypes.byref(dims),
                                             _stream_handle(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_recurrent_step" if qk_eps is None else "kda_recurrent_step_qknorm")
    return out


def kda_recurrent_steps(q, k, v, g, beta, state, state_indices=None, num_tokens=None, *,
                        out=None, want_out=True, update_state=True, stream=None,
                        qk_eps: float | None = None):
    """Up to T decode tokens per row through libkda (speculative decoding).

    q, k, g: [N, T, H, dk]; v: [N, T, H, dv]; beta: [N, T, H]; state: fp32 [P, H, dk, dv];
    state_indices, num_tokens: int32 [N] or None.  With update_state the state after each
    row's tokens is written in place; without, the state is only read.  Returns out
    [N, T, H, dv] (tokens past a row's count are left as they were), or None when
    ``want_out`` is false.  qk_eps: when given, kda_recurrent_steps_qknorm (q and k
    L2-normalised first).
    """
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta)):
        _check_dev(name, t, dev, q.dtype)
    _check_dev("state", state, dev, torch.float32)
    _check_dev("state_indices", state_indices, dev, torch.int32)
    _check_dev("num_tokens", num_tokens, dev, torch.int32)
    N, T, H, dk = q.shape
    dv = v.shape[-1]
    if state.shape[1:] != (H, dk, dv):
        raise ValueError("state must be [P, H, dk, dv]")
    dims = KdaDims(N, T, state.shape[0], H, dk, dv, _dtype_code(q.dtype))
    if want_out and out is None:
        out = torch.zeros((N, T, H, dv), dtype=q.dtype, device=dev)
    if out is not None:
        _check_dev("out", out, dev, q.dtype)
    if qk_eps is None:
        st = lib().kda_recurrent_steps(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state),
                                       _ptr(state_indices), _ptr(num_tokens),
                                       _ptr(out) if want_out else None, int(bool(update_state)),
                                       ctypes.byref(dims), _stream_handle(stream))
    else:
        st = lib().kda_recurrent_steps_qknorm(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                              ctypes.c_float(qk_eps), _ptr(state),
                                              _ptr(state_indices), _ptr(num_tokens),
                                              _ptr(out) if want_out else None,
                                              int(bool(update_state)), ctypes.byref(dims),
                                              _stream_handle(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_recurrent_steps" if qk_eps is None else "kda_recurrent_steps_qknorm")
    return out if want_out else None


def checkpoint_offsets(q, cu_seqlens, interval: int):
    """int32 [N+1] device offsets giving each sequence one slot per multiple of ``interval``
    strictly inside it (the layout kda_chunk_fwd_checkpointed fills)."""
    if cu_seqlens is None:
        B, T = q.shape[:2]
        lens = torch.full((B,), T, dtype=torch.int64, device=q.device)
    else:
        lens = (cu_seqlens[1:] - cu_seqlens[:-1]).to(torch.int64)
    counts = torch.clamp((lens - 1) // interval, min=0)
    off = torch.zeros(counts.numel() + 1, dtype=torch.int64, device=q.device)
    off[1:] = torch.cumsum(counts, 0)
    return off.to(torch.int32)


def kda_chunk_fwd_checkpointed(q, k, v, g, beta, initial_state=None, cu_seqlens=None, *,
                               interval: int = 512, out=None, final_state=None,
                               checkpoints=None, offsets=None, stream=None):
    """kda_chunk_fwd that also returns the state at every multiple of ``interval`` tokens
    strictly inside each sequence (prefix caching).

    Returns (out, final_state, checkpoints fp32 [slots, H, dk, dv], offsets int32 [N+1]);
    sequence n's k-th checkpoint (the state after (k+1)*interval tokens) is
    checkpoints[offsets[n] + k].
    """
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta)):
        _check_dev(name, t, dev, q.dtype)
    _check_dev("initial_state", initial_state, dev, torch.float32)
    _check_dev("cu_seqlens", cu_seqlens, dev, torch.int32)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    dims = chunk_dims(q, v, cu_seqlens)
    if offsets is None:
        offsets = checkpoint_offsets(q, cu_seqlens, interval)
    _check_dev("offsets", offsets, dev, torch.int32)
    if checkpoints is None:
        slots = int(offsets[-1].item())
        checkpoints = torch.empty((max(slots, 1), H, dk, dv), dtype=torch.float32, device=dev)
    _check_dev("checkpoints", checkpoints, dev, torch.float32)
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=q.dtype, device=dev)
    _check_dev("out", out, dev, q.dtype)
    if final_state is None:
        final_state = torch.empty((dims.num_seqs, H, dk, dv), dtype=torch.float32, device=dev)
    _check_dev("final_state", final_state, dev, torch.float32)
    st = lib().kda_chunk_fwd_checkpointed(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                          _ptr(initial_state), _ptr(cu_seqlens), _ptr(out),
                                          _ptr(final_state), _ptr(checkpoints), _ptr(offsets),
                                          int(interval), ctypes.byref(dims), _stream_handle(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_chunk_fwd_checkpointed")
    return out, final_state, checkpoints, offsets


def kda_chunk_fwd_gated(q, k, v, g, beta, gate, norm_weight=None, eps: float = 1e-6,
                        initial_state=None, cu_seqlens=None, *, out=None, final_state=None,
                        output_final_state: bool = True, stream=None):
    """kda_chunk_fwd with the KDA output gate fused into the output store:
    out = RMSNorm(o) * norm_weight * sigmoid(gate) over the value channels.

    gate: [B, T, H, dv] logits (q's dtype); norm_weight: fp32 [dv] or None.
    Returns (out [B, T, H, dv], final_state or None).
    """
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("gate", gate)):
        _check_dev(name, t, dev, q.dtype)
    _check_dev("norm_weight", norm_weight, dev, torch.float32)
    _check_dev("initial_state", initial_state, dev, torch.float32)
    _check_dev("cu_seqlens", cu_seqlens, dev, torch.int32)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if gate.shape != v.shape:
        raise ValueError("gate must be shaped like v")
    dims = chunk_dims(q, v, cu_seqlens)
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=q.dtype, device=dev)
    _check_dev("out", out, dev, q.dtype)
    if final_state is None and output_final_state:
        final_state = torch.empty((dims.num_seqs, H, dk, dv), dtype=torch.float32, device=dev)
    _check_dev("final_state", final_state, dev, torch.float32)
    st = lib().kda_chunk_fwd_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(gate),
                                   _ptr(norm_weight), ctypes.c_float(eps), _ptr(initial_state),
                                   _ptr(cu_seqlens), _ptr(out), _ptr(final_state),
                                   ctypes.byref(dims), _stream_handle(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_chunk_fwd_gated")
    return out, final_state
