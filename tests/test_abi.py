"""libkda loads without a GPU, exports every symbol include/kda.h declares, and
rejects bad arguments on the host before anything is launched.

None of these calls reaches a kernel: each one fails validation first, so they
run on a machine without a GPU (the pointers are never dereferenced).
"""
import ctypes
import os
import re

import pytest

from linear_attention_fwd_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


@pytest.fixture(scope="module")
def K():
    kbuild.build()
    from linear_attention_fwd_gb300 import kda
    kda.lib()
    return kda


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(K):
    names = declared_functions()
    assert set(names) == set(K.EXPORTED), names
    for n in names:
        assert hasattr(K.lib(), n), n


def test_status_strings(K):
    for code in range(9):
        s = K.kda_status_string(code)
        assert s and s != "unknown status"
    assert K.kda_status_string(99) == "unknown status"


FAKE = 1 << 20          # 16-byte aligned, never dereferenced (validation fails first)


def dims(**kw):
    from linear_attention_fwd_gb300.kda import KdaDims
    d = dict(batch=2, seqlen=100, num_seqs=2, heads=4, dk=128, dv=128, dtype=1)
    d.update(kw)
    return KdaDims(**d)


def call_chunk(K, d, impl=0, q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, s0=None, cu=None,
               out=FAKE, sT=None):
    vp = ctypes.c_void_p
    args = [vp(x) if x is not None else None for x in (q, k, v, g, beta, s0, cu, out, sT)]
    dp = ctypes.byref(d) if d is not None else None
    return K.lib().kda_chunk_fwd_with(impl, *args, dp, None)


@pytest.mark.parametrize("kw,code", [
    (dict(dk=96), 3), (dict(dv=32), 3), (dict(dtype=7), 3),
    (dict(heads=0), 2), (dict(batch=0), 2), (dict(seqlen=-1), 2), (dict(num_seqs=3), 2),
])
def test_chunk_rejects_bad_dims(K, kw, code):
    assert call_chunk(K, dims(**kw)) == code


def test_chunk_rejects_null_and_misaligned(K):
    assert call_chunk(K, None) == K.KDA_ERR_NULL
    assert call_chunk(K, dims(), q=None) == K.KDA_ERR_NULL
    assert call_chunk(K, dims(), out=None) == K.KDA_ERR_NULL
    assert call_chunk(K, dims(), v=FAKE + 8) == K.KDA_ERR_ALIGN
    assert call_chunk(K, dims(), s0=FAKE + 4) == K.KDA_ERR_ALIGN
    assert call_chunk(K, dims(), beta=FAKE + 1) == K.KDA_ERR_ALIGN
    # packed sequences need batch == 1
    assert call_chunk(K, dims(batch=2, num_seqs=5), cu=FAKE) == K.KDA_ERR_SHAPE
    # partially overlapping initial / final states
    assert call_chunk(K, dims(), s0=FAKE, sT=FAKE + 4096) == K.KDA_ERR_SHAPE
    # unknown kernel choice
    assert call_chunk(K, dims(), impl=9) == K.KDA_ERR_UNSUPPORTED


def call_ckpt(K, d, ck=FAKE, off=FAKE, interval=512, q=FAKE):
    vp = ctypes.c_void_p
    a = [vp(x) if x is not None else None
         for x in (q, FAKE, FAKE, FAKE, FAKE, None, None, FAKE, None, ck, off)]
    return K.lib().kda_chunk_fwd_checkpointed(*a, interval, ctypes.byref(d) if d is not None else None,
                                              None)


def test_checkpointed_validation(K):
    assert call_ckpt(K, dims(), ck=None) == K.KDA_ERR_NULL
    assert call_ckpt(K, dims(), off=None) == K.KDA_ERR_NULL
    assert call_ckpt(K, dims(), interval=0) == K.KDA_ERR_SHAPE
    assert call_ckpt(K, dims(), interval=100) == K.KDA_ERR_SHAPE   # not a multiple of 64
    assert call_ckpt(K, dims(), ck=FAKE + 4) == K.KDA_ERR_ALIGN
    assert call_ckpt(K, dims(), off=FAKE + 2) == K.KDA_ERR_ALIGN
    assert call_ckpt(K, dims(), q=None) == K.KDA_ERR_NULL          # the usual chunk checks run


def call_gated(K, d, gate=FAKE, w=None, eps=1e-6, q=FAKE):
    vp = ctypes.c_void_p
    a = [vp(x) if x is not None else None for x in (q, FAKE, FAKE, FAKE, FAKE, gate, w)]
    b = [vp(x) if x is not None else None for x in (None, None, FAKE, None)]
    return K.lib().kda_chunk_fwd_gated(*a, ctypes.c_float(eps), *b,
                                       ctypes.byref(d) if d is not None else None, None)


def test_gated_validation(K):
    assert call_gated(K, dims(), gate=None) == K.KDA_ERR_NULL
    assert call_gated(K, dims(), eps=-1.0) == K.KDA_ERR_SHAPE
    assert call_gated(K, dims(), eps=float("nan")) == K.KDA_ERR_SHAPE
    assert call_gated(K, dims(), gate=FAKE + 2) == K.KDA_ERR_ALIGN
    assert call_gated(K, dims(), w=FAKE + 2) == K.KDA_ERR_ALIGN
    assert call_gated(K, dims(), q=None) == K.KDA_ERR_NULL          # the usual chunk checks run


def test_tc_kernel_refuses_shapes_it_does_not_cover(K):
    assert call_chunk(K, dims(dtype=0), impl=2) == K.KDA_ERR_UNSUPPORTED   # fp32
    assert call_chunk(K, dims(dk=96), impl=2) == K.KDA_ERR_UNSUPPORTED     # not a supported head size


def test_selected_impl(K):
    sel = K.lib().kda_chunk_fwd_selected_impl
    assert sel(ctypes.byref(dims(dtype=0))) == 1           # fp32 -> SIMT kernel
    assert sel(ctypes.byref(dims(dtype=0, dk=64, dv=64))) == 1
    assert sel(ctypes.byref(dims(dk=64, dv=64))) == 2      # bf16 64-wide heads -> tensor cores, padded
    assert sel(ctypes.byref(dims(dk=64, dv=128))) == 2
    assert sel(ctypes.byref(dims(dk=96))) == -1
    assert sel(ctypes.byref(dims())) in (1, 2)


def call_step(K, d, q=FAKE, state=FAKE, idx=None, beta=FAKE, out=FAKE):
    vp = ctypes.c_void_p
    a = [vp(x) if x is not None else None for x in (q, FAKE, FAKE, FAKE, beta, state, idx, out)]
    return K.lib().kda_recurrent_step(*a, ctypes.byref(d) if d is not None else None, None)


def test_recurrent_step_validation(K):
    d1 = lambda **kw: dims(**{**dict(batch=8, seqlen=1, num_seqs=8), **kw})
    assert call_step(K, None) == K.KDA_ERR_NULL
    assert call_step(K, d1(seqlen=2)) == K.KDA_ERR_SHAPE
    assert call_step(K, d1(num_seqs=4)) == K.KDA_ERR_SHAPE     # pool smaller than rows
    assert call_step(K, d1(dk=48)) == K.KDA_ERR_UNSUPPORTED
    assert call_step(K, d1(), state=None) == K.KDA_ERR_NULL
    assert call_step(K, d1(), q=FAKE + 2) == K.KDA_ERR_ALIGN
    assert call_step(K, d1(), idx=FAKE + 2) == K.KDA_ERR_ALIGN
    assert call_step(K, d1(batch=0)) == K.KDA_OK                # no rows: nothing to do


def call_steps(K, d, q=FAKE, state=FAKE, idx=None, num=None, out=FAKE, update=1):
    vp = ctypes.c_void_p
    a = [vp(x) if x is not None else None for x in (q, FAKE, FAKE, FAKE, FAKE, state, idx, num, out)]
    return K.lib().kda_recurrent_steps(*a, update, ctypes.byref(d) if d is not None else None, None)


def test_recurrent_steps_validation(K):
    d1 = lambda **kw: dims(**{**dict(batch=8, seqlen=4, num_seqs=8), **kw})
    assert call_steps(K, None) == K.KDA_ERR_NULL
    assert call_steps(K, d1(seqlen=0)) == K.KDA_ERR_SHAPE
    assert call_steps(K, d1(num_seqs=4)) == K.KDA_ERR_SHAPE    # pool smaller than rows
    assert call_steps(K, d1(dv=80)) == K.KDA_ERR_UNSUPPORTED
    assert call_steps(K, d1(), state=None) == K.KDA_ERR_NULL
    assert call_steps(K, d1(), q=FAKE + 4) == K.KDA_ERR_ALIGN
    assert call_steps(K, d1(), num=FAKE + 2) == K.KDA_ERR_ALIGN
    assert call_steps(K, d1(), out=FAKE + 8) == K.KDA_ERR_ALIGN
    assert call_steps(K, d1(batch=0)) == K.KDA_OK                # no rows: nothing to do
    assert call_steps(K, d1(), out=None, update=0) == K.KDA_OK   # nothing to write


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    from linear_attention_fwd_gb300 import kda
    monkeypatch.setattr(kda, "_lib", None)
    monkeypatch.setattr(kda, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        kda.lib()


def test_cta_count_the_library_picks(K):
    # dense: the balanced schedule over min(SMs, units x chunks) CTAs; packed with fewer units than
    # twice the SMs: the same over min(SMs, heads x (ceil(tokens / 64) + sequences)), a bound on
    # the items the device counts; packed with more: one CTA per unit
    f = K.kda_chunk_fwd_auto_ctas
    assert f(dims(batch=4, seqlen=8192, num_seqs=4, heads=32), False, 152) == 152     # 128 units
    assert f(dims(batch=1, seqlen=65536, num_seqs=1, heads=64), False, 152) == 152
    assert f(dims(batch=1, seqlen=1100, num_seqs=1, heads=1), False, 152) == 18       # 18 chunks
    assert f(dims(batch=2, seqlen=64, num_seqs=2, heads=3), False, 152) == 6
    assert f(dims(batch=1, seqlen=65536, num_seqs=1, heads=64), True, 152) == 152
    assert f(dims(batch=1, seqlen=1100, num_seqs=1, heads=1), True, 152) == 19        # 18 chunks + 1
    assert f(dims(batch=1, seqlen=100, num_seqs=3, heads=2), True, 152) == 2 * (2 + 3)
    assert f(dims(batch=1, seqlen=2**20, num_seqs=16, heads=32), True, 152) == 512    # 512 units >= 2 x 152
    assert f(dims(batch=1, seqlen=2**20, num_seqs=16, heads=32), True, 400) == 256    # at most 256
    # 64-wide bf16 heads run on the tensor-core kernel too; it does not run fp32; empty, invalid
    # dims and SM counts give 0
    assert f(dims(batch=1, seqlen=65536, num_seqs=1, heads=4, dk=64, dv=64), False, 152) == 152
    assert f(dims(batch=1, seqlen=65536, num_seqs=1, heads=4, dtype=0), False, 152) == 0
    assert f(dims(batch=1, seqlen=65536, num_seqs=1, heads=0), False, 152) == 0
    assert f(dims(batch=1, seqlen=0, num_seqs=1, heads=4), False, 152) == 0
    assert f(dims(batch=1, seqlen=65536, num_seqs=1, heads=4), False, 0) == 0


def test_segment_count_argument_is_checked(K):
    # segments outside [0, 64] are refused before any launch
    vp = ctypes.c_void_p
    d = dims()
    for bad in (-1, 65):
        st = K.lib().kda_chunk_fwd_segmented(2, *[vp(FAKE)] * 5, None, None, vp(FAKE), None,
                                             ctypes.c_int32(bad), ctypes.byref(d), None)
        assert st == 2   # KDA_ERR_SHAPE


def test_noalloc_limit_and_rejection(K):
    # the binding's copy of the scratch limit is the header's
    src = open(HEADER).read()
    m = re.search(r"#define KDA_NOALLOC_SCRATCH_BYTES \(\(size_t\)(\d+) << (\d+)\)", src)
    assert m and int(m.group(1)) << int(m.group(2)) == K.NOALLOC_SCRATCH_BYTES
    vp = ctypes.c_void_p
    args = [vp(FAKE)] * 5 + [None, None, vp(FAKE), None]
    assert K.lib().kda_chunk_fwd_noalloc(*args, None, None) == K.KDA_ERR_NULL
    # a workspace above the limit is rejected on the host, before the device is touched
    big = dims(batch=1, seqlen=1 << 20, num_seqs=1, heads=32)
    assert K.lib().kda_chunk_fwd_workspace_bytes(ctypes.byref(big)) > K.NOALLOC_SCRATCH_BYTES
    assert K.lib().kda_chunk_fwd_noalloc(*args, ctypes.byref(big), None) == K.KDA_ERR_WORKSPACE


def test_debug_build_reports_its_checks(K):
    # the release library runs no device-side input check; the debug build (separate objects,
    # libkda_debug.so) runs both, and exports the same symbols
    assert K.kda_debug_checks() == 0
    path = kbuild.build(debug=True)
    assert path.endswith("libkda_debug.so")
    dbg = ctypes.CDLL(path)
    dbg.kda_debug_checks.restype = ctypes.c_int
    assert dbg.kda_debug_checks() == 3
    for n in declared_functions():
        assert hasattr(dbg, n), n
    dbg.kda_status_string.restype = ctypes.c_char_p
    assert b"debug-build" in dbg.kda_status_string(K.KDA_ERR_INPUT)


def test_qknorm_validation(K):
    # the fused normalisation's epsilon is checked before anything else; the rest of each
    # call's checks are those of the call it extends
    vp, L = ctypes.c_void_p, K.lib()

    def chunk(eps, q=FAKE, d=None):
        d = dims() if d is None else d
        a = [vp(x) if x is not None else None for x in (q, FAKE, FAKE, FAKE, FAKE)]
        return L.kda_chunk_fwd_qknorm(*a, ctypes.c_float(eps), None, None, vp(FAKE), None,
                                      ctypes.byref(d), None)

    def step(eps, q=FAKE):
        d = dims(batch=8, seqlen=1, num_seqs=8)
        a = [vp(x) if x is not None else None for x in (q, FAKE, FAKE, FAKE, FAKE)]
        return L.kda_recurrent_step_qknorm(*a, ctypes.c_float(eps), vp(FAKE), None, vp(FAKE),
                                           ctypes.byref(d), None)

    def steps(eps, q=FAKE):
        d = dims(batch=8, seqlen=4, num_seqs=8)
        a = [vp(x) if x is not None else None for x in (q, FAKE, FAKE, FAKE, FAKE)]
        return L.kda_recurrent_steps_qknorm(*a, ctypes.c_float(eps), vp(FAKE), None, None,
                                            vp(FAKE), 1, ctypes.byref(d), None)

    for f in (chunk, step, steps):
        for bad in (-1.0, float("nan"), float("inf")):
            assert f(bad) == K.KDA_ERR_SHAPE, (f.__name__, bad)
        assert f(1e-6, q=None) == K.KDA_ERR_NULL, f.__name__
        assert f(1e-6, q=FAKE + 2) == K.KDA_ERR_ALIGN, f.__name__
    assert chunk(1e-6, d=dims(dk=96)) == K.KDA_ERR_UNSUPPORTED
