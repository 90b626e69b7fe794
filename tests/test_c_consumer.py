"""include/kda.h from plain C: a C99 program compiled with gcc against the header and linked
against libkda.so calls the host-only entry points (no GPU needed: every call below returns
before anything reaches the device) and checks their results.  This pins the header as valid
C and the exported symbols as callable with the declared C types."""
import os
import shutil
import subprocess

import pytest

from linear_attention_fwd_gb300 import build as kbuild

C_SRC = r"""
#include <stdio.h>
#include <string.h>
#include "kda.h"

int main(void) {
    kda_dims_t d;
    int bad = 0;
    if (strcmp(kda_status_string(KDA_OK), "ok") != 0) bad |= 1;
    if (kda_chunk_fwd(0, 0, 0, 0, 0, 0, 0, 0, 0, NULL, 0) != KDA_ERR_NULL) bad |= 2;
    d.batch = 1; d.seqlen = 65536; d.num_seqs = 1; d.heads = 64; d.dk = 128; d.dv = 128;
    d.dtype = KDA_BF16;
    if (kda_chunk_fwd_selected_impl(&d) != KDA_IMPL_TC) bad |= 4;
    if (kda_chunk_fwd_auto_ctas(&d, 0, 152) != 152 || kda_chunk_fwd_auto_ctas(&d, 1, 152) != 152) bad |= 8;
    d.dtype = KDA_F32; d.dk = 64; d.dv = 64;
    if (kda_chunk_fwd_selected_impl(&d) != KDA_IMPL_SIMT) bad |= 16;
    d.heads = 0;   /* non-positive dimensions are refused on the host */
    if (kda_chunk_fwd(0, 0, 0, 0, 0, 0, 0, 0, 0, &d, 0) != KDA_ERR_SHAPE) bad |= 32;
    if (kda_chunk_fwd_segmented(KDA_IMPL_AUTO, 0, 0, 0, 0, 0, 0, 0, 0, 0, 65, &d, 0) != KDA_ERR_SHAPE)
        bad |= 64;
    printf("bad=%d\n", bad);
    return bad;
}
"""


def _cuda_include():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "include")
    return inc if os.path.exists(os.path.join(inc, "cuda_runtime_api.h")) else None


def test_header_compiles_as_c99_and_the_library_links(tmp_path):
    gcc = shutil.which("gcc")
    inc = _cuda_include()
    if gcc is None or inc is None:
        pytest.skip("gcc or the CUDA headers are not available")
    lib = kbuild.build()
    src = tmp_path / "consumer.c"
    src.write_text(C_SRC)
    exe = tmp_path / "consumer"
    libdir = os.path.dirname(lib)
    subprocess.check_call([gcc, "-std=c99", "-Wall", "-Werror", "-I", kbuild.INCLUDE, "-I", inc,
                           str(src), "-o", str(exe), lib, "-Wl,-rpath," + libdir])
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "bad=0" in r.stdout
