"""Build libkda.so in-tree for sm_103a (nvcc, no cmake).

Each .cu under csrc/ compiles to its own object in parallel; the objects link
into ``libkda.so`` beside this file.  The CUDA runtime is linked statically and
the driver API is reached through ``cudaGetDriverEntryPointByVersion``, so the
library loads on a machine without a GPU driver (it only needs one to run).
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libkda.so")
LIB_DEBUG = os.path.join(HERE, "libkda_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-Xptxas", "-v"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    hs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return sorted(hs)


def _digest(paths, extra=""):
    h = hashlib.sha256(extra.encode())
    for p in paths:
        h.update(p.encode())
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def build(verbose: bool = False, force: bool = False, debug: bool = False) -> str:
    """Compile csrc/*.cu for sm_103a and link libkda.so; returns its path.

    debug=True builds libkda_debug.so instead (objects in _build_debug/): the same kernels with
    KDA_DEBUG_CHECKS defined, so that every chunk forward and decode call first checks g and the
    packed offsets on the device (kda_debug_checks, kda_device_status)."""
    build_dir = BUILD + "_debug" if debug else BUILD
    lib_path = LIB_DEBUG if debug else LIB
    flags = NVCC_FLAGS + (["-DKDA_DEBUG_CHECKS=1"] if debug else [])
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()
    srcs = _sources()
    hdr_digest = _digest(_headers(), " ".join(ARCH + flags))
    stamp = os.path.join(build_dir, "stamp")
    want = _digest(srcs, hdr_digest)
    if not force and os.path.exists(lib_path) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read() == want:
                return lib_path

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *flags, "-I", INCLUDE, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        with open(obj + ".log", "w") as f:
            f.write(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    with open(stamp, "w") as f:
        f.write(want)
    if verbose:
        for o in objs:
            with open(o + ".log") as f:
                sys.stdout.write(f.read())
    return lib_path


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv, debug="--debug" in sys.argv))
