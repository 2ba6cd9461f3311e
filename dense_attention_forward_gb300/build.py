"""Compile the CUDA sources of this package in-tree for sm_103a (no torch extension build).

Produces, next to this file:
  libattn.so          -- the product: attn_fwd and friends, the C ABI of include/attn.h
  libattn_selftest.so -- single-tile tcgen05 GEMM checks used by the GPU tests

build_trace() makes libattn_trace.so on demand (the same kernels with -DATTN_TRACE, see
include/attn_trace.h); the ordinary build does not.

Both are plain shared libraries (static CUDA runtime; the driver is loaded lazily at the
first CUDA call), so they load on a machine without a GPU.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC,-O2",
         "-I" + INCLUDE, "-I" + CSRC, "--cudart", "static"]

TARGETS = {
    "libattn.so": ["attn_fwd.cu"],
    "libattn_selftest.so": ["selftest.cu"],
}


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put /usr/local/cuda/bin on PATH)")


def _compile(target: str, sources: list[str], verbose: bool, defines: tuple = ()) -> str:
    out = os.path.join(PKG, target)
    srcs = [os.path.join(CSRC, s) for s in sources]
    deps = srcs + [os.path.join(CSRC, "ptx.cuh"), os.path.join(INCLUDE, "attn.h")]
    if os.path.exists(out) and all(os.path.getmtime(out) >= os.path.getmtime(d) for d in deps):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, *FLAGS, *defines, "-Xptxas", "-v", "-o", tmp, *srcs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if verbose or res.returncode != 0:
        sys.stderr.write(res.stdout + res.stderr)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {target}: {' '.join(cmd)}")
    os.replace(tmp, out)
    return out


def build(verbose: bool = False) -> list[str]:
    with ThreadPoolExecutor(max_workers=len(TARGETS)) as ex:
        futs = [ex.submit(_compile, t, s, verbose) for t, s in TARGETS.items()]
        return [f.result() for f in futs]


def build_trace(verbose: bool = False) -> str:
    """libattn_trace.so: libattn.so's kernels with the timeline stamps compiled in."""
    return _compile("libattn_trace.so", ["attn_fwd.cu"], verbose, ("-DATTN_TRACE",))


if __name__ == "__main__":
    for p in build(verbose="-v" in sys.argv):
        print(p)
