"""Compile the CUDA sources of this package in-tree for sm_103a (no torch extension build).

Produces, next to this file:
  libattn.so           -- the product: attn_fwd and friends, the C ABI of include/attn.h
  libattn_testhooks.so -- the same kernels with -DATTN_TEST_HOOKS: attn.h plus
                          include/attn_test_hooks.h (attn_fwd_withhold, used by the tests of the
                          bounded waits)
  libattn_trace.so     -- the same kernels with -DATTN_TRACE: attn.h plus include/attn_trace.h
                          (per-CTA timeline stamps)
  libattn_selftest.so  -- single-tile tcgen05 GEMM and softmax-helper checks for the GPU tests

All are plain shared libraries (static CUDA runtime; the driver is loaded lazily at the first
CUDA call), so they load on a machine without a GPU.

Freshness is decided by content, not by file times: each library gets a `<name>.buildhash`
file beside it holding the SHA-256 of the compiler's version line, the flags and every source
and header it depends on. A library is recompiled unless it exists and its hash file matches;
`build()` reports for each library whether it compiled it or found it up to date.
"""
from __future__ import annotations

import hashlib
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

KERNEL_SOURCES = ["attn_fwd.cu", "attn_noalloc.cu"]

# target -> (sources, extra defines)
TARGETS = {
    "libattn.so": (KERNEL_SOURCES, ()),
    "libattn_testhooks.so": (KERNEL_SOURCES, ("-DATTN_TEST_HOOKS",)),
    "libattn_trace.so": (KERNEL_SOURCES, ("-DATTN_TRACE",)),
    "libattn_selftest.so": (["selftest.cu"], ()),
}

# What the last build() / _compile() call did per library: "compiled" or "up to date".
last_status: dict[str, str] = {}


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put /usr/local/cuda/bin on PATH)")


def _nvcc_version(exe: str) -> str:
    res = subprocess.run([exe, "--version"], capture_output=True, text=True)
    lines = [ln for ln in res.stdout.splitlines() if ln.strip()]
    return lines[-1] if lines else ""


def _deps(sources: list[str]) -> list[str]:
    """The sources plus every header under csrc/ and include/ (all of them, so that a new
    include never goes unnoticed)."""
    hdrs = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h")))
    hdrs += sorted(os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h"))
    return [os.path.join(CSRC, s) for s in sources] + hdrs


def build_hash(target: str, sources: list[str], defines: tuple, exe: str, version: str) -> str:
    h = hashlib.sha256()
    h.update(version.encode() + b"\0")
    for part in (*ARCH, *FLAGS, *defines, target):
        h.update(part.replace(ROOT, "<root>").encode() + b"\0")
    for path in _deps(sources):
        h.update(os.path.relpath(path, ROOT).encode() + b"\0")
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def _compile(target: str, sources: list[str], verbose: bool, defines: tuple = (),
             version: str | None = None) -> str:
    out = os.path.join(PKG, target)
    stamp = out + ".buildhash"
    exe = nvcc()
    digest = build_hash(target, sources, defines, exe, version if version is not None else _nvcc_version(exe))
    if os.path.exists(out) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == digest:
                last_status[target] = "up to date"
                return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = [exe, *ARCH, *FLAGS, *defines, "-Xptxas", "-v", "-o", tmp, *[os.path.join(CSRC, s) for s in sources]]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if verbose or res.returncode != 0:
        sys.stderr.write(res.stdout + res.stderr)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {target}: {' '.join(cmd)}")
    os.replace(tmp, out)
    with open(stamp, "w") as f:
        f.write(digest + "\n")
    last_status[target] = "compiled"
    return out


def build(verbose: bool = False) -> list[str]:
    exe = nvcc()
    version = _nvcc_version(exe)
    with ThreadPoolExecutor(max_workers=len(TARGETS)) as ex:
        futs = [ex.submit(_compile, t, s, verbose, d, version) for t, (s, d) in TARGETS.items()]
        paths = [f.result() for f in futs]
    sys.stderr.write("build: " + ", ".join(f"{t} {last_status[t]}" for t in TARGETS) + "\n")
    return paths


def build_trace(verbose: bool = False) -> str:
    """libattn_trace.so: libattn.so's kernels with the timeline stamps compiled in."""
    s, d = TARGETS["libattn_trace.so"]
    return _compile("libattn_trace.so", s, verbose, d)


def build_test_hooks(verbose: bool = False) -> str:
    """libattn_testhooks.so: libattn.so's kernels plus attn_fwd_withhold."""
    s, d = TARGETS["libattn_testhooks.so"]
    return _compile("libattn_testhooks.so", s, verbose, d)


if __name__ == "__main__":
    for p in build(verbose="-v" in sys.argv):
        print(p)
