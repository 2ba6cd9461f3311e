"""The C ABI from plain C: tests/c_abi_client.c (CUDA runtime for memory, no PyTorch) is built
against include/attn.h and libattn.so, runs attn_fwd / attn_fwd_causal on seeded inputs
written to a file, and its outputs match the fp64 oracle."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import workloads as wl
from dense_attention_forward_gb300 import _lib
from oracle import attn_ref as ref
from tests.gpu_util import compare
from workloads import to_f64

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


@pytest.fixture(scope="module")
def client(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    _lib.lib()  # builds nothing; fails loudly if libattn.so is missing
    exe = str(tmp_path_factory.mktemp("capi") / "c_abi_client")
    pkg = os.path.dirname(_lib.LIB_PATH)
    subprocess.run([cc, "-std=c99", "-O2", os.path.join(ROOT, "tests", "c_abi_client.c"),
                    "-I" + os.path.join(ROOT, "include"), "-I" + os.path.join(CUDA, "include"),
                    "-L" + pkg, "-lattn", "-L" + os.path.join(CUDA, "lib64"), "-lcudart",
                    "-Wl,-rpath," + pkg + ":" + os.path.join(CUDA, "lib64"), "-o", exe], check=True)
    return exe


@pytest.mark.parametrize("causal", [0, 1])
def test_c_client_matches_oracle(client, tmp_path, causal):
    B, H, S = 2, 3, 300
    q, k, v = wl.make_custom(B, H, S, seed=95 + causal)
    inp, out = tmp_path / "in.bin", tmp_path / "out.bin"
    with open(inp, "wb") as f:
        f.write(np.array([B, H, S, causal], dtype=np.int32).tobytes())
        for t in (q, k, v):
            f.write(t.contiguous().view(torch.int16).numpy().tobytes())
    r = subprocess.run([client, str(inp), str(out)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    raw = np.fromfile(out, dtype=np.uint8)
    n = B * H * S * 128
    o_bits = raw[:2 * n].view(np.int16).reshape(B, H, S, 128)
    o = torch.from_numpy(o_bits.copy()).view(torch.bfloat16).double().numpy()
    lse = raw[2 * n:].view(np.float32).reshape(B, H, S).astype(np.float64)
    o_ref, lse_ref = ref.attention(to_f64(q), to_f64(k), to_f64(v), 1.0 / np.sqrt(128), causal=bool(causal))
    compare(o, lse, o_ref, lse_ref)
