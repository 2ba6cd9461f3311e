"""attn_fwd_host_noalloc: the host-to-host call for callers that cannot allocate device memory.

Some callers may not call cudaMalloc (another allocator owns the device memory of their
process, or allocations are forbidden where they run), so they cannot provide the device
buffers attn_fwd_host stages through. attn_fwd_host_noalloc stages through a fixed array the
library holds instead. These tests call it through the C ABI and compare it with attn_fwd_host
on the same inputs, twice in a row, so that the second call runs over the first call's leftover
contents of the shared array. (The file name makes pytest collect it last.)"""
import ctypes
import math
import os
import re

import numpy as np
import pytest
import torch

import dense_attention_forward_gb300 as attn
import workloads as wl
from dense_attention_forward_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# Parity tolerances of the GPU tests (O: 1.5e-2 absolute, lse: 1e-3 absolute).
O_TOL, LSE_TOL = 1.5e-2, 1e-3


def noalloc(q, k, v, out, lse, scale, causal, stream):
    """Direct C-ABI call; returns the status code."""
    B, H, S, D = q.shape
    return _lib.lib().attn_fwd_host_noalloc(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
        lse.data_ptr() if lse is not None else None, B, H, S, D, scale, causal, stream)


def test_header_and_binding_agree_on_the_limit():
    text = open(os.path.join(ROOT, "include", "attn.h")).read()
    assert int(re.search(r"#define ATTN_NOALLOC_MAX_ROWS (\d+)", text).group(1)) == _lib.NOALLOC_MAX_ROWS


@pytest.mark.parametrize("B,H,S,expected", [
    (1, 1, 32769, 1), (2, 16, 1025, 1), (1 << 20, 1 << 10, 4096, 1),  # beyond the array
    (0, 1, 256, 1), (1, 1, 0, 1),
])
def test_sizes_beyond_the_array_are_rejected_first(B, H, S, expected):
    # Rejected before any CUDA call (fake host addresses, never read).
    h = 0x61000000
    assert _lib.lib().attn_fwd_host_noalloc(h, h + 0x1000000, h + 0x2000000, h + 0x3000000, None,
                                            B, H, S, 128, 0.088, 0, None) == expected


def test_without_a_device():
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = 0x61000000
    assert _lib.lib().attn_fwd_host_noalloc(h, h + 0x1000000, h + 0x2000000, h + 0x3000000, None,
                                            1, 2, 300, 128, 0.088, 0, None) == 4
    assert _lib.lib().attn_fwd_host_noalloc(h, h, h, h, None, 1, 2, 300, 64, 0.088, 0, None) == 2


@pytest.mark.gpu
def test_noalloc_matches_host_entry_twice_in_a_row():
    stream = torch.cuda.current_stream()
    cases = [
        # (B, H, S, causal, seed): the second call is smaller, so the shared array still holds
        # the first call's data beyond it.
        (2, 4, 1000, 0, 201),
        (1, 3, 517, 1, 202),
    ]
    for B, H, S, causal, seed in cases:
        assert B * H * S <= _lib.NOALLOC_MAX_ROWS
        q, k, v = wl.make_custom(B, H, S, seed=seed)
        scale = 1.0 / math.sqrt(128)
        out = torch.full((B, H, S, 128), float("nan"), dtype=torch.bfloat16)
        lse = torch.full((B, H, S), float("nan"), dtype=torch.float32)
        assert noalloc(q, k, v, out, lse, scale, causal, stream.cuda_stream) == 0
        stream.synchronize()
        o_ref, l_ref, _ = attn.fwd_host(q, k, v, scale, causal=bool(causal))
        torch.cuda.synchronize()
        o_err = (out.double() - o_ref.double()).abs().max().item()
        l_err = (lse.double() - l_ref.double()).abs().max().item()
        assert np.isfinite(o_err) and o_err <= O_TOL, (B, H, S, o_err)
        assert np.isfinite(l_err) and l_err <= LSE_TOL, (B, H, S, l_err)
        # The same kernel on the same inputs: in fact bit for bit.
        assert torch.equal(out, o_ref) and torch.equal(lse, l_ref)
    # Without lse, and the size limit on a device: rejected, nothing enqueued.
    q, k, v = wl.make_custom(1, 2, 300, seed=203)
    out = torch.empty(q.shape, dtype=torch.bfloat16)
    assert noalloc(q, k, v, out, None, 0.088, 0, stream.cuda_stream) == 0
    stream.synchronize()
    o_ref, _, _ = attn.fwd_host(q, k, v, 0.088)
    torch.cuda.synchronize()
    assert torch.equal(out, o_ref)
    big = torch.empty(1, 1, _lib.NOALLOC_MAX_ROWS + 1, 128, dtype=torch.bfloat16)
    assert noalloc(big, big, big, big, None, 0.088, 0, stream.cuda_stream) == 1
    assert attn.device_status(reset=False) == 0
