"""attn_fwd_host (host buffers in and out, through the caller's device buffers) against the
device-pointer call on the same inputs: bit-identical O and lse."""
import math

import pytest
import torch

import dense_attention_forward_gb300 as attn
import workloads as wl
from dense_attention_forward_gb300 import _lib

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("pinned", [True, False])
def test_fwd_host_matches_device_call(causal, pinned):
    q, k, v = wl.make_custom(2, 3, 333, seed=97)
    out = torch.empty(q.shape, dtype=torch.bfloat16)
    lse = torch.empty(q.shape[:3], dtype=torch.float32)
    if pinned:  # every host buffer page-locked: the copies in both directions run asynchronously
        q, k, v, out, lse = (t.pin_memory() for t in (q, k, v, out, lse))
        assert all(t.is_pinned() for t in (q, k, v, out, lse))
    out, lse, _ = attn.fwd_host(q, k, v, out=out, lse=lse, causal=causal)
    torch.cuda.synchronize()
    o_ref, l_ref = attn.fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(out, o_ref.cpu()) and torch.equal(lse, l_ref.cpu())


def test_fwd_host_without_lse():
    B, H, S, D = 1, 2, 200, 128
    q, k, v = (t.pin_memory() for t in wl.make_custom(B, H, S, seed=98))
    out = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
    qd, kd, vd, od = (torch.empty(q.shape, device="cuda", dtype=torch.bfloat16) for _ in range(4))
    st = _lib.lib().attn_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), None,
                                  qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), od.data_ptr(), None,
                                  B, H, S, D, 1.0 / math.sqrt(D), 0, torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    o_ref, _ = attn.fwd(q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    assert torch.equal(out, o_ref.cpu())
    assert attn.device_status(reset=False) == 0


def test_fwd_host_caller_buffers_on_a_side_stream():
    # The caller's own device buffers and a non-default stream: everything is enqueued on that
    # stream, so synchronising it alone suffices before reading the host outputs.
    B, H, S, D = 1, 4, 700, 128
    q, k, v = (t.pin_memory() for t in wl.make_custom(B, H, S, seed=99))
    out = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
    lse = torch.empty(q.shape[:3], dtype=torch.float32).pin_memory()
    dev = tuple(torch.empty(q.shape, device="cuda", dtype=torch.bfloat16) for _ in range(4)) + (
        torch.empty(q.shape[:3], device="cuda", dtype=torch.float32),)
    side = torch.cuda.Stream()
    torch.cuda.synchronize()
    o2, l2, d2 = attn.fwd_host(q, k, v, out=out, lse=lse, dev=dev, stream=side)
    side.synchronize()
    assert o2 is out and l2 is lse and d2 is dev
    o_ref, l_ref = attn.fwd(q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    assert torch.equal(out, o_ref.cpu()) and torch.equal(lse, l_ref.cpu())
    # The device buffers hold the copied inputs and the results.
    assert torch.equal(dev[0].cpu(), q) and torch.equal(dev[3].cpu(), out) and torch.equal(dev[4].cpu(), lse)
    assert attn.device_status(reset=False) == 0
