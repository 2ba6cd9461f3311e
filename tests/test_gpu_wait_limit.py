"""The kernel's bounded waits, made to run out on purpose.

attn_fwd_withhold (test-hook build, libattn_testhooks.so) runs the dense kernel with its TMA
producer skipping one K/V token, a barrier phase that nothing completes. The waits that need it
must give up after about two seconds, record the status word (0xA77E0000 | role << 8 |
barrier), drain, free tensor memory and exit, leaving the context usable. No fault, trap or
endless wait is involved: every CTA leaves by its own bounded waits."""
import ctypes
import time

import numpy as np
import pytest
import torch

import dense_attention_forward_gb300 as attn
import workloads as wl
from dense_attention_forward_gb300 import _lib
from dense_attention_forward_gb300 import build as _build
from gpu_util import compare, full_parity
from oracle import attn_ref as ref
from workloads import to_f64

pytestmark = pytest.mark.gpu

ROLES = {1: "TMA producer", 2: "MMA issue", 3: "softmax", 4: "O correction"}


@pytest.fixture(scope="module")
def hooks():
    _build.build_test_hooks()
    return _lib.test_hooks_lib()


def status_word(h, reset):
    """The test-hook library's own device status word (each library holds its own)."""
    w = ctypes.c_uint(0)
    assert h.attn_device_status(ctypes.byref(w), 1 if reset else 0) == 0
    return w.value


# Token 0 (K tile 0) is waited on before the first QK; token 5 (V tile 2) inside the loop,
# after two tiles of normal work; token 6 (K tile 3, the last K tile of S = 512) by the last QK.
@pytest.mark.parametrize("token", [0, 5, 6])
def test_withheld_token_gives_up_cleanly(hooks, token):
    torch.cuda.synchronize()
    assert status_word(hooks, reset=True) == 0
    B, H, S = 1, 2, 512  # 4 CTAs, 4 K/V tiles each
    q, k, v = wl.make_custom(B, H, S, seed=70 + token)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o = torch.empty_like(qd)
    lse = torch.empty(B, H, S, device="cuda", dtype=torch.float32)
    scale = 1.0 / np.sqrt(128)
    stream = torch.cuda.current_stream().cuda_stream
    t0 = time.monotonic()
    st = hooks.attn_fwd_withhold(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(),
                                 lse.data_ptr(), B, H, S, 128, scale, token, stream)
    assert st == 0
    torch.cuda.synchronize()
    elapsed = time.monotonic() - t0
    word = status_word(hooks, reset=False)
    assert word >> 16 == 0xA77E, hex(word)
    assert (word >> 8) & 0xFF in ROLES, hex(word)
    assert (word & 0xFF) < 20, hex(word)  # 18 mbarriers, then the two S-seen counts
    assert status_word(hooks, reset=True) == word
    assert status_word(hooks, reset=False) == 0  # cleared
    assert 1.5 < elapsed < 30.0, elapsed
    # The context is intact: the same library's ordinary call on the same inputs matches the
    # oracle and no wait gives up; so does the product library's.
    assert hooks.attn_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), lse.data_ptr(),
                          B, H, S, 128, scale, stream) == 0
    torch.cuda.synchronize()
    o_ref, lse_ref = ref.attention(to_f64(q), to_f64(k), to_f64(v), scale)
    compare(to_f64(o.float().cpu()), lse.double().cpu().numpy(), o_ref, lse_ref)
    assert status_word(hooks, reset=False) == 0
    full_parity(q, k, v, scale)
    torch.cuda.synchronize()
    assert attn.device_status(reset=False) == 0



def test_withheld_token_with_several_items_per_cta(hooks):
    # 160 heads x 1 item: more items than SMs, so some CTAs walk two items. V tile 0 of every
    # CTA's first item never arrives; every CTA still gives up within its bounded waits, and the
    # next ordinary calls (the test-hook and the product library) match the oracle.
    torch.cuda.synchronize()
    assert status_word(hooks, reset=True) == 0
    B, H, S = 1, 160, 256
    q, k, v = wl.make_custom(B, H, S, seed=80)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o = torch.empty_like(qd)
    lse = torch.empty(B, H, S, device="cuda", dtype=torch.float32)
    scale = 1.0 / np.sqrt(128)
    stream = torch.cuda.current_stream().cuda_stream
    t0 = time.monotonic()
    assert hooks.attn_fwd_withhold(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                   B, H, S, 128, scale, 1, stream) == 0
    torch.cuda.synchronize()
    assert 1.5 < time.monotonic() - t0 < 30.0
    word = status_word(hooks, reset=True)
    assert word >> 16 == 0xA77E and (word >> 8) & 0xFF in ROLES, hex(word)
    assert hooks.attn_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), lse.data_ptr(),
                          B, H, S, 128, scale, stream) == 0
    torch.cuda.synchronize()
    o_ref, lse_ref = ref.attention(to_f64(q), to_f64(k), to_f64(v), scale)
    compare(to_f64(o.float().cpu()), lse.double().cpu().numpy(), o_ref, lse_ref)
    assert status_word(hooks, reset=False) == 0
    full_parity(q, k, v, scale)
    assert attn.device_status(reset=False) == 0
