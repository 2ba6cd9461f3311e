"""Unit checks of the kernel's PTX helpers on the GPU: single-tile tcgen05 GEMMs through the
three operand forms the attention kernel uses (against PyTorch fp32 matmul of the same BF16
values), and the softmax's per-element helpers (against exact host values)."""
import pytest
import torch

from dense_attention_forward_gb300 import _lib

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_single_tile_gemm(mode):
    g = torch.Generator().manual_seed(100 + mode)
    a = torch.randn(128, 128, generator=g).to(torch.bfloat16).cuda()
    b = torch.randn(128, 128, generator=g).to(torch.bfloat16).cuda()
    c = torch.full((128, 128), float("nan"), device="cuda")
    st = _lib.selftest_lib().attn_selftest_gemm(a.data_ptr(), b.data_ptr(), c.data_ptr(), mode, None)
    assert st == 0
    torch.cuda.synchronize()
    want = a.float() @ (b.float().t() if mode == 0 else b.float())
    err = (c - want).abs().max().item()
    assert err < 1e-3, (mode, err)


def test_elementwise_helpers():
    """The softmax's per-element helpers against exact host values: MUFU 2^x (flushing results
    below 2^-126 to zero, 2^0 exactly 1), BF16 packing with round-to-nearest-even (bit for bit
    against PyTorch's conversion), exact widening back to fp32, and the three-input max."""
    import numpy as np
    rng = np.random.default_rng(7)
    x = np.concatenate([
        -rng.random(200000) * 140.0,                   # 2^x over [-140, 0], across the flush point
        rng.standard_normal(100000) * 4.0,
        np.array([0.0, -0.0, 1.0, 8.0, -1.0, -126.0, -127.5, -150.0, -np.inf, 0.5, -0.5]),
        # BF16 halfway cases: 1 + 2^-8 (ties to 1.0), 1 + 3 * 2^-8 (ties to 1 + 2^-6)
        np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8)]),
    ]).astype(np.float32)
    y = (rng.standard_normal(x.size) * 100.0).astype(np.float32)
    xd, yd = torch.from_numpy(x).cuda(), torch.from_numpy(y).cuda()
    u = torch.zeros(x.size, dtype=torch.int32, device="cuda")
    f = torch.zeros(4 * x.size, dtype=torch.float32, device="cuda")
    st = _lib.selftest_lib().attn_selftest_elementwise(xd.data_ptr(), yd.data_ptr(), u.data_ptr(), f.data_ptr(),
                                                       x.size, None)
    assert st == 0
    torch.cuda.synchronize()
    f = f.cpu().numpy().reshape(-1, 4)
    u = u.cpu().numpy().view(np.uint32)

    ref = np.exp2(x.astype(np.float64))
    normal = ref >= 2.0 ** -126
    rel = np.abs(f[normal, 0] - ref[normal]) / ref[normal]
    assert rel.max() < 2.0 ** -20, rel.max()
    assert np.all(f[x < -126.0, 0] == 0.0)
    assert f[np.where(x == 0.0)[0], 0].tolist() == [1.0, 1.0]

    bits = lambda a: torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    want = (bits(y).astype(np.uint32) << 16) | bits(x).astype(np.uint32)
    assert np.array_equal(u, want)
    widen = lambda a: torch.from_numpy(a).to(torch.bfloat16).float().numpy()  # noqa: E731
    assert np.array_equal(f[:, 1], widen(x)) and np.array_equal(f[:, 2], widen(y))
    assert np.array_equal(f[:, 3], np.maximum(np.maximum(x, y), -x))
