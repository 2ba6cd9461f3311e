"""Single-tile tcgen05 GEMMs through the three operand forms the attention kernel uses,
against PyTorch fp32 matmul of the same BF16 values."""
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
