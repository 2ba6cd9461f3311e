"""Numerical edge cases of the CUDA path: extreme softmax scales, huge scores, and two exact
invariants of the kernel's arithmetic (bit for bit, no tolerance): scaling V by a power of
two scales O by the same power, and permuting the query rows permutes the output rows."""
import numpy as np
import pytest
import torch

import dense_attention_forward_gb300 as attn
import workloads as wl
from oracle import attn_ref as ref
from tests.gpu_util import compare, full_parity, run_gpu
from workloads import to_f64

pytestmark = pytest.mark.gpu


def test_tiny_scale_nearly_uniform():
    # scale 1e-3: every row's weights are within 1 % of uniform; O is close to the mean of V.
    q, k, v = wl.make_custom(1, 3, 700, seed=81)
    full_parity(q, k, v, 1e-3)
    o, _ = run_gpu(q, k, v, 1e-3)
    assert np.max(np.abs(o - to_f64(v).mean(axis=2, keepdims=True))) < 0.05


@pytest.mark.parametrize("thr", [0, 1, 8])
def test_large_scale_nearly_one_hot(thr):
    # Q, K x2 and scale 1: score spread ~45 per row, so almost every row is dominated by one key.
    q, k, v = wl.make_custom(1, 2, 600, seed=82, qk_gain=2.0)
    full_parity(q, k, v, 1.0, thr)


@pytest.mark.parametrize("causal", [False, True])
def test_large_scores_parity(causal):
    # Q, K x4 (scores std ~16 after the 1/sqrt(128) scale): the max trick keeps every row finite.
    q, k, v = wl.make_custom(1, 2, 530, seed=83, qk_gain=4.0)
    full_parity(q, k, v, 1.0 / np.sqrt(128), 0, causal=causal)


def test_huge_scores_stay_finite():
    # Q, K x16: scores of several hundred. O stays a convex combination of V rows and lse
    # follows the oracle to fp32 relative precision.
    q, k, v = wl.make_custom(1, 2, 300, seed=84, qk_gain=16.0)
    o, lse = run_gpu(q, k, v, 1.0 / np.sqrt(128))
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    vf = to_f64(v)
    assert np.all(o <= vf.max(axis=2, keepdims=True) + 1e-2)
    assert np.all(o >= vf.min(axis=2, keepdims=True) - 1e-2)
    _, lse_ref = ref.attention(to_f64(q), to_f64(k), vf, 1.0 / np.sqrt(128))
    assert np.max(np.abs(lse - lse_ref) / np.abs(lse_ref)) < 1e-4


@pytest.mark.parametrize("e", [-6, 5])
def test_v_power_of_two_scaling_is_exact(e):
    # P does not depend on V, and every product, sum, the 1/l scaling and the BF16 rounding
    # commute with multiplication by 2^e (no overflow or subnormals here): O scales exactly.
    q, k, v = wl.make_custom(2, 2, 333, seed=85)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o1, l1 = attn.fwd(qd, kd, vd)
    o2, l2 = attn.fwd(qd, kd, vd * (2.0 ** e))
    torch.cuda.synchronize()
    assert torch.equal(o2, o1 * (2.0 ** e))
    assert torch.equal(l1, l2)


def test_query_permutation_is_exact():
    # Rows are computed independently of their position in the tile (dense attention; under
    # the causal mask a row's keys depend on its position): a permutation of the query rows
    # permutes the output rows bit for bit.
    q, k, v = wl.make_custom(1, 2, 400, seed=86)
    perm = torch.randperm(400, generator=torch.Generator().manual_seed(86))
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o1, l1 = attn.fwd(qd, kd, vd)
    o2, l2 = attn.fwd(qd[:, :, perm.cuda()].contiguous(), kd, vd)
    torch.cuda.synchronize()
    assert torch.equal(o2, o1[:, :, perm.cuda()])
    assert torch.equal(l2, l1[:, :, perm.cuda()])


def test_causal_packed_qkv_slices():
    # Causal mask on q, k, v read in place from one packed [B, S, 3, H, D] buffer.
    B, H, S, D = 1, 3, 390, 128
    g = torch.Generator().manual_seed(87)
    qkv = torch.randn(B, S, 3, H, D, generator=g).to(torch.bfloat16)
    q, k, v = (qkv[:, :, j].transpose(1, 2) for j in range(3))
    qkv_d = qkv.cuda()
    qd, kd, vd = (qkv_d[:, :, j].transpose(1, 2) for j in range(3))
    o, lse = attn.fwd(qd, kd, vd, causal=True)
    torch.cuda.synchronize()
    o_ref, lse_ref = ref.attention(to_f64(q), to_f64(k), to_f64(v), 1.0 / np.sqrt(128), causal=True)
    compare(to_f64(o.float().cpu()), lse.double().cpu().numpy(), o_ref, lse_ref)


def test_causal_threshold8_many_heads():
    # 3 x 40 heads, ragged S, causal with the pages' rebase threshold 8 (several waves of CTAs).
    q, k, v = wl.make_custom(3, 40, 333, seed=88, qk_gain=2.0)
    full_parity(q, k, v, 1.0 / np.sqrt(128), 8, causal=True)
    assert attn.device_status(reset=False) == 0
