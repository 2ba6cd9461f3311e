"""GPU parity of the causal variant (query i sees keys j <= i) against the fp64 oracle, through
the C ABI (attn_fwd_strided with causal = 1 via the Python binding)."""
import numpy as np
import pytest
import torch

import dense_attention_forward_gb300 as attn
import workloads as wl
from oracle import attn_ref as ref
from workloads import to_f64

from tests.gpu_util import compare, full_parity, run_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("thr", [0, 1, 8])
@pytest.mark.parametrize("S", [1, 2, 17, 127, 128, 129, 255, 256, 257, 383, 511, 512, 640, 1000])
def test_causal_edge_lengths_full(S, thr):
    # Lengths around the 128-row tile and the 256-row CTA: diagonal tiles, the masked tile
    # after the first Q tile's diagonal, an odd tile count (second Q tile past S), ragged tails.
    q, k, v = wl.make_custom(2, 2, S, seed=100 + S)
    full_parity(q, k, v, 1.0 / np.sqrt(128), thr, causal=True)


@pytest.mark.parametrize("thr", [0, 1, 8])
def test_causal_peaky_rows_full(thr):
    q, k, v = wl.make_custom(1, 2, 1500, seed=7, qk_gain=3.0)
    full_parity(q, k, v, 1.0 / np.sqrt(128), thr, causal=True)


def test_causal_first_row_is_exactly_v0():
    # Row 0 sees key 0 alone: P = 1, l = 1, so O[0] = V[0] exactly and lse[0] = s_00.
    q, k, v = wl.make_custom(2, 3, 700, seed=5)
    o, lse = run_gpu(q, k, v, 0.0884, causal=True)
    assert np.array_equal(o[:, :, 0], to_f64(v)[:, :, 0])
    s00 = 0.0884 * np.einsum("bhd,bhd->bh", to_f64(q)[:, :, 0], to_f64(k)[:, :, 0])
    assert np.max(np.abs(lse[:, :, 0] - s00)) < 1e-4


@pytest.mark.parametrize("name,thr", [("s4k", 1), ("s8k", 1), ("s16k", 1), ("ragged", 1), ("s4k", 0),
                                      ("s16k", 8)])
def test_causal_full_size_sampled(name, thr):
    w = wl.ALL[name]
    q, k, v = wl.make_qkv(w)
    o_gpu, lse_gpu = run_gpu(q, k, v, w.scale, thr, causal=True)
    rng = np.random.default_rng(w.seed)
    rows = set(range(0, 130)) | set(range(250, 262)) | set(range(w.S - 140, w.S))
    rows |= set(rng.integers(0, w.S, size=64).tolist())
    rows = np.array(sorted(rows))
    o_ref, lse_ref = ref.attention_rows(to_f64(q), to_f64(k), to_f64(v), w.scale, rows, causal=True)
    compare(o_gpu[..., rows, :], lse_gpu[..., rows], o_ref, lse_ref)
    assert np.all(np.isfinite(o_gpu)) and np.all(np.isfinite(lse_gpu))


def test_causal_bshd_layout():
    B, H, S, D = 2, 3, 515, 128
    q, k, v = wl.make_custom(B, H, S, seed=32)
    qd, kd, vd = (t.transpose(1, 2).contiguous().cuda().transpose(1, 2) for t in (q, k, v))
    out = torch.empty(B, S, H, D, device="cuda", dtype=torch.bfloat16).transpose(1, 2)
    o, lse = attn.fwd(qd, kd, vd, out=out, causal=True)
    torch.cuda.synchronize()
    o_ref, lse_ref = ref.attention(to_f64(q), to_f64(k), to_f64(v), 1.0 / np.sqrt(128), causal=True)
    compare(to_f64(o.float().cpu()), lse.double().cpu().numpy(), o_ref, lse_ref)


def test_causal_differs_from_dense_and_last_row_agrees():
    q, k, v = wl.make_custom(1, 2, 384, seed=9)
    oc, lc = run_gpu(q, k, v, 0.0884, causal=True)
    od, ld = run_gpu(q, k, v, 0.0884, causal=False)
    assert np.max(np.abs(oc[:, :, :200] - od[:, :, :200])) > 0.05
    assert np.max(np.abs(oc[:, :, -1] - od[:, :, -1])) < 1e-2
    assert np.max(np.abs(lc[:, :, -1] - ld[:, :, -1])) < 1e-4
    assert attn.device_status(reset=False) == 0
