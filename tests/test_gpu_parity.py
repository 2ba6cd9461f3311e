"""Parity of the CUDA path (through the C ABI) with the fp64 CPU oracle on seeded inputs."""
import numpy as np
import pytest
import torch

import dense_attention_forward_gb300 as attn
import workloads as wl
from oracle import attn_ref as ref
from tests.gpu_util import compare, full_parity, run_gpu, sample_rows
from workloads import to_f64

pytestmark = pytest.mark.gpu


def test_tiny_workload_full():
    w = wl.TINY
    q, k, v = wl.make_qkv(w)
    full_parity(q, k, v, w.scale)


@pytest.mark.parametrize("thr", [0, 1, 8])
@pytest.mark.parametrize("S", [1, 2, 17, 127, 128, 129, 255, 256, 257, 383, 640, 1000])
def test_edge_lengths_full(S, thr):
    q, k, v = wl.make_custom(2, 3, S, seed=S)
    full_parity(q, k, v, 1.0 / np.sqrt(128), thr)


@pytest.mark.parametrize("thr", [0, 1, 8])
@pytest.mark.parametrize("S", [300, 1024, 1500])
def test_peaky_rows_full(S, thr):
    # Q and K x3 before the BF16 cast: score std ~9, rows rebase often.
    q, k, v = wl.make_custom(1, 4, S, seed=7 + S, qk_gain=3.0)
    full_parity(q, k, v, 1.0 / np.sqrt(128), thr)


def test_rising_scores_rebase_every_tile():
    # Key norms grow along the sequence, so every K/V tile raises the row max (by more than
    # 8 base-2 units between the first and the last tiles): the rescale path runs at both
    # thresholds and the two results agree with the oracle.
    S = 1024
    g = torch.Generator().manual_seed(21)
    q = torch.randn(1, 2, S, 128, generator=g)
    k = torch.randn(1, 2, S, 128, generator=g) * torch.linspace(0.2, 3.0, S).view(1, 1, S, 1)
    v = torch.randn(1, 2, S, 128, generator=g)
    q, k, v = (t.to(torch.bfloat16) for t in (q, k, v))
    for thr in (0, 1, 8):
        full_parity(q, k, v, 1.0 / np.sqrt(128), thr)


def test_bf16_midpoint_output():
    # Two equally weighted keys (q = 0) with V = 4 and 4.03125: the exact O, 4.015625, lies
    # half-way between two BF16 numbers; the result must be one of them.
    S, D = 2, 128
    q = torch.zeros(1, 1, S, D, dtype=torch.bfloat16)
    k = torch.randn(1, 1, S, D).to(torch.bfloat16)
    v = torch.empty(1, 1, S, D, dtype=torch.bfloat16)
    v[0, 0, 0] = 4.0
    v[0, 0, 1] = 4.03125
    o, lse = attn.fwd(q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    vals = set(o.float().flatten().tolist())
    assert vals <= {4.0, 4.03125}, vals
    assert torch.allclose(lse.float().cpu(), torch.full((1, 1, S), float(np.log(2.0))), atol=1e-6)


def test_other_scale():
    q, k, v = wl.make_custom(1, 2, 700, seed=3)
    full_parity(q, k, v, 0.05)


@pytest.mark.parametrize("name", ["s4k", "s8k", "s16k"])
def test_full_size_workloads_every_row(name):
    # The three sequence lengths of the pages at their full sizes, in the launch configuration
    # the bench times (the default threshold 1): every row of every head against the oracle
    # (rows are independent, so the oracle runs them in blocks; 0.55 / 1.1 / 2.2 TFLOP of fp64).
    w = wl.ALL[name]
    q, k, v = wl.make_qkv(w)
    o_gpu, lse_gpu = run_gpu(q, k, v, w.scale)
    o_ref, lse_ref = ref.attention(to_f64(q), to_f64(k), to_f64(v), w.scale, row_block=1024)
    stats = compare(o_gpu, lse_gpu, o_ref, lse_ref)
    assert stats["n_rows"] == w.B * w.H * w.S


@pytest.mark.parametrize("name,thr", [("ragged", 1), ("ragged", 0), ("s4k", 0), ("s4k", 8), ("s16k", 8),
                                      ("ragged", 8)])
def test_full_size_workloads_sampled(name, thr):
    w = wl.ALL[name]
    q, k, v = wl.make_qkv(w)
    o_gpu, lse_gpu = run_gpu(q, k, v, w.scale, thr)
    rows = sample_rows(w.S, seed=w.seed)
    o_ref, lse_ref = ref.attention_rows(to_f64(q), to_f64(k), to_f64(v), w.scale, rows)
    compare(o_gpu[..., rows, :], lse_gpu[..., rows], o_ref, lse_ref)
    # Properties at every row: O is a convex combination of V rows, lse finite.
    vf = v.float()
    vmax = vf.amax(dim=2, keepdim=True).double().numpy()
    vmin = vf.amin(dim=2, keepdim=True).double().numpy()
    assert np.all(o_gpu <= vmax + 1e-2) and np.all(o_gpu >= vmin - 1e-2)
    assert np.all(np.isfinite(lse_gpu))


@pytest.mark.parametrize("thr", [0, 1, 8])
def test_bshd_layout(thr):
    # [B, S, H, D] buffers viewed as [B, H, S, D] through transpose(1, 2): the kernel reads
    # and writes them in place through 4-D tensor maps.
    B, H, S, D = 2, 3, 515, 128
    q, k, v = wl.make_custom(B, H, S, seed=31)
    qd, kd, vd = (t.transpose(1, 2).contiguous().cuda().transpose(1, 2) for t in (q, k, v))
    assert not qd.is_contiguous()
    out = torch.empty(B, S, H, D, device="cuda", dtype=torch.bfloat16).transpose(1, 2)
    o, lse = attn.fwd(qd, kd, vd, out=out, rebase_threshold=thr)
    torch.cuda.synchronize()
    o_ref, lse_ref = ref.attention(to_f64(q), to_f64(k), to_f64(v), 1.0 / np.sqrt(128))
    compare(to_f64(o.float().cpu()), lse.double().cpu().numpy(), o_ref, lse_ref)


def test_packed_qkv_slices():
    # q, k, v as slices of one packed [B, S, 3, H, D] buffer (strides: S*3*H*D, D, 3*H*D).
    B, H, S, D = 1, 4, 300, 128
    g = torch.Generator().manual_seed(41)
    qkv = torch.randn(B, S, 3, H, D, generator=g).to(torch.bfloat16)
    q, k, v = (qkv[:, :, j].transpose(1, 2) for j in range(3))
    qkv_d = qkv.cuda()
    qd, kd, vd = (qkv_d[:, :, j].transpose(1, 2) for j in range(3))
    o, lse = attn.fwd(qd, kd, vd)
    torch.cuda.synchronize()
    o_ref, lse_ref = ref.attention(to_f64(q), to_f64(k), to_f64(v), 1.0 / np.sqrt(128))
    compare(to_f64(o.float().cpu()), lse.double().cpu().numpy(), o_ref, lse_ref)


def test_guard_regions_untouched():
    B, H, S, D = 1, 2, 200, 128
    q, k, v = (t.cuda() for t in wl.make_custom(B, H, S, seed=11))
    n = B * H * S * D
    guard = 4096
    obuf = torch.full((n + 2 * guard,), 7.0, device="cuda", dtype=torch.bfloat16)
    lbuf = torch.full((B * H * S + 2 * 64,), 7.0, device="cuda", dtype=torch.float32)
    o = obuf[guard:guard + n].view(B, H, S, D)
    lse = lbuf[64:64 + B * H * S].view(B, H, S)
    attn.fwd(q, k, v, out=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.all(obuf[:guard] == 7.0) and torch.all(obuf[guard + n:] == 7.0)
    assert torch.all(lbuf[:64] == 7.0) and torch.all(lbuf[64 + B * H * S:] == 7.0)
    o_ref, lse_ref = ref.attention(*(to_f64(t.cpu()) for t in (q, k, v)), 1.0 / np.sqrt(128))
    compare(to_f64(o.float().cpu()), lse.double().cpu().numpy(), o_ref, lse_ref)


def test_side_stream_and_determinism():
    q, k, v = (t.cuda() for t in wl.make_custom(2, 2, 777, seed=5))
    o1, l1 = attn.fwd(q, k, v)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        o2, l2 = attn.fwd(q, k, v)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_without_lse():
    q, k, v = (t.cuda() for t in wl.make_custom(1, 2, 333, seed=9))
    o1, l1 = attn.fwd(q, k, v)
    o2, l2 = attn.fwd(q, k, v, return_lse=False)
    torch.cuda.synchronize()
    assert l2 is None and torch.equal(o1, o2)


def test_gpu_argument_errors():
    x = torch.zeros(1, 1, 64, 64, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(attn.AttnError) as e:
        attn.fwd(x, x, x)
    assert e.value.status == 2
    buf = torch.zeros(1 + 1 * 1 * 64 * 128, device="cuda", dtype=torch.bfloat16)
    y = buf[1:].view(1, 1, 64, 128)  # 2-byte offset: not 16-byte aligned
    z = torch.zeros(1, 1, 64, 128, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(attn.AttnError) as e:
        attn.fwd(y, z, z)
    assert e.value.status == 3


def test_no_wait_gave_up():
    torch.cuda.synchronize()
    assert attn.device_status(reset=False) == 0


def test_many_heads_full():
    # 256 (b, h) pairs x 2 CTAs: more CTAs than SMs, several waves, ragged S.
    q, k, v = wl.make_custom(4, 64, 300, seed=51)
    full_parity(q, k, v, 1.0 / np.sqrt(128))


@pytest.mark.parametrize("causal", [False, True])
def test_long_sequence_sampled(causal):
    # S = 65536 + 77: 514 K/V tiles per CTA, rows sampled at the start, middle and tail.
    B, H, S = 1, 2, 65536 + 77
    q, k, v = wl.make_custom(B, H, S, seed=61)
    o_gpu, lse_gpu = run_gpu(q, k, v, 1.0 / np.sqrt(128), 0, causal=causal)
    rng = np.random.default_rng(61)
    rows = np.array(sorted(set(range(0, 40)) | set(range(S - 300, S)) | set(rng.integers(0, S, 40).tolist())))
    o_ref, lse_ref = ref.attention_rows(to_f64(q), to_f64(k), to_f64(v), 1.0 / np.sqrt(128), rows, causal=causal)
    compare(o_gpu[..., rows, :], lse_gpu[..., rows], o_ref, lse_ref)
