"""GB300 (sm_103a) fused dense attention forward: O = softmax(scale * Q K^T) V and lse.

Python face of the C ABI in include/attn.h. Only argument checking and marshalling happen
here; every step of the computation runs in the CUDA kernel of libattn.so. PyTorch provides
device memory and the current stream.
"""
from __future__ import annotations

import math

from ._lib import (AttnError, attn_fwd, attn_fwd_ex, attn_fwd_strided, check_device_status,  # noqa: F401
                   device_status, lib)

__all__ = ["fwd", "fwd_host", "fwd_host_noalloc", "attn_fwd", "attn_fwd_ex", "attn_fwd_strided", "device_status", "check_device_status",
           "AttnError", "lib"]


def _check(name, t, shape=None):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
    if t.dim() != 4:
        raise ValueError(f"{name} must be 4-D [B, H, S, D]")
    if t.stride(-1) != 1:
        raise ValueError(f"{name} must have a contiguous head dimension")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def fwd(q, k, v, scale: float | None = None, out=None, lse=None, return_lse: bool = True,
        stream=None, rebase_threshold: int = 1, causal: bool = False):
    """Attention forward on the current CUDA stream (or `stream`).

    q, k, v: bfloat16 CUDA tensors shaped [B, H, S, 128] with a contiguous last dimension;
    any other strides (e.g. a [B, S, H, D] buffer viewed through transpose(1, 2)) are passed
    to the kernel as they are. scale defaults to 1/sqrt(128).
    Returns (o, lse) with o bfloat16 [B, H, S, 128] (contiguous unless `out` is given) and
    lse float32 [B, H, S] (natural log), or (o, None) when return_lse is False.
    rebase_threshold (1, the default of the C entry points, 0 or 8) selects the online-softmax
    rebase rule (see attn_fwd_ex).
    causal=True applies the causal mask (query i sees keys j <= i; see attn_fwd_causal).
    """
    import torch
    _check("q", q)
    B, H, S, D = q.shape
    _check("k", k, q.shape)
    _check("v", v, q.shape)
    if q.device != k.device or q.device != v.device:
        raise ValueError("q, k, v must be on the same device")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, H, S, D), device=q.device, dtype=torch.bfloat16)
    else:
        _check("out", out, q.shape)
    if return_lse:
        if lse is None:
            lse = torch.empty((B, H, S), device=q.device, dtype=torch.float32)
        elif lse.dtype != torch.float32 or not lse.is_contiguous() or tuple(lse.shape) != (B, H, S):
            raise ValueError("lse must be a contiguous float32 [B, H, S] tensor")
    else:
        lse = None
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    lse_ptr = lse.data_ptr() if lse is not None else None
    with torch.cuda.device(q.device):
        if not causal and all(t.is_contiguous() for t in (q, k, v, out)):
            st = attn_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse_ptr,
                             B, H, S, D, float(scale), int(rebase_threshold), stream.cuda_stream)
        else:
            st = attn_fwd_strided(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse_ptr,
                                  B, H, S, D, float(scale), q.stride()[:3], k.stride()[:3],
                                  v.stride()[:3], out.stride()[:3], int(rebase_threshold),
                                  int(bool(causal)), stream.cuda_stream)
    if st != 0:
        raise AttnError(st)
    return out, lse


def _check_device_buffers(dev, B, H, S, D):
    """fwd_host's `dev`: (q_d, k_d, v_d, o_d, lse_d), contiguous bfloat16 [B, H, S, D] x 4 and
    float32 [B, H, S], all CUDA tensors on one device (the C call writes into them by address,
    so a smaller buffer would be overrun)."""
    import torch
    if not isinstance(dev, (tuple, list)) or len(dev) != 5:
        raise ValueError("dev must be a tuple (q_d, k_d, v_d, o_d, lse_d)")
    names = ("q_d", "k_d", "v_d", "o_d", "lse_d")
    for i, (name, t) in enumerate(zip(names, dev)):
        dt, shape = (torch.float32, (B, H, S)) if i == 4 else (torch.bfloat16, (B, H, S, D))
        if not isinstance(t, torch.Tensor) or t.dtype != dt or tuple(t.shape) != shape or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous {dt} tensor of shape {shape}")
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.device != dev[0].device:
            raise ValueError("the device buffers must all be on one device")


def fwd_host(q, k, v, scale: float | None = None, out=None, lse=None, dev=None, causal: bool = False,
             stream=None):
    """attn_fwd_host: host q, k, v in, host o and lse out, through the caller's device buffers.

    q, k, v: contiguous CPU bfloat16 tensors [B, H, S, 128] (pinned for asynchronous copies);
    scale defaults to 1/sqrt(128).
    out, lse: CPU tensors to receive o (bfloat16) and lse (float32); pinned ones are created if
    not given. dev: (q_d, k_d, v_d, o_d, lse_d) contiguous CUDA tensors of the same shapes on one
    device (checked: shape, dtype, contiguity, device), created on the current device if not
    given; `stream`, when given, must be on that device. The call only enqueues work on `stream` (default: the current
    stream): synchronise before reading out / lse. Returns (out, lse, dev).
    """
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CPU bfloat16 tensor")
        if t.dim() != 4 or tuple(t.shape) != tuple(q.shape):
            raise ValueError(f"{name} must be [B, H, S, D] like q")
    B, H, S, D = q.shape
    if out is None:
        out = torch.empty((B, H, S, D), dtype=torch.bfloat16).pin_memory()
    if lse is None:
        lse = torch.empty((B, H, S), dtype=torch.float32).pin_memory()
    for name, t, dt, shape in (("out", out, torch.bfloat16, (B, H, S, D)), ("lse", lse, torch.float32, (B, H, S))):
        if t.is_cuda or t.dtype != dt or not t.is_contiguous() or tuple(t.shape) != shape:
            raise ValueError(f"{name} must be a contiguous CPU {dt} tensor of shape {shape}")
    if dev is None:
        dev = tuple(torch.empty((B, H, S, D), device="cuda", dtype=torch.bfloat16) for _ in range(4)) + (
            torch.empty((B, H, S), device="cuda", dtype=torch.float32),)
    else:
        _check_device_buffers(dev, B, H, S, D)
    if stream is None:
        stream = torch.cuda.current_stream(dev[0].device)
    elif stream.device != dev[0].device:
        raise ValueError(f"stream is on {stream.device}, the device buffers on {dev[0].device}")
    with torch.cuda.device(dev[0].device):
        st = lib().attn_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                 *(t.data_ptr() for t in dev), B, H, S, D,
                                 float(scale if scale is not None else 1.0 / math.sqrt(D)),
                                 int(bool(causal)), stream.cuda_stream)
    if st != 0:
        raise AttnError(st, "attn_fwd_host")
    return out, lse, dev


def fwd_host_noalloc(q, k, v, scale: float | None = None, out=None, lse=None, causal: bool = False,
                     stream=None):
    """attn_fwd_host_noalloc: host q, k, v in, host o and lse out, staged through the library's
    own fixed device array, so nothing is allocated on the device (for callers that may not
    allocate device memory). B * H * S must not exceed NOALLOC_MAX_ROWS (32768).

    q, k, v: contiguous CPU bfloat16 tensors [B, H, S, 128]; out / lse: contiguous CPU tensors
    for o (bfloat16) and lse (float32), plain CPU tensors if not given; lse=False skips lse.
    Calls share the array: order them on one stream. The call only enqueues work on `stream`
    (default: the current stream); synchronise before reading out / lse. Returns (out, lse).
    """
    import torch
    from ._lib import NOALLOC_MAX_ROWS
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CPU bfloat16 tensor")
        if t.dim() != 4 or tuple(t.shape) != tuple(q.shape):
            raise ValueError(f"{name} must be [B, H, S, D] like q")
    B, H, S, D = q.shape
    if B * H * S > NOALLOC_MAX_ROWS:
        raise ValueError(f"B*H*S = {B * H * S} exceeds the {NOALLOC_MAX_ROWS} rows of the library's "
                         "staging array; use fwd_host with device buffers of your own")
    if out is None:
        out = torch.empty((B, H, S, D), dtype=torch.bfloat16)
    if lse is None:
        lse = torch.empty((B, H, S), dtype=torch.float32)
    elif lse is False:
        lse = None
    for name, t, dt, shape in (("out", out, torch.bfloat16, (B, H, S, D)), ("lse", lse, torch.float32, (B, H, S))):
        if t is None:
            continue
        if t.is_cuda or t.dtype != dt or not t.is_contiguous() or tuple(t.shape) != shape:
            raise ValueError(f"{name} must be a contiguous CPU {dt} tensor of shape {shape}")
    if stream is None:
        stream = torch.cuda.current_stream()
    with torch.cuda.device(stream.device):
        st = lib().attn_fwd_host_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                         lse.data_ptr() if lse is not None else None, B, H, S, D,
                                         float(scale if scale is not None else 1.0 / math.sqrt(D)),
                                         int(bool(causal)), stream.cuda_stream)
    if st != 0:
        raise AttnError(st, "attn_fwd_host_noalloc")
    return out, lse
