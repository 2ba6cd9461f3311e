"""Per-CTA timeline of one attention launch, from the trace build of the kernels.

    python -m dense_attention_forward_gb300.trace [--B 4 --H 16 --S 4096] [--causal]

builds libattn_trace.so if needed (the kernels of libattn.so with -DATTN_TRACE, see
include/attn_trace.h), runs three warm-up launches, writes 256 MB to flush L2, runs one traced
launch and prints one JSON line: the mean duration of each phase of a CTA's first item, the
rest of its items, the mean time per item, and the span of the launch. The
numbers come from the GPU's nanosecond timer, so they include the stamps' own small cost;
use them for where the time goes, not as the kernel's speed (bench.py measures that).
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math

import numpy as np

from . import build as _build

_trace_lib = None
WORDS = 16  # trace words per CTA

_ARGS = [ctypes.c_void_p] * 5 + [ctypes.c_int] * 4 + [ctypes.c_float, ctypes.c_void_p]


def trace_lib():
    global _trace_lib
    if _trace_lib is None:
        h = ctypes.CDLL(_build.build_trace())
        for name in ("attn_fwd", "attn_fwd_causal"):
            getattr(h, name).argtypes = _ARGS
            getattr(h, name).restype = ctypes.c_int
        h.attn_trace_read.argtypes = [ctypes.POINTER(ctypes.c_ulonglong), ctypes.c_int]
        h.attn_trace_read.restype = ctypes.c_int
        h.attn_trace_clear.argtypes = []
        h.attn_trace_clear.restype = ctypes.c_int
        _trace_lib = h
    return _trace_lib


def timeline(B: int, H: int, S: int, causal: bool = False, seed: int = 0) -> dict:
    """One traced launch on seeded N(0,1) BF16 inputs; returns the phase summary."""
    import torch

    lib = trace_lib()
    g = torch.Generator(device="cpu").manual_seed(seed)
    q, k, v = (torch.randn(B, H, S, 128, generator=g).to(torch.bfloat16).cuda() for _ in range(3))
    o = torch.empty_like(q)
    lse = torch.empty(B, H, S, device="cuda", dtype=torch.float32)
    fn = lib.attn_fwd_causal if causal else lib.attn_fwd
    stream = torch.cuda.current_stream().cuda_stream
    call = lambda: fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),  # noqa: E731
                      B, H, S, 128, 1.0 / math.sqrt(128), stream)
    for _ in range(3):
        if call() != 0:
            raise RuntimeError("attn launch failed")
    flush = torch.empty(64 << 20, device="cuda", dtype=torch.float32)
    flush.fill_(1.0)
    torch.cuda.synchronize()
    if lib.attn_trace_clear() != 0:
        raise RuntimeError("attn_trace_clear failed")
    if call() != 0:
        raise RuntimeError("attn launch failed")
    torch.cuda.synchronize()
    items = B * H * ((S + 255) // 256)
    sms = torch.cuda.get_device_properties(q.device).multi_processor_count
    ctas = min(items, sms)  # one CTA per SM, each walking its share of the items
    cap = min(ctas, 4096)
    buf = (ctypes.c_ulonglong * (WORDS * cap))()
    if lib.attn_trace_read(buf, cap) != 0:
        raise RuntimeError("attn_trace_read failed")
    t = np.frombuffer(buf, dtype=np.uint64).reshape(cap, WORDS).astype(np.int64)
    return summarize(t, items, ctas, f"B={B} H={H} S={S} D=128" + (" causal" if causal else ""))


BOUNDARY = {  # word -> name, times relative to word 8 (the first item's last S seen)
    9: "last_p_stored", 3: "o_full", 10: "o_read", 11: "epilogue_done",
    14: "next_qk_issued", 12: "next_s_seen", 13: "next_p_stored", 15: "next_pv_issued",
}


def summarize(t: np.ndarray, items: int, ctas: int, workload: str) -> dict:
    """Phase means (microseconds) of a [ctas, 16] array of trace words (layout in
    include/attn_trace.h): the first item of each CTA phase by phase, then the rest of its items
    up to the final barrier, and the mean time per item. items is the launch's work-item count,
    ctas its CTA count; the gap between one CTA's exit and the next CTA's entry on the same SM
    is reported only where an SM ran several CTAs. "boundary" gives the medians, over the CTAs
    with a second item, of the boundary stamps (Q tile 0) after the first item's last S."""
    cap = t.shape[0]
    first_end = np.maximum(t[:, 3], t[:, 4])
    gaps = []
    for sm in np.unique(t[:, 6]):
        sel = t[t[:, 6] == sm]
        sel = sel[np.argsort(sel[:, 0])]
        gaps.extend((sel[1:, 0] - sel[:-1, 7]).tolist())

    def mean_us(a):
        return round(float(np.mean(a)) / 1e3, 3)

    per_cta = items / ctas
    two = t[(t[:, 12] > 0) & (t[:, 8] > 0)]
    boundary = None
    if len(two):
        boundary = {"ctas": int(len(two))}
        for w, name in BOUNDARY.items():
            boundary[name + "_us"] = round(float(np.median(two[:, w] - two[:, 8])) / 1e3, 3)
    return {
        "workload": workload,
        "items": items, "ctas": ctas, "ctas_traced": cap, "items_per_cta": round(per_cta, 3),
        "sms": int(len(np.unique(t[:, 6]))),
        "span_us": round(float(t[:, 7].max() - t[:, 0].min()) / 1e3, 1),
        "cta_us": mean_us(t[:, 7] - t[:, 0]),
        "per_item_us": mean_us((t[:, 5] - t[:, 0]) / per_cta),
        "setup_us": mean_us(t[:, 1] - t[:, 0]),
        "to_first_s_us": mean_us(t[:, 2] - t[:, 1]),
        "first_item_kv_loop_us": mean_us(t[:, 3] - t[:, 2]),
        "o0_to_o1_us": mean_us(t[:, 4] - t[:, 3]),
        "later_items_us": mean_us(t[:, 5] - first_end),
        "final_barrier_to_exit_us": mean_us(t[:, 7] - t[:, 5]),
        "gap_between_ctas_us": round(float(np.mean(gaps)) / 1e3, 3) if gaps else None,
        "all_exited": bool(np.all(t[:, 7] > 0)),
        "boundary": boundary,
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--B", type=int, default=4)
    ap.add_argument("--H", type=int, default=16)
    ap.add_argument("--S", type=int, default=4096)
    ap.add_argument("--causal", action="store_true")
    args = ap.parse_args()
    print(json.dumps(timeline(args.B, args.H, args.S, args.causal)))


if __name__ == "__main__":
    main()
