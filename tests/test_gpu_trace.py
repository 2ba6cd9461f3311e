"""The trace build (libattn_trace.so, -DATTN_TRACE) and its per-CTA timeline tool: every CTA
stamps its phases in order, and the traced kernels still compute the same output."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("causal", [False, True])
def test_trace_timeline(causal):
    from dense_attention_forward_gb300 import trace
    # 2 x 8 heads x 16 items = 256 items: more than the SMs, so CTAs walk several items.
    d = trace.timeline(2, 8, 4096, causal=causal)
    assert d["items"] == 2 * 8 * 16 and d["ctas_traced"] == d["ctas"] <= d["items"]
    assert d["items_per_cta"] > 1.0
    assert d["all_exited"] and d["sms"] == d["ctas"]  # one CTA per SM
    for key in ("setup_us", "to_first_s_us", "first_item_kv_loop_us", "later_items_us",
                "final_barrier_to_exit_us", "per_item_us"):
        assert d[key] >= 0.0, (key, d)
    assert d["to_first_s_us"] > 0.0 and d["first_item_kv_loop_us"] > 0.0 and d["later_items_us"] > 0.0
    assert d["cta_us"] <= d["span_us"] + 1e-3
    assert d["cta_us"] >= d["setup_us"] + d["to_first_s_us"] + d["first_item_kv_loop_us"] - 1e-3
    # The boundary between a CTA's first two items, in the order the protocol imposes.
    b = d["boundary"]
    assert b is not None and b["ctas"] >= 1
    # (stamps of one thread are ordered; the issuing warp's may pass the softmax warp's own
    # stamp of a barrier arrival, so only S seen orders the next PV)
    assert 0 < b["last_p_stored_us"] <= b["o_full_us"] <= b["o_read_us"] <= b["epilogue_done_us"]
    assert b["epilogue_done_us"] <= b["next_s_seen_us"] <= b["next_p_stored_us"]
    assert b["next_qk_issued_us"] <= b["next_s_seen_us"] <= b["next_pv_issued_us"]


def test_trace_build_matches_product():
    import ctypes
    import math

    import torch

    import dense_attention_forward_gb300 as attn
    import workloads as wl
    from dense_attention_forward_gb300 import trace

    lib = trace.trace_lib()
    q, k, v = (t.cuda() for t in wl.make_custom(1, 3, 500, seed=99))
    o1, l1 = attn.fwd(q, k, v)
    o2 = torch.empty_like(q)
    l2 = torch.empty_like(l1)
    st = lib.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o2.data_ptr(), l2.data_ptr(), 1, 3, 500, 128,
                      1.0 / math.sqrt(128), torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    buf = (ctypes.c_ulonglong * trace.WORDS)()
    assert lib.attn_trace_read(buf, 1) == 0
    t = np.frombuffer(buf, dtype=np.uint64).astype(np.int64)
    assert t[0] <= t[1] <= t[2] <= max(t[3], t[4]) <= t[5] <= t[7]
