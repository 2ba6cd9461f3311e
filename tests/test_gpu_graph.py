"""attn.fwd inside a CUDA graph: the call enqueues one kernel whose arguments are all passed by
value (tensor maps included), so a captured graph replays it; replays match the eager call
bit for bit, also after the input buffers are refilled in place."""
import pytest
import torch

import dense_attention_forward_gb300 as attn
import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("causal", [False, True])
def test_graph_replay_matches_eager(causal):
    q, k, v = (t.cuda() for t in wl.make_custom(2, 3, 700, seed=91))
    o = torch.empty_like(q)
    lse = torch.empty(2, 3, 700, device="cuda", dtype=torch.float32)
    o_eager, lse_eager = attn.fwd(q, k, v, causal=causal)  # also prepares the device once
    torch.cuda.synchronize()

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            attn.fwd(q, k, v, out=o, lse=lse, causal=causal)
    torch.cuda.current_stream().wait_stream(side)

    o.zero_()
    lse.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, o_eager) and torch.equal(lse, lse_eager)

    # New inputs in the same buffers: the replay computes on them.
    q2, k2, v2 = (t.cuda() for t in wl.make_custom(2, 3, 700, seed=92))
    q.copy_(q2)
    k.copy_(k2)
    v.copy_(v2)
    g.replay()
    o_ref, lse_ref = attn.fwd(q2, k2, v2, causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
    assert attn.device_status(reset=False) == 0
