"""Property-based pins of the oracle (CPU): for random small shapes, scales and input
magnitudes, the row-blocked definition equals the pure-Python brute force, and the pages'
online-softmax recurrence (any tile size, any rebase threshold) equals the definition."""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

from oracle import attn_ref as ref  # noqa: E402

CASES = st.fixed_dictionaries({
    "S": st.integers(1, 12),
    "D": st.integers(1, 6),
    "Dv": st.integers(1, 5),
    "heads": st.integers(1, 3),
    "scale": st.floats(0.01, 3.0),
    "gain": st.sampled_from([0.1, 1.0, 4.0, 20.0]),
    "causal": st.booleans(),
    "seed": st.integers(0, 2 ** 31 - 1),
})


def _inputs(c):
    rng = np.random.default_rng(c["seed"])
    q = rng.standard_normal((c["heads"], c["S"], c["D"])) * c["gain"]
    k = rng.standard_normal((c["heads"], c["S"], c["D"])) * c["gain"]
    v = rng.standard_normal((c["heads"], c["S"], c["Dv"]))
    return q, k, v


@settings(max_examples=80, deadline=None)
@given(CASES, st.integers(1, 5))
def test_definition_equals_bruteforce(c, row_block):
    q, k, v = _inputs(c)
    o, lse = ref.attention(q, k, v, c["scale"], row_block=row_block, causal=c["causal"])
    ob, lb = ref.attention_bruteforce(q, k, v, c["scale"], causal=c["causal"])
    assert np.allclose(o, ob, rtol=1e-10, atol=1e-12)
    assert np.allclose(lse, lb, rtol=1e-12, atol=1e-10)


@settings(max_examples=80, deadline=None)
@given(CASES, st.integers(1, 5), st.sampled_from([0.0, 1.5, 8.0, 30.0]))
def test_online_recurrence_equals_definition(c, tile, threshold):
    q, k, v = _inputs(c)
    o, lse = ref.attention(q, k, v, c["scale"], causal=c["causal"])
    oo, lo = ref.online_softmax_attention(q, k, v, c["scale"], tile=tile, rebase_threshold=threshold,
                                          causal=c["causal"])
    assert np.allclose(oo, o, rtol=1e-9, atol=1e-10)
    assert np.allclose(lo, lse, rtol=1e-12, atol=1e-9)
