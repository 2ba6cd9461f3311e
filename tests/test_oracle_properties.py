"""Property pins of the oracle (CPU): for random small shapes, scales and input magnitudes, the
row-blocked definition equals the pure-Python brute force, and the pages' online-softmax
recurrence (any tile size, any rebase threshold) equals the definition.

The cases are drawn two ways. A fixed-seed generator always runs (120 cases per property), so
the pins hold on a machine without Hypothesis; where Hypothesis is installed it draws (and
shrinks) further cases through the same checks."""
import numpy as np
import pytest

from oracle import attn_ref as ref

THRESHOLDS = (0.0, 1.5, 8.0, 30.0)
GAINS = (0.1, 1.0, 4.0, 20.0)


def _inputs(c):
    rng = np.random.default_rng(c["seed"])
    q = rng.standard_normal((c["heads"], c["S"], c["D"])) * c["gain"]
    k = rng.standard_normal((c["heads"], c["S"], c["D"])) * c["gain"]
    v = rng.standard_normal((c["heads"], c["S"], c["Dv"]))
    return q, k, v


def check_definition_equals_bruteforce(c, row_block):
    q, k, v = _inputs(c)
    o, lse = ref.attention(q, k, v, c["scale"], row_block=row_block, causal=c["causal"])
    ob, lb = ref.attention_bruteforce(q, k, v, c["scale"], causal=c["causal"])
    assert np.allclose(o, ob, rtol=1e-10, atol=1e-12), c
    assert np.allclose(lse, lb, rtol=1e-12, atol=1e-10), c


def check_online_recurrence_equals_definition(c, tile, threshold):
    q, k, v = _inputs(c)
    o, lse = ref.attention(q, k, v, c["scale"], causal=c["causal"])
    oo, lo = ref.online_softmax_attention(q, k, v, c["scale"], tile=tile, rebase_threshold=threshold,
                                          causal=c["causal"])
    assert np.allclose(oo, o, rtol=1e-9, atol=1e-10), (c, tile, threshold)
    assert np.allclose(lo, lse, rtol=1e-12, atol=1e-9), (c, tile, threshold)


def seeded_cases(n, seed):
    """n cases over the same ranges as the Hypothesis strategy, from a fixed seed."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        c = {"S": int(rng.integers(1, 13)), "D": int(rng.integers(1, 7)), "Dv": int(rng.integers(1, 6)),
             "heads": int(rng.integers(1, 4)), "scale": float(rng.uniform(0.01, 3.0)),
             "gain": float(GAINS[rng.integers(len(GAINS))]), "causal": bool(rng.integers(2)),
             "seed": int(rng.integers(0, 2 ** 31 - 1))}
        out.append((c, int(rng.integers(1, 6)), float(THRESHOLDS[rng.integers(len(THRESHOLDS))])))
    return out


@pytest.mark.parametrize("c,block,_thr", seeded_cases(120, 2024))
def test_definition_equals_bruteforce_seeded(c, block, _thr):
    check_definition_equals_bruteforce(c, block)


@pytest.mark.parametrize("c,tile,thr", seeded_cases(120, 4096))
def test_online_recurrence_equals_definition_seeded(c, tile, thr):
    check_online_recurrence_equals_definition(c, tile, thr)


def test_seeded_cases_cover_the_ranges():
    # The fixed cases reach both masks, every threshold and gain, S = 1 and S = 12.
    cases = seeded_cases(120, 2024) + seeded_cases(120, 4096)
    assert {c["causal"] for c, _, _ in cases} == {False, True}
    assert {t for _, _, t in cases} == set(THRESHOLDS)
    assert {c["gain"] for c, _, _ in cases} == set(GAINS)
    assert {1, 12} <= {c["S"] for c, _, _ in cases}


try:
    from hypothesis import given, settings
    from hypothesis import strategies as st
except ImportError:  # the seeded cases above still run
    given = None

if given is not None:
    CASES = st.fixed_dictionaries({
        "S": st.integers(1, 12),
        "D": st.integers(1, 6),
        "Dv": st.integers(1, 5),
        "heads": st.integers(1, 3),
        "scale": st.floats(0.01, 3.0),
        "gain": st.sampled_from(list(GAINS)),
        "causal": st.booleans(),
        "seed": st.integers(0, 2 ** 31 - 1),
    })

    @settings(max_examples=80, deadline=None)
    @given(CASES, st.integers(1, 5))
    def test_definition_equals_bruteforce_hypothesis(c, row_block):
        check_definition_equals_bruteforce(c, row_block)

    @settings(max_examples=80, deadline=None)
    @given(CASES, st.integers(1, 5), st.sampled_from(list(THRESHOLDS)))
    def test_online_recurrence_equals_definition_hypothesis(c, tile, threshold):
        check_online_recurrence_equals_definition(c, tile, threshold)
