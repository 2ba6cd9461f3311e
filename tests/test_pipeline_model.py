"""The kernel's synchronisation protocol, checked on the CPU under random timing.

tests/pipeline_model.py models one CTA of attn_fwd_kernel role by role (see its docstring). These
tests run it over item lists like the ones the persistent grid gives a CTA (dense: equal lengths;
causal: mixed lengths in any order, 1 to 6 K/V tiles here) with random wake-up delays, with and
without random multi-microsecond stalls in every role, and with a K/V token withheld (the
test-hook build's failure path). They also keep the failure the producer's earlier parity waits
had, so that a change that brings it back is caught."""
import pytest

import pipeline_model as pm

DENSE = [[1], [2], [4], [1, 1, 1], [2, 2], [2, 2, 2, 2], [3, 3, 3], [5, 5]]
MIXED = [[6, 2, 4], [2, 1, 2, 1], [1, 2, 3, 2, 1], [2, 6], [6, 2, 2, 2], [3, 1, 1, 3]]


@pytest.mark.parametrize("items", DENSE + MIXED, ids=str)
@pytest.mark.parametrize("stalls", [False, True], ids=["prompt", "stalls"])
def test_ordinary_runs_complete_without_hazards(items, stalls):
    for seed in range(60):
        c = pm.run(items, seed, stalls=stalls)
        assert c.status is None, (items, seed, c.status)
        assert c.seen == [sum(items)] * 2


@pytest.mark.parametrize("items,token", [
    ([4], 0), ([4], 5), ([4], 6),          # K tile 0, V tile 2, the last K tile
    ([2, 2], 1), ([3, 3], 1), ([3, 3], 7),  # a later item that never starts; a token of the second item
    ([2, 6], 3), ([6, 2, 4], 13),
], ids=str)
def test_withheld_token_gives_up_and_drains(items, token):
    for seed in range(40):
        c = pm.run(items, seed, withhold=token, stalls=seed % 2 == 1)
        assert c.status is not None, (items, token, seed)  # some bounded wait ran out ...
        assert c.stopped == [True, True] or c.abort      # ... and every role left (run() checked the exit)


def test_parity_waits_rearm_a_busy_q_barrier():
    # The earlier producer waited on the parity of the S-full barriers. With two items of two
    # K/V tiles no ring wait precedes the second item's Q reload, so it waited for phase 1 of a
    # barrier still in phase 0, passed, and re-armed the Q barrier with its first load in flight.
    for seed in range(5):
        with pytest.raises(pm.ModelError, match="QFull0: arrival with the arrival count used up"):
            pm.run([2, 2], seed, producer_form="parity")


def test_parity_waits_can_give_up_spuriously():
    # With longer items the same waits could find the barrier two phases on and block until their
    # limit: a give-up with nothing withheld.
    statuses = [pm.run([4, 4, 4], seed, producer_form="parity", stalls=True).status for seed in range(400)]
    assert any(s is not None for s in statuses)
    assert all(s is None for s in (pm.run([4, 4, 4], seed, stalls=True).status for seed in range(400)))


def test_model_catches_a_planted_named_barrier_double_arrival():
    # A softmax warp arriving a second time before the issuing warp has passed the barrier (the
    # earlier give-up path) is reported, not absorbed.
    c = pm.CTA([2], 0)
    c.nb_arrive(2, "softmax0.0")
    with pytest.raises(pm.ModelError, match="arrives twice"):
        c.nb_arrive(2, "softmax0.0")
