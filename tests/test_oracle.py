"""Pins for the CPU oracle: facts fixed by the mathematics and by the pages, none of which
re-types the oracle's own formula. CPU only."""
import math
import os

import numpy as np
import pytest
import torch

from oracle import attn_ref as ref

RNG = np.random.default_rng(1234)


def _rand(*shape, gain=1.0):
    return RNG.standard_normal(shape) * gain


# --- 1. brute force on tiny inputs --------------------------------------------------------

@pytest.mark.parametrize("S", [1, 2, 3, 17, 32])
@pytest.mark.parametrize("D", [1, 5, 8])
def test_matches_bruteforce(S, D):
    q, k, v = _rand(2, S, D, gain=2.0), _rand(2, S, D, gain=2.0), _rand(2, S, D)
    scale = 1.0 / math.sqrt(D)
    o, lse = ref.attention(q, k, v, scale, row_block=7)
    ob, lseb = ref.attention_bruteforce(q, k, v, scale)
    assert np.max(np.abs(o - ob)) < 1e-12
    assert np.max(np.abs(lse - lseb)) < 1e-12


def test_bruteforce_rectangular_value_dim():
    # D_v != D_qk catches a transposed or swapped operand.
    q, k, v = _rand(1, 6, 3), _rand(1, 6, 3), _rand(1, 6, 4)
    o, lse = ref.attention(q, k, v, 0.7)
    ob, lseb = ref.attention_bruteforce(q, k, v, 0.7)
    assert o.shape == (1, 6, 4)
    assert np.max(np.abs(o - ob)) < 1e-12 and np.max(np.abs(lse - lseb)) < 1e-12


# --- 2. closed forms ----------------------------------------------------------------------

def test_single_key():
    q, k, v = _rand(3, 1, 8), _rand(3, 1, 8), _rand(3, 1, 8)
    o, lse = ref.attention(q, k, v, 0.3)
    assert np.allclose(o, v, atol=1e-15)
    assert np.allclose(lse[..., 0], 0.3 * np.sum(q[:, 0] * k[:, 0], axis=-1), atol=1e-14)


def test_zero_query_gives_mean_and_log_s():
    S = 37
    q, k, v = np.zeros((2, S, 8)), _rand(2, S, 8, gain=5.0), _rand(2, S, 8)
    o, lse = ref.attention(q, k, v, 0.5)
    assert np.allclose(o, v.mean(axis=1, keepdims=True), atol=1e-13)
    assert np.allclose(lse, math.log(S), atol=1e-13)


def test_identical_keys():
    S = 29
    u = _rand(8)
    q, k, v = _rand(1, S, 8), np.tile(u, (1, S, 1)), _rand(1, S, 8)
    o, lse = ref.attention(q, k, v, 0.25)
    assert np.allclose(o, v.mean(axis=1, keepdims=True), atol=1e-13)
    assert np.allclose(lse[0], 0.25 * (q[0] @ u) + math.log(S), atol=1e-13)


def test_constant_values():
    q, k = _rand(2, 50, 8, gain=3.0), _rand(2, 50, 8, gain=3.0)
    v = np.full((2, 50, 8), -1.75)
    o, _ = ref.attention(q, k, v, 0.4)
    assert np.allclose(o, -1.75, atol=1e-14)


def test_two_keys_three_to_one():
    # Scores ln 3 and 0 give weights exactly 3/4 and 1/4, and lse = ln 4.
    q = np.array([[[1.0]]])
    k = np.array([[[math.log(3.0)], [0.0]]])
    v = np.array([[[8.0], [-4.0]]])
    q2 = np.concatenate([q, q], axis=1)  # two identical query rows
    o, lse = ref.attention(q2, k, v, 1.0)
    assert np.allclose(o, 0.75 * 8.0 + 0.25 * -4.0, atol=1e-14)
    assert np.allclose(lse, math.log(4.0), atol=1e-14)


# --- 3. invariants ------------------------------------------------------------------------

def test_probability_rows_sum_to_one_and_are_positive():
    p = ref.probabilities(_rand(2, 40, 8, gain=3.0), _rand(2, 40, 8, gain=3.0), 0.35)
    assert np.all(p > 0)
    assert np.allclose(p.sum(axis=-1), 1.0, atol=1e-14)


def test_probabilities_two_keys_with_a_non_unit_scale():
    # Raw scores 2 ln 3 and 0 at scale 1/2 are ln 3 and 0: weights exactly 3/4 and 1/4. A
    # dropped scale gives 9/10 and 1/10, a doubled one 81/82 and 1/82.
    q = np.array([[[1.0], [-1.0]]])
    k = np.array([[[2.0 * math.log(3.0)], [0.0]]])
    p = ref.probabilities(q, k, 0.5)
    assert np.allclose(p[0, 0], [0.75, 0.25], atol=1e-15)
    assert np.allclose(p[0, 1], [0.25, 0.75], atol=1e-15)  # row 1: scores -ln 3 and 0


def test_probabilities_times_values_is_the_attention_output():
    # softmax(scale Q K^T) V is O by the definition; attention() is pinned independently
    # (brute force, closed forms, torch SDPA), so a wrong scale, axis or transpose in
    # probabilities() shows here.
    q, k, v = _rand(3, 23, 6, gain=2.0), _rand(3, 23, 6, gain=2.0), _rand(3, 23, 4)
    p = ref.probabilities(q, k, 0.37)
    o, _ = ref.attention(q, k, v, 0.37)
    assert p.shape == (3, 23, 23)
    assert np.max(np.abs(p @ v - o)) < 1e-13


def test_probabilities_match_bruteforce_on_large_scores():
    # Entries written out with math.exp around each row's own maximum; scores of order 10^3
    # overflow unless the maximum is taken along the key axis of each row.
    q, k = _rand(1, 7, 3, gain=25.0), _rand(1, 7, 3, gain=25.0)
    scale = 0.8
    p = ref.probabilities(q, k, scale)
    for i in range(7):
        s = [scale * sum(q[0, i, d] * k[0, j, d] for d in range(3)) for j in range(7)]
        mx = max(s)
        e = [math.exp(x - mx) for x in s]
        tot = sum(e)
        for j in range(7):
            assert abs(p[0, i, j] - e[j] / tot) < 1e-13


def test_output_is_convex_combination_of_values():
    q, k, v = _rand(1, 64, 8, gain=2.0), _rand(1, 64, 8, gain=2.0), _rand(1, 64, 8)
    o, _ = ref.attention(q, k, v, 0.5)
    assert np.all(o <= v.max(axis=1, keepdims=True) + 1e-14)
    assert np.all(o >= v.min(axis=1, keepdims=True) - 1e-14)


def test_key_shift_invariance():
    # K <- K + 1 u^T adds scale * q_i . u to every score of row i: O unchanged, lse shifted.
    q, k, v = _rand(1, 45, 8), _rand(1, 45, 8), _rand(1, 45, 8)
    u = _rand(8, gain=4.0)
    scale = 0.3
    o1, l1 = ref.attention(q, k, v, scale)
    o2, l2 = ref.attention(q, k + u, v, scale)
    assert np.max(np.abs(o1 - o2)) < 1e-12
    assert np.max(np.abs((l2 - l1) - scale * (q[0] @ u))) < 1e-12


def test_joint_key_value_permutation():
    q, k, v = _rand(1, 33, 8), _rand(1, 33, 8), _rand(1, 33, 8)
    perm = RNG.permutation(33)
    o1, l1 = ref.attention(q, k, v, 0.4)
    o2, l2 = ref.attention(q, k[:, perm], v[:, perm], 0.4)
    assert np.max(np.abs(o1 - o2)) < 1e-13 and np.max(np.abs(l1 - l2)) < 1e-13


def test_query_permutation_permutes_rows():
    q, k, v = _rand(1, 21, 8), _rand(1, 21, 8), _rand(1, 21, 8)
    perm = RNG.permutation(21)
    o1, l1 = ref.attention(q, k, v, 0.4)
    o2, l2 = ref.attention(q[:, perm], k, v, 0.4)
    assert np.max(np.abs(o1[:, perm] - o2)) < 1e-13 and np.max(np.abs(l1[:, perm] - l2)) < 1e-13


def test_value_linearity():
    q, k, v, w = _rand(1, 30, 8), _rand(1, 30, 8), _rand(1, 30, 8), _rand(1, 30, 8)
    o_v, _ = ref.attention(q, k, v, 0.4)
    o_w, _ = ref.attention(q, k, w, 0.4)
    o_mix, _ = ref.attention(q, k, 2.5 * v - 0.5 * w, 0.4)
    assert np.max(np.abs(o_mix - (2.5 * o_v - 0.5 * o_w))) < 1e-12


def test_rows_subset_is_exact():
    q, k, v = _rand(2, 3, 70, 8), _rand(2, 3, 70, 8), _rand(2, 3, 70, 8)
    rows = np.array([0, 5, 69, 33])
    o, lse = ref.attention(q, k, v, 0.4)
    o_r, lse_r = ref.attention_rows(q, k, v, 0.4, rows, row_block=3)
    # BLAS may block a 3-row product differently from a 70-row one: equal to rounding.
    assert np.max(np.abs(o[..., rows, :] - o_r)) < 1e-14
    assert np.max(np.abs(lse[..., rows] - lse_r)) < 1e-14


def test_large_scores_do_not_overflow():
    # Scores of order 1e3: exp without the max trick would overflow.
    q, k, v = _rand(1, 20, 8, gain=30.0), _rand(1, 20, 8, gain=30.0), _rand(1, 20, 8)
    o, lse = ref.attention(q, k, v, 1.0)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    s = q[0] @ k[0].T
    assert np.all(lse[0] >= s.max(axis=1) - 1e-9)
    assert np.all(lse[0] <= s.max(axis=1) + math.log(20) + 1e-9)


# --- 4. library special case: PyTorch SDPA in fp64 on the CPU -----------------------------

def test_matches_torch_sdpa_fp64():
    q, k, v = (torch.from_numpy(_rand(2, 3, 150, 16, gain=g)) for g in (2.0, 2.0, 1.0))
    scale = 0.21
    o_t = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=scale)
    lse_t = torch.logsumexp(scale * (q @ k.transpose(-1, -2)), dim=-1)
    o, lse = ref.attention(q.numpy(), k.numpy(), v.numpy(), scale)
    assert np.max(np.abs(o - o_t.numpy())) < 1e-10
    assert np.max(np.abs(lse - lse_t.numpy())) < 1e-10


# --- 5. the pages' online recurrence equals the definition, whatever the threshold -------

@pytest.mark.parametrize("threshold", [0.0, 8.0, 16.0])
@pytest.mark.parametrize("S,tile", [(300, 128), (97, 16), (128, 128), (1, 128)])
def test_online_recurrence_threshold_invariance(threshold, S, tile):
    q, k, v = _rand(2, S, 16, gain=3.0), _rand(2, S, 16, gain=3.0), _rand(2, S, 16)
    scale = 1.0 / 4.0
    o, lse = ref.attention(q, k, v, scale)
    o2, lse2 = ref.online_softmax_attention(q, k, v, scale, tile=tile, rebase_threshold=threshold)
    assert np.max(np.abs(o - o2)) < 1e-11
    assert np.max(np.abs(lse - lse2)) < 1e-11


def test_online_recurrence_increasing_scores_force_rebases():
    # Scores that grow tile after tile: every tile rebases at threshold 0 and none at 1e9
    # (the kept max is then the first tile's), and both equal the definition.
    S, D = 64, 1
    q = np.ones((1, S, D))
    k = np.linspace(0.0, 60.0, S).reshape(1, S, D)
    v = _rand(1, S, D)
    o, lse = ref.attention(q, k, v, 1.0)
    for thr in (0.0, 8.0, 1e9):
        o2, lse2 = ref.online_softmax_attention(q, k, v, 1.0, tile=8, rebase_threshold=thr)
        assert np.max(np.abs(o - o2)) < 1e-11 and np.max(np.abs(lse - lse2)) < 1e-11


# --- 6. the pages' printed numbers --------------------------------------------------------

def _golden(name):
    path = os.path.join(os.path.dirname(__file__), "golden", name)
    out = {}
    with open(path) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                key, val, dec = line.split()
                out[key] = (float(val), int(dec))
    return out


def test_rebase_threshold_numbers_from_the_pages():
    g = _golden("rebase_threshold.txt")
    max_p, natural, raw = ref.rebase_threshold_in_other_units(8.0, 128)
    gap_778 = ref.rebase_threshold_in_other_units(7.78, 128)[0]
    # The page prints these with "~="; some are truncated (219.79 -> 219), so allow one unit
    # of the last printed decimal.
    for key, got in (("threshold_8_max_p", max_p), ("threshold_8_natural", natural),
                     ("threshold_8_raw_d128", raw), ("gap_7.78_max_p", gap_778)):
        val, dec = g[key]
        assert abs(got - val) <= 10.0 ** -dec, key
    assert max_p == 256.0


# --- 7. the output format: no BF16 O can meet a 1.5e-2 bound everywhere once |O| >= 4 ---

def test_bf16_output_cannot_always_be_within_1p5e2():
    # Exact O = 4.015625 (two equally weighted keys with V = 4 and 4.03125, both BF16
    # numbers); its BF16 neighbours are 4.0 and 4.03125, each 0.015625 away.
    q = np.zeros((1, 2, 1))
    k = np.array([[[0.3], [-1.2]]])
    v = np.array([[[4.0], [4.03125]]])
    o, lse = ref.attention(q, k, v, 1.0)
    assert o[0, 0, 0] == 4.015625 and abs(lse[0, 0] - math.log(2.0)) < 1e-15
    # 4.0 and 4.03125 are adjacent BF16 numbers (7 stored mantissa bits: spacing 2^-5 in [4, 8)).
    assert torch.tensor([4.0, 4.03125]).to(torch.bfloat16).view(torch.int16).tolist() == [0x4080, 0x4081]
    assert torch.tensor([4.015625]).to(torch.bfloat16).item() in (4.0, 4.03125)
    assert min(abs(4.015625 - 4.0), abs(4.015625 - 4.03125)) == 0.015625 > 1.5e-2


# --- 8. the causal variant (not on the pages: the usual decoder mask, key j visible to
#        query i iff j <= i) ----------------------------------------------------------------

@pytest.mark.parametrize("S", [1, 2, 3, 17, 32])
def test_causal_matches_bruteforce(S):
    q, k, v = _rand(2, S, 5, gain=2.0), _rand(2, S, 5, gain=2.0), _rand(2, S, 5)
    o, lse = ref.attention(q, k, v, 0.6, row_block=7, causal=True)
    ob, lseb = ref.attention_bruteforce(q, k, v, 0.6, causal=True)
    assert np.max(np.abs(o - ob)) < 1e-12 and np.max(np.abs(lse - lseb)) < 1e-12


def test_causal_first_row_is_first_value():
    # Row 0 sees key 0 only: O = V[0], lse = s_00.
    q, k, v = _rand(3, 40, 8), _rand(3, 40, 8), _rand(3, 40, 8)
    o, lse = ref.attention(q, k, v, 0.35, causal=True)
    assert np.max(np.abs(o[:, 0] - v[:, 0])) < 1e-14
    assert np.max(np.abs(lse[:, 0] - 0.35 * np.einsum("nd,nd->n", q[:, 0], k[:, 0]))) < 1e-14


def test_causal_row_is_plain_attention_over_its_prefix():
    # Row i equals the non-causal definition on q_i and the first i + 1 keys and values,
    # and the last row sees every key.
    q, k, v = _rand(2, 70, 6, gain=2.0), _rand(2, 70, 6, gain=2.0), _rand(2, 70, 6)
    o, lse = ref.attention(q, k, v, 0.4, row_block=16, causal=True)
    for i in (1, 5, 31, 32, 69):
        op, lp = ref.attention(q[:, : i + 1], k[:, : i + 1], v[:, : i + 1], 0.4)
        assert np.max(np.abs(o[:, i] - op[:, i])) < 1e-13 and np.max(np.abs(lse[:, i] - lp[:, i])) < 1e-13
    of, lf = ref.attention(q, k, v, 0.4)
    assert np.max(np.abs(o[:, -1] - of[:, -1])) < 1e-13 and np.max(np.abs(lse[:, -1] - lf[:, -1])) < 1e-13


def test_causal_ignores_the_future():
    # Changing keys and values after position t leaves rows 0..t unchanged.
    q, k, v = _rand(1, 50, 4), _rand(1, 50, 4), _rand(1, 50, 4)
    o, lse = ref.attention(q, k, v, 0.5, causal=True)
    k2, v2 = k.copy(), v.copy()
    k2[:, 21:] = _rand(1, 29, 4, gain=5.0)
    v2[:, 21:] = _rand(1, 29, 4, gain=5.0)
    o2, lse2 = ref.attention(q, k2, v2, 0.5, causal=True)
    assert np.array_equal(o[:, :21], o2[:, :21]) and np.array_equal(lse[:, :21], lse2[:, :21])
    assert np.max(np.abs(o[:, 21:] - o2[:, 21:])) > 1e-3


def test_causal_rows_subset_is_exact():
    q, k, v = _rand(2, 300, 8), _rand(2, 300, 8), _rand(2, 300, 8)
    rows = np.array([0, 1, 127, 128, 255, 299])
    o, lse = ref.attention(q, k, v, 0.3, causal=True)
    os_, ls_ = ref.attention_rows(q, k, v, 0.3, rows, row_block=4, causal=True)
    assert np.max(np.abs(o[:, rows] - os_)) < 1e-14 and np.max(np.abs(lse[:, rows] - ls_)) < 1e-14


def test_causal_matches_torch_sdpa_fp64():
    q, k, v = (torch.from_numpy(_rand(2, 3, 45, 16, gain=1.5)) for _ in range(3))
    o, lse = ref.attention(q.numpy(), k.numpy(), v.numpy(), 0.2, causal=True)
    o_t = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, scale=0.2)
    mask = torch.ones(45, 45, dtype=torch.bool).tril()
    s = torch.where(mask, 0.2 * q @ k.transpose(-1, -2), torch.tensor(-math.inf, dtype=torch.float64))
    assert np.max(np.abs(o - o_t.numpy())) < 1e-10
    assert np.max(np.abs(lse - torch.logsumexp(s, dim=-1).numpy())) < 1e-10


@pytest.mark.parametrize("threshold", [0.0, 8.0])
@pytest.mark.parametrize("S,tile", [(300, 128), (97, 16), (256, 128)])
def test_causal_online_recurrence(threshold, S, tile):
    # Tiles wholly in a row's future leave its state alone; the recurrence still equals the
    # definition.
    q, k, v = _rand(2, S, 8, gain=2.5), _rand(2, S, 8, gain=2.5), _rand(2, S, 8)
    o, lse = ref.attention(q, k, v, 0.3, causal=True)
    oo, lo = ref.online_softmax_attention(q, k, v, 0.3, tile=tile, rebase_threshold=threshold, causal=True)
    assert np.max(np.abs(o - oo)) < 1e-12 and np.max(np.abs(lse - lo)) < 1e-12
