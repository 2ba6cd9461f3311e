"""CPU oracle for the dense attention forward pass: plain, slow, fp64.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports, links or runs this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may.
It shares no code, table or helper with the CUDA path.

Sources (the pages are four web pages about one B200 attention kernel):

* "B200 attention kernel from scratch to ~SOTA in 60 figures (CUDA/PTX)", Japanese
  translation at hackernews.jp/story/49535281 -- cited below as [B200-attn].
  - Ch. 1 §ii "work parallelisation": Q, K, V and O share the shape [B, heads, S, D]; each
    (batch, head, q-tile) is independent; the output is O / rowsum after the K/V loop.
  - Ch. 1 §B "online softmax": the per-tile state update (tile rowmax, new rowmax,
    rescale = exp(old - new), rowsum and O rescaled, P = exp(S - new), rowsum += sum P,
    O += P @ V) and the max trick (subtract the row max before exponentiating).
  - Ch. 8 "hardware approximations": exp(x) = exp2(x * log2 e); the softmax scale and
    log2 e are folded into one factor and the row max is found on raw S, then multiplied.
  - Ch. 11 "skip O rescale": keep the old row max unless the new tile's max exceeds it by
    the threshold (8 in base-2 units); skipping loses nothing because the same P enters
    both O and rowsum, and the final O / rowsum cancels the common factor.

What is computed (the plain definition, for every (b, h) and query row i < S, over all
keys j < S, non-causal, no mask):

    s_ij  = scale * sum_d Q[i, d] K[j, d]
    m_i   = max_j s_ij
    l_i   = sum_j exp(s_ij - m_i)
    O[i]  = sum_j exp(s_ij - m_i) V[j] / l_i
    lse_i = m_i + ln l_i          (natural log of sum_j exp(s_ij); the pages do not print
                                   lse, this is the usual FlashAttention convention)

Causal variant (``causal=True``). The pages fix their scope to non-causal attention; the
causal mask is the usual decoder one, with queries and keys on the same positions 0..S-1:
query i sees keys j <= i only, i.e. s_ij = -inf for j > i before the softmax, and every max,
sum and product above runs over j <= i. Row i then equals the non-causal definition applied
to q_i and the first i + 1 keys and values.

All arithmetic is float64. Inputs are whatever float arrays the caller passes (the tests
pass the BF16 tensors the GPU reads, widened exactly).
"""
from __future__ import annotations

import math

import numpy as np

LOG2E = 1.4426950408889634  # log2(e)
LN2 = 0.6931471805599453    # ln(2)


def _as_heads(x: np.ndarray) -> np.ndarray:
    """View [..., S, D] as [N, S, D] (N = product of the leading dims)."""
    x = np.asarray(x, dtype=np.float64)
    if x.ndim < 2:
        raise ValueError("expected [..., S, D]")
    return x.reshape((-1,) + x.shape[-2:])


def _softmax_rows(q_rows: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
                  row_ids=None):
    """Exact softmax attention for a block of query rows of one head ([B200-attn] Ch. 1 §ii,
    with the max trick of Ch. 1 §B). With ``row_ids`` (the rows' positions) the causal mask
    hides keys j > row_id."""
    s = scale * (q_rows @ k.T)                 # scores, [rows, S]
    if row_ids is not None:
        s = np.where(np.arange(k.shape[0])[None, :] > np.asarray(row_ids)[:, None], -np.inf, s)
    m = s.max(axis=1, keepdims=True)           # row max
    e = np.exp(s - m)                          # unnormalised probabilities
    l = e.sum(axis=1, keepdims=True)           # row sum
    o = (e @ v) / l
    lse = m[:, 0] + np.log(l[:, 0])
    return o, lse


def attention(q, k, v, scale: float, row_block: int = 512, causal: bool = False):
    """O and lse for every row of every head. q, k, v: [..., S, D]; returns
    (o [..., S, D], lse [..., S]) in float64."""
    qh, kh, vh = _as_heads(q), _as_heads(k), _as_heads(v)
    n, S, D = qh.shape
    o = np.empty((n, S, vh.shape[-1]))
    lse = np.empty((n, S))
    for h in range(n):
        for r0 in range(0, S, row_block):
            r1 = min(S, r0 + row_block)
            ids = np.arange(r0, r1) if causal else None
            o[h, r0:r1], lse[h, r0:r1] = _softmax_rows(qh[h, r0:r1], kh[h], vh[h], scale, ids)
    lead = np.asarray(q).shape[:-2]
    return o.reshape(lead + (S, vh.shape[-1])), lse.reshape(lead + (S,))


def attention_rows(q, k, v, scale: float, rows, row_block: int = 512, causal: bool = False):
    """O and lse for a subset of query rows (the same rows in every head). Rows are
    independent in the definition, so this is exact for those rows."""
    rows = np.asarray(rows, dtype=np.int64)
    qh, kh, vh = _as_heads(q), _as_heads(k), _as_heads(v)
    n = qh.shape[0]
    o = np.empty((n, rows.size, vh.shape[-1]))
    lse = np.empty((n, rows.size))
    for h in range(n):
        for r0 in range(0, rows.size, row_block):
            sel = rows[r0:r0 + row_block]
            o[h, r0:r0 + sel.size], lse[h, r0:r0 + sel.size] = _softmax_rows(
                qh[h, sel], kh[h], vh[h], scale, sel if causal else None)
    lead = np.asarray(q).shape[:-2]
    return o.reshape(lead + (rows.size, vh.shape[-1])), lse.reshape(lead + (rows.size,))


def probabilities(q, k, scale: float):
    """The normalised attention matrix softmax(scale * Q K^T) per head (small cases)."""
    qh, kh = _as_heads(q), _as_heads(k)
    s = scale * np.einsum("nid,njd->nij", qh, kh)
    e = np.exp(s - s.max(axis=2, keepdims=True))
    p = e / e.sum(axis=2, keepdims=True)
    lead = np.asarray(q).shape[:-2]
    return p.reshape(lead + p.shape[1:])


def attention_bruteforce(q, k, v, scale: float, causal: bool = False):
    """The definition with pure-Python loops and math.exp, for tiny inputs only."""
    qh, kh, vh = _as_heads(q).tolist(), _as_heads(k).tolist(), _as_heads(v).tolist()
    o_all, lse_all = [], []
    for qq, kk, vv in zip(qh, kh, vh):
        S = len(qq)
        o_h, lse_h = [], []
        for i in range(S):
            scores = []
            keys = range(i + 1) if causal else range(S)
            for j in keys:
                acc = 0.0
                for d in range(len(qq[i])):
                    acc += qq[i][d] * kk[j][d]
                scores.append(scale * acc)
            mx = max(scores)
            w = [math.exp(x - mx) for x in scores]
            tot = sum(w)
            row = []
            for d in range(len(vv[0])):
                acc = 0.0
                for j in keys:
                    acc += w[j] * vv[j][d]
                row.append(acc / tot)
            o_h.append(row)
            lse_h.append(mx + math.log(tot))
        o_all.append(o_h)
        lse_all.append(lse_h)
    lead = np.asarray(q).shape[:-2]
    S = np.asarray(q).shape[-2]
    Dv = np.asarray(v).shape[-1]
    return (np.array(o_all).reshape(lead + (S, Dv)), np.array(lse_all).reshape(lead + (S,)))


def online_softmax_attention(q, k, v, scale: float, tile: int = 128,
                             rebase_threshold: float = 8.0, causal: bool = False):
    """The pages' online-softmax recurrence, one K/V tile at a time, in fp64.

    Follows [B200-attn] Ch. 1 §B (state update per K/V tile), Ch. 8 (base-2 exponent with
    scale*log2(e) folded into one factor, row max taken on raw scores then multiplied) and
    Ch. 11 (rebase only when the new tile max exceeds the kept max by at least
    ``rebase_threshold`` base-2 units; threshold 0 rebases whenever the max grows). Keys
    past S in the last tile are excluded (they contribute nothing). Returns (o, lse) like
    :func:`attention`; the pages' claim is that the result does not depend on the
    threshold, which the tests check against the plain definition. With ``causal`` the
    scores of keys j > i are -inf before the tile max, so a tile entirely in row i's future
    leaves that row's state unchanged.
    """
    qh, kh, vh = _as_heads(q), _as_heads(k), _as_heads(v)
    n, S, _ = qh.shape
    scale_log2 = scale * LOG2E
    o_out = np.empty((n, S, vh.shape[-1]))
    lse_out = np.empty((n, S))
    for h in range(n):
        kept = np.full(S, -np.inf)            # running (kept) row max, base-2 units
        rowsum = np.zeros(S)
        acc = np.zeros((S, vh.shape[-1]))    # running unnormalised O
        for j0 in range(0, S, tile):
            j1 = min(S, j0 + tile)
            s_raw = qh[h] @ kh[h, j0:j1].T    # this tile's raw scores
            if causal:
                s_raw = np.where(np.arange(j0, j1)[None, :] > np.arange(S)[:, None], -np.inf, s_raw)
            tile_max = s_raw.max(axis=1) * scale_log2
            candidate = np.maximum(kept, tile_max)
            first = np.isneginf(kept)
            rebase = first | (candidate - kept >= rebase_threshold)
            rescale = np.where(rebase & ~first, np.exp2(kept - candidate), 1.0)
            rowsum *= rescale
            acc *= rescale[:, None]
            kept = np.where(rebase, candidate, kept)
            p = np.exp2(s_raw * scale_log2 - kept[:, None])
            rowsum += p.sum(axis=1)
            acc += p @ vh[h, j0:j1]
        o_out[h] = acc / rowsum[:, None]
        lse_out[h] = (kept + np.log2(rowsum)) * LN2
    lead = np.asarray(q).shape[:-2]
    return o_out.reshape(lead + (S, vh.shape[-1])), lse_out.reshape(lead + (S,))


def rebase_threshold_in_other_units(threshold_log2: float, head_dim: int):
    """[B200-attn] Ch. 11 'the actual threshold': a base-2 exponent gap expressed as the
    largest unnormalised P it allows, as a natural-exponent gap, and as a raw Q.K score gap
    when the softmax scale is 1/sqrt(head_dim). Returns (max_p, natural_gap, raw_gap)."""
    natural = threshold_log2 / LOG2E
    return 2.0 ** threshold_log2, natural, natural * math.sqrt(head_dim)
