"""The timeline tool's host arithmetic on a synthetic trace (CPU): phase means of the first
item, the time per item, and the gap between CTAs that share an SM."""
import numpy as np

from dense_attention_forward_gb300.trace import WORDS, summarize


def pad(t):
    """Words 0-7 given, the item-boundary words 8-15 zero (one item per CTA, or not reached)."""
    return np.concatenate([t, np.zeros((t.shape[0], WORDS - t.shape[1]), dtype=np.int64)], axis=1)


def test_summarize_synthetic_trace():
    # words: entry, setup, first S, O0 full, O1 full (first item), before final barrier, SM id,
    # exit (ns). Two CTAs on two SMs, 4 items: 2 per CTA.
    t = pad(np.array([
        [0, 200, 2200, 50000, 50800, 101000, 0, 102000],
        [0, 300, 2300, 50100, 50900, 101200, 1, 102100],
    ], dtype=np.int64))
    d = summarize(t, 4, 2, "synthetic")
    assert d["items"] == 4 and d["ctas"] == 2 and d["ctas_traced"] == 2 and d["sms"] == 2
    assert d["items_per_cta"] == 2.0
    assert d["setup_us"] == 0.25 and d["to_first_s_us"] == 2.0
    assert d["first_item_kv_loop_us"] == 47.8
    assert d["o0_to_o1_us"] == 0.8
    assert d["later_items_us"] == 50.25          # from the later of O0 / O1 full to the final barrier
    assert d["per_item_us"] == 50.55             # (101000 + 101200) / 2 / 2 ns
    assert d["final_barrier_to_exit_us"] == 0.95
    assert d["gap_between_ctas_us"] is None      # one CTA per SM
    assert d["span_us"] == 102.1 and d["all_exited"]


def test_summarize_gap_between_ctas_on_one_sm():
    t = pad(np.array([
        [0, 200, 2200, 50000, 50800, 51000, 0, 52000],
        [52800, 53000, 55000, 103000, 103800, 104000, 0, 105000],   # next CTA on SM 0: gap 800
    ], dtype=np.int64))
    d = summarize(t, 2, 2, "synthetic")
    assert d["gap_between_ctas_us"] == 0.8 and d["items_per_cta"] == 1.0


def test_summarize_item_boundary():
    # Words 8-15 of two CTAs with a second item; the medians are taken relative to word 8, with
    # word 3 (O tile 0 full) as the O-full time of the first item.
    base = [0, 200, 2200, 50000, 50800, 101000, 0, 102000]
    rows = []
    for shift, sm in ((0, 0), (100, 1)):
        w = base.copy()
        w[6] = sm
        w[3] = 49000 + 1310 + shift
        # 8 last S, 9 last P, 10 O read, 11 epilogue done, 12 next S, 13 next P0, 14 next QK, 15 next PV0
        w += [49000 + shift, 49670 + shift, 50570 + shift, 51400 + shift, 51850 + shift, 52140 + shift,
              50600 + shift, 52420 + shift]
        rows.append(w)
    d = summarize(np.array(rows, dtype=np.int64), 4, 2, "synthetic")
    b = d["boundary"]
    assert b["ctas"] == 2
    assert b["last_p_stored_us"] == 0.67 and b["o_full_us"] == 1.31 and b["o_read_us"] == 1.57
    assert b["epilogue_done_us"] == 2.4 and b["next_qk_issued_us"] == 1.6 and b["next_s_seen_us"] == 2.85
    assert b["next_p_stored_us"] == 3.14 and b["next_pv_issued_us"] == 3.42


def test_summarize_without_a_second_item():
    t = pad(np.array([[0, 200, 2200, 50000, 50800, 51000, 0, 52000]], dtype=np.int64))
    assert summarize(t, 1, 1, "synthetic")["boundary"] is None
