"""The timeline tool's host arithmetic on a synthetic trace (CPU): phase means and the gap
between one CTA's exit and the next CTA's entry on the same SM."""
import numpy as np

from dense_attention_forward_gb300.trace import summarize


def test_summarize_synthetic_trace():
    # words: entry, setup, first S, O0 full, O1 full, before final barrier, SM id, exit (ns)
    t = np.array([
        [0, 200, 2200, 50000, 50800, 51000, 0, 52000],
        [0, 300, 2300, 50100, 50900, 51200, 1, 52100],
        [52800, 53000, 55000, 103000, 103800, 104000, 0, 105000],    # next CTA on SM 0: gap 800
        [53100, 53300, 55300, 103300, 104100, 104300, 1, 105300],    # next CTA on SM 1: gap 1000
    ], dtype=np.int64)
    d = summarize(t, 4, "synthetic")
    assert d["ctas"] == 4 and d["ctas_traced"] == 4 and d["sms"] == 2
    assert d["setup_us"] == 0.225 and d["to_first_s_us"] == 2.0   # (200 + 300 + 200 + 200) / 4 ns
    assert d["kv_loop_us"] == 47.9        # (47800 + 47800 + 48000 + 48000) / 4 ns
    assert d["o0_to_o1_us"] == 0.8
    assert d["to_final_barrier_us"] == 0.225   # from the later of O0 / O1 full
    assert d["final_barrier_to_exit_us"] == 0.975
    assert d["gap_between_ctas_us"] == 0.9
    assert d["span_us"] == 105.3 and d["all_exited"]
    assert d["cta_us"] == 52.125
