"""Host logic of the profitability sweep's summary (no GPU): pick and
profitability accuracy, the misses within 2 % of parity, and the predicted
and measured crossover widths, on hand-made points."""
from dsmem_thread_block_gb300 import sweep


def _pt(cols, predicted, measured, correct, tuned, gap):
    return {"cols": cols, "predicted_profitable": predicted, "measured_profitable": measured,
            "correct": correct, "tuned_correct": tuned,
            "profitability_correct": predicted == measured, "parity_gap": gap}


def test_summary_of_hand_made_points():
    pts = [_pt(1024, False, False, True, True, -3.0),
           _pt(2048, False, True, False, True, 0.015),   # a miss within 2 % of parity
           _pt(4096, False, True, False, True, 0.30),    # a miss outside it
           _pt(8192, True, True, True, False, 0.50),
           _pt(16384, True, True, True, True, 0.51)]
    s = sweep.summarize(pts)
    assert s["points"] == 5
    assert s["pick_accuracy"] == 3 / 5
    assert s["tuned_pick_accuracy"] == 4 / 5
    assert s["profitability_accuracy"] == 3 / 5
    assert s["profitability_errors_within_2pct"] == 1
    assert s["predicted_crossover_cols"] == 8192 and s["measured_crossover_cols"] == 2048
    assert s["crossover_interval_error"] == 2  # 2048 -> 8192: two doublings


def test_summary_without_a_profitable_width():
    pts = [_pt(1024, False, False, True, True, None), _pt(2048, False, False, True, True, None)]
    s = sweep.summarize(pts)
    assert s["predicted_crossover_cols"] is None and s["crossover_interval_error"] is None
    assert s["profitability_accuracy"] == 1.0
