"""Host logic of the phase-trace summary (no GPU): phase medians, CTA
lifetimes, idle gaps between consecutive CTAs on an SM and each SM's busy
share, on hand-made stamps."""
import numpy as np

from dsmem_thread_block_gb300 import trace as T


def _cta(t0, phases, sm):
    t = [t0]
    for p in phases:
        t.append(t[-1] + p)
    return t + [sm]


def test_summary_of_hand_made_stamps():
    # SM 0 runs two CTAs back to back with a 500 ns gap; SM 1 runs two that
    # overlap; every CTA has phases 100, 200, 300, 400, 500, 600 ns
    ph = [100, 200, 300, 400, 500, 600]  # life 2100 ns
    rows = [_cta(1000, ph, 0), _cta(1000 + 2100 + 500, ph, 0),
            _cta(1000, ph, 1), _cta(2000, ph, 1)]
    s = T.summarize(np.array(rows, dtype=np.int64))
    assert s["ctas"] == 4 and s["sms"] == 2
    assert s["phase_median_us"] == {n: p / 1000 for n, p in zip(T.PHASES, ph)}
    assert s["cta_life_median_us"] == 2.1
    # span: first entry to last exit = 2100 + 500 + 2100 ns
    assert abs(s["span_us"] - 4.7) < 1e-9
    # only SM 0 has a gap (SM 1's CTAs overlap)
    assert s["sm_gap_median_us"] == 0.5
    # SM 0 busy 4200 of 4700 ns, SM 1 busy all of its 3100 ns
    assert abs(s["sm_busy_share_median"] - round((4200 / 4700 + 1.0) / 2, 4)) < 1e-4
