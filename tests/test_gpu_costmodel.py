"""The profiling-fed cost model: its report is consistent, its choice is a
legal plan that the automatic planner then reuses, and on the full bf16
softmax profitability sweep its untimed prediction gets profitability and
the crossover right and its pick stays close to the fastest candidate."""
import pytest
import torch

from dsmem_thread_block_gb300 import _credit as C
from dsmem_thread_block_gb300 import sweep
from dsmem_thread_block_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def test_report_is_consistent_and_choice_is_cached():
    rows, cols = 256, 131072  # 256 KiB bf16 rows: the baseline is the two-pass pair
    C.credit_calibrate(0, 3)
    plan, rep = C.credit_plan_profiled(C.SOFTMAX, rows, cols, C.BF16, -1, 0, 3, 0)
    assert rep.baseline_variant == C.TWO_PASS
    assert rep.cand[0].legal and rep.cand[0].pred_us == rep.t_base_us > 0
    legal = [c for c in rep.cand[1:] if c.legal]
    assert legal, "some cluster size must fit a 256 KiB row"
    best = min([rep.t_base_us] + [c.pred_us for c in legal])
    assert abs(plan.pred_us - best) <= 1e-3 * best + 1e-3
    assert rep.model_cluster_size == rep.chosen_cluster_size  # no tuning requested
    assert rep.chosen_cluster_size == plan.cluster_size or (
        rep.chosen_cluster_size == 1 and plan.variant == C.TWO_PASS)
    auto = C.credit_plan(C.SOFTMAX, rows, cols, C.BF16, 0)
    assert auto.variant == plan.variant and auto.cluster_size == plan.cluster_size


def test_local_staging_baseline_for_narrow_rows():
    plan, rep = C.credit_plan_profiled(C.LAYERNORM, 4096, 4096, C.BF16, C.F32, 0, 3, 0)
    assert rep.baseline_variant == C.CLUSTER and rep.cand[0].plan.cluster_size == 1
    assert rep.b_base_bytes == rep.b_credit_bytes


def test_tuning_times_the_top_candidates():
    plan, rep = C.credit_plan_profiled(C.LAYERNORM, 256, 262144, C.BF16, C.F32, 0, 3, 3)
    timed = [c for c in rep.cand[1:] if c.legal and c.measured_us > 0]
    assert 1 <= len(timed) <= 3
    best = min([rep.t_base_us] + [c.measured_us for c in timed] +
               [c.persistent_us for c in timed if c.persistent_us > 0] +
               [c.pipelined_us for c in timed if c.pipelined_us > 0] +
               [c.tail_us for c in timed if c.tail_us > 0])
    # the plan carries its measured time: the mean of three medians of the
    # confirmation round, which re-times the fastest plans of the first
    assert best * 0.9 <= plan.pred_us <= best * 1.1 + 1e-3
    assert plan.cluster_size == rep.chosen_cluster_size or plan.variant == C.TWO_PASS


def test_softmax_sweep_profitability_and_crossover_at_full_size():
    # the bf16 softmax profitability sweep as specified: 2^28 elements, 1024 to
    # 1048576 columns.  The model alone -- primitives measured on calibration
    # shapes, one timing of the non-DSMEM baseline, no timing of any clustered
    # candidate -- decides clustered or not; then every staging form of every
    # legal cluster size is timed ("C. Cost-Model Validation": profitability
    # accuracy and crossover prediction)
    C.credit_calibrate(0, 7)
    pts = [sweep.run_point(c, runs=7) for c in wl.SWEEP_COLS]
    s = sweep.summarize(pts)
    report = [(p["cols"], p["picked_variant"], round(p["picked_us"], 1), p["measured_best_variant"],
               round(p["best_us"], 1), p["predicted_profitable"], p["measured_profitable"])
              for p in pts]
    print(s, report)
    # profitability right at >= 90 % of the widths; a miss where the best
    # clustered candidate and the baseline are within 2 % of each other is a
    # tie that timing noise decides, as the pages count it
    hard = [p for p in pts if not p["profitability_correct"] and
            (p["parity_gap"] is None or abs(p["parity_gap"]) > 0.02)]
    assert len(pts) - len(hard) >= 0.9 * len(pts), (s, report)
    # the predicted crossover (smallest profitable width) lands within one x2
    # interval of the measured one
    assert s["crossover_interval_error"] is not None and s["crossover_interval_error"] <= 1, (s, report)
    # the model's own pick, untimed, is never far from the fastest candidate
    for p in pts:
        assert p["picked_us"] <= 1.15 * p["best_us"], (p["cols"], report)
    torch.cuda.synchronize()


def test_stage_copy_rate_residency_and_bounds():
    # the staged-copy primitive: the footprint sets the residency asked for;
    # bulk-copy staging streams near the copy roofline at any residency (the
    # measured spread from one to eight CTAs per SM is a few percent)
    rates = {}
    for k in (1, 3, 8):
        g, res = C.credit_stage_copy_rate(0, k, 3)
        assert res == k, (k, res)
        assert 3000.0 < g < 9000.0
        rates[k] = g
    assert min(rates.values()) > 0.8 * max(rates.values())
    with pytest.raises(C.CreditError):
        C.credit_stage_copy_rate(0, 9, 3)
    torch.cuda.synchronize()


def test_large_shape_is_timed_on_its_first_rows():
    # 8 GiB of bf16 input: the model times the first 1 GiB of rows and plans
    # the chosen configuration for every row
    rows, cols = 8192, 524288
    plan, rep = C.credit_plan_profiled(C.RMSNORM, rows, cols, C.BF16, C.BF16, 0, 3, 2)
    assert rep.t_base_us > 0
    if plan.variant == C.CLUSTER:
        assert plan.waves == -(-rows // (plan.active_clusters * plan.rows_per_cluster))
    elif plan.variant in (C.CLUSTER_PERSISTENT, C.CLUSTER_PIPELINED):
        assert plan.waves == -(-rows // plan.active_clusters)
    auto = C.credit_plan(C.RMSNORM, rows, cols, C.BF16, 0)
    assert auto.variant == plan.variant and auto.cluster_size == plan.cluster_size
    torch.cuda.synchronize()
