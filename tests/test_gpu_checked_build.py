"""The checked build (libcredit_checked.so, -DCREDIT_DEBUG) on the GPU: its
index-check path records CREDIT_ERR_DEVICE_BOUNDS without touching memory;
every kernel family, run through it on legal shapes, matches the oracle with
no check firing; and its phase trace is complete and ordered."""
import numpy as np
import pytest
import torch

from dsmem_thread_block_gb300 import _credit as C
from dsmem_thread_block_gb300 import trace as T
from dsmem_thread_block_gb300 import workloads as wl

from gpu_helpers import DT, OPS, check, check_pearson, check_quant, make_plan, run

pytestmark = pytest.mark.gpu


def _w(op, dtype, rows, cols, seed, **kw):
    return wl.Workload(f"{op}_{dtype}_{rows}x{cols}", op, dtype, rows, cols, seed, **kw)


def test_bounds_selftest_records_and_clears():
    dev = torch.cuda.current_device()
    with C.use_checked_build():
        assert C.credit_debug_build() == 1
        assert C.credit_selftest_bounds(dev) == C.ERR_DEVICE_BOUNDS
        assert C.credit_get_device_error(dev) == C.OK  # read and cleared


def _plan_with(w, variant, P, **kw):
    dev = torch.cuda.current_device()
    return C.credit_plan_with(OPS[w.op], w.rows, w.cols, DT[w.dtype], dev, variant, P, **kw)


def test_every_kernel_family_passes_its_checks():
    dev = torch.cuda.current_device()
    ln = _w(wl.LAYERNORM, "bf16", 9, 65536, 300, x_mean=0.5, x_std=2.0, eps=1e-5, param_dtype="f32")
    sm = _w(wl.SOFTMAX, "f32", 7, 32768, 301, x_std=4.0, spike_frac=0.01)
    sm4 = _w(wl.SOFTMAX, "f32", 7, 8192, 307, x_std=4.0)
    rms = _w(wl.RMSNORM, "bf16", 3, 786432, 302, eps=1e-6, param_dtype="bf16")
    rag = _w(wl.SOFTMAX, "bf16", 3, 10001, 303)
    q = _w(wl.QUANTIZE, "f32", 5, 65536, 304, x_std=3.0)
    ws = _w(wl.WEIGHTED_STD, "f32", 5, 40960, 305, x_mean=1.0, x_std=2.0, eps=1e-5,
            param_dtype="f32")
    pe = _w(wl.PEARSON, "f32", 4, 65536, 306, x_mean=0.5, x_std=2.0, eps=1e-5)
    with C.use_checked_build():
        cases = [
            (ln, make_plan(ln, C.CLUSTER, 8)),
            (ln, _plan_with(ln, C.CLUSTER, 4, rows_per_cluster=2)),
            (ln, make_plan(ln, C.CLUSTER_PERSISTENT, 4)),
            (ln, make_plan(ln, C.CLUSTER_PIPELINED, 4)),
            (ln, make_plan(ln, C.TWO_PASS)),
            (sm, make_plan(sm, C.CLUSTER, 3)),
            (sm4, _plan_with(sm4, C.CLUSTER, 1, rows_per_cluster=4)),
            (sm, _plan_with(sm, C.CLUSTER, 4, exchange=C.EXCHANGE_BARRIER)),
            (rms, make_plan(rms, C.CLUSTER, 16)),
            (rag, make_plan(rag, C.CLUSTER, 3)),
        ]
        for w, p in cases:
            inp = w.generate()
            check(w, run(w, inp, p), inp)
        inp = q.generate()
        check_quant(run(q, inp, make_plan(q, C.CLUSTER, 6)), inp)
        inp = ws.generate()
        check(ws, run(ws, inp, make_plan(ws, C.CLUSTER, 5)), inp)
        inp = pe.generate()
        check_pearson(pe, run(pe, inp, make_plan(pe, C.CLUSTER, 7)), inp)
        assert C.credit_get_device_error(dev) == C.OK


def test_phase_trace_is_complete_and_ordered():
    r = T.run("softmax_f32_64x4096", 4)
    assert r["device_error"] == C.status_string(C.OK)
    assert r["ctas"] == 64 * 4 and r["sms"] >= 2
    assert all(v >= 0 for v in r["phase_median_us"].values())
    assert 0 < r["cta_life_median_us"] < r["span_us"] + 1e-9
    # the raw stamps: every CTA wrote all seven, in order
    with C.use_checked_build():
        s = C.credit_debug_trace(64 * 4)
    assert (s[:, :7] > 0).all()
    assert (np.diff(s[:, :7], axis=1) >= 0).all()
