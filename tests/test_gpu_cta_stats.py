"""Every CTA of a cluster rebuilds bit-identical row statistics.

The replicated push lets each of the P CTAs fold the same P partials, in
rank order, with local reads only (CREDIT summary page, "C. Cluster
Reduction and Reuse Protocol", All-Gather Trade-off and Output Generation);
the output is only consistent across a row's slices if every CTA ends up
with the same bits.  The checked build records, for each row and each rank,
the combined statistics that CTA holds (credit_debug_stats).  For cluster
sizes 2, 3 (unequal slices), 8 and 16, both exchanges, one and two rows per
cluster, L2-tail plans (also with small 128-thread CTAs), the persistent ring
and the warp-specialised kernel, every
operator: the P records of a row are bit-identical, no other rank wrote one,
and the statistics match the oracle's fp64 values of the same row (max and
absmax exactly).
"""
import numpy as np
import pytest
import torch

import oracle
from dsmem_thread_block_gb300 import _credit as C
from dsmem_thread_block_gb300 import workloads as wl

from gpu_helpers import DT, OPS, run

pytestmark = pytest.mark.gpu

ROWS = 5


def _w(op, dtype, cols, seed, **kw):
    return wl.Workload(f"{op}_{dtype}_{ROWS}x{cols}", op, dtype, ROWS, cols, seed, **kw)


WORKLOADS = [
    _w(wl.SOFTMAX, "f32", 32768, 400, x_std=4.0, spike_frac=0.01),
    _w(wl.SOFTMAX, "bf16", 65536, 401),
    _w(wl.LAYERNORM, "bf16", 65536, 402, x_mean=0.5, x_std=2.0, eps=1e-5, param_dtype="f32"),
    _w(wl.RMSNORM, "bf16", 65536, 403, eps=1e-6, param_dtype="bf16"),
    _w(wl.QUANTIZE, "f32", 32768, 404, x_std=3.0),
    _w(wl.WEIGHTED_STD, "f32", 32768, 405, x_mean=1.0, x_std=2.0, eps=1e-5, param_dtype="f32"),
    _w(wl.PEARSON, "f32", 32768, 406, x_mean=0.5, x_std=2.0, eps=1e-5),
]
RING_OPS = (wl.SOFTMAX, wl.LAYERNORM, wl.RMSNORM)
TAIL_OPS = (wl.SOFTMAX, wl.LAYERNORM, wl.RMSNORM)


def _plans(w, P):
    """(label, plan) of every kernel family at cluster size P that is legal."""
    dev = torch.cuda.current_device()
    out = []

    def add(label, variant, **kw):
        try:
            out.append((label, C.credit_plan_with(OPS[w.op], w.rows, w.cols, DT[w.dtype], dev,
                                                  variant, P, **kw)))
        except C.CreditError as e:
            assert e.status == C.ERR_NO_LEGAL_PLAN, (label, e)

    for xc, name in ((C.EXCHANGE_BARRIER, "barrier"), (C.EXCHANGE_ASYNC, "async")):
        add(f"cluster:{name}", C.CLUSTER, exchange=xc)
        if out and w.op in TAIL_OPS and (w.op != wl.SOFTMAX or w.dtype == "bf16"):
            # an L2-tail plan staging half of the slice
            vec = 4 if w.dtype == "f32" else 8
            half = max(vec, out[-1][1].slice_elems // 2 // vec * vec)
            add(f"tail:{name}", C.CLUSTER, exchange=xc, staged_elems=half)
            add(f"tail2:{name}", C.CLUSTER, exchange=xc, staged_elems=half, rows_per_cluster=2)
            # small CTAs with a long tail (the 64-register instantiation for
            # bf16 softmax and LayerNorm)
            add(f"small:{name}", C.CLUSTER, exchange=xc,
                staged_elems=max(vec, half // 2 // vec * vec), threads=128)
        if w.op != wl.PEARSON:
            add(f"cluster2:{name}", C.CLUSTER, exchange=xc, rows_per_cluster=2)
        if w.op in RING_OPS:
            add(f"persist:{name}", C.CLUSTER_PERSISTENT, exchange=xc)
    if w.op in RING_OPS:
        add("pipe", C.CLUSTER_PIPELINED)
    return out


def _oracle_stats(w, inp):
    """fp64 statistics per row, in the record's slot order."""
    x = oracle.widen(inp["x"])
    if w.op == wl.SOFTMAX:
        m = x.max(axis=1)
        return np.stack([m, np.exp(x - m[:, None]).sum(axis=1)], axis=1)
    if w.op == wl.LAYERNORM:
        mu = x.mean(axis=1)
        return np.stack([np.full(ROWS, w.cols), mu, ((x - mu[:, None]) ** 2).sum(axis=1)], axis=1)
    if w.op == wl.RMSNORM:
        return (x * x).sum(axis=1)[:, None]
    if w.op == wl.QUANTIZE:
        return np.abs(x).max(axis=1)[:, None]
    if w.op == wl.WEIGHTED_STD:
        wt = oracle.widen(inp["weight"])
        W = wt.sum()
        mu = (x * wt).sum(axis=1) / W
        return np.stack([np.full(ROWS, W), mu, (wt * (x - mu[:, None]) ** 2).sum(axis=1)], axis=1)
    u = oracle.widen(inp["u"])
    mx, mu = x.mean(axis=1), u.mean(axis=1)
    dx, du = x - mx[:, None], u - mu[:, None]
    return np.stack([np.full(ROWS, w.cols), mx, mu, (dx * dx).sum(axis=1), (du * du).sum(axis=1),
                     (dx * du).sum(axis=1)], axis=1)


def _check_against_oracle(w, inp, label, rec, want):
    """rec: [ROWS, nstats] (one CTA's record per row) vs the fp64 values:
    maxima exactly, means within 1e-5 of the row's rms (an fp32 sum errs
    relative to its summands), the rest within 1e-5 relative."""
    got = rec[:, :want.shape[1]].astype(np.float64)
    if w.op in (wl.SOFTMAX, wl.QUANTIZE):
        # the maximum is exact in any order: bit-equal to the fp32 input's
        assert np.array_equal(got[:, 0], want[:, 0]), (w.name, label)
    means = {wl.LAYERNORM: {1: "x"}, wl.WEIGHTED_STD: {1: "x"}, wl.PEARSON: {1: "x", 2: "u"}}
    for j in range(want.shape[1]):
        ref = want[:, j]
        scale = np.abs(ref)
        src = means.get(w.op, {}).get(j)
        if src:
            v = oracle.widen(inp[src])
            scale = np.sqrt((v * v).mean(axis=1))
        assert (np.abs(got[:, j] - ref) <= 1e-5 * scale + 1e-30).all(), \
            (w.name, label, j, got[:, j], ref)


@pytest.mark.parametrize("w", WORKLOADS, ids=[w.name for w in WORKLOADS])
def test_every_cta_holds_identical_statistics(w):
    inp = w.generate()
    want = _oracle_stats(w, inp)
    ran = 0
    with C.use_checked_build():
        C.credit_debug_stats()  # reset the record
        for P in (2, 3, 8, 16):
            for label, plan in _plans(w, P):
                run(w, inp, plan)
                rec = C.credit_debug_stats(ROWS)  # [ROWS, 16, 8], then reset
                bits = rec.view(np.uint32)
                for r in range(ROWS):
                    # the P records of row r: written, bit-identical, P stamped
                    assert not np.isnan(rec[r, :P, :want.shape[1]]).any(), (label, P, r)
                    assert (bits[r, :P] == bits[r, 0]).all(), \
                        f"{w.name} {label} P={P} row {r}: CTAs disagree\n{rec[r, :P]}"
                    assert (rec[r, :P, 7] == P).all()
                    # no rank outside the cluster wrote one
                    assert np.isnan(rec[r, P:, 7]).all(), (label, P, r)
                _check_against_oracle(w, inp, f"{label} P={P}", rec[:, 0], want)
                ran += 1
        assert C.credit_get_device_error(torch.cuda.current_device()) == C.OK
    assert ran >= 8
