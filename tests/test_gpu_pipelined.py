"""GPU parity of the warp-specialised persistent kernel (CREDIT_CLUSTER_PIPELINED):
reducer warps fold, exchange and combine one row while storer warps write the
previous one.  Every operator it runs (softmax fp32 / bf16, LayerNorm and
RMSNorm with fp32, bf16 or absent parameters) against the oracle at cluster
sizes with ragged last slices; row counts from one to many rows per cluster
(hand-off, ring and mbarrier-phase reuse); the smallest and largest reducer /
storer splits; one and two CTAs per SM; the operators and requests it does not
offer; the misaligned fallback."""
import itertools

import numpy as np
import pytest
import torch

from dsmem_thread_block_gb300 import _credit as C
from dsmem_thread_block_gb300 import workloads as wl

from gpu_helpers import DT, OPS, call, check, run, to_device, to_host

pytestmark = pytest.mark.gpu


def _w(op, dtype, rows, cols, seed, **kw):
    return wl.Workload(f"{op}_{dtype}_{rows}x{cols}", op, dtype, rows, cols, seed, **kw)


def _plan(w, P, **kw):
    dev = torch.cuda.current_device()
    try:
        return C.credit_plan_with(OPS[w.op], w.rows, w.cols, DT[w.dtype], dev,
                                  C.CLUSTER_PIPELINED, P, **kw)
    except C.CreditError as e:
        assert e.status == C.ERR_NO_LEGAL_PLAN
        return None


CASES = [
    _w(wl.SOFTMAX, "f32", 37, 65536, 200, x_std=4.0, spike_frac=0.01),
    _w(wl.SOFTMAX, "bf16", 41, 131072, 201),
    _w(wl.LAYERNORM, "bf16", 29, 98304, 202, x_mean=0.5, x_std=2.0, eps=1e-5, param_dtype="f32"),
    _w(wl.LAYERNORM, "f32", 23, 49152, 203, x_mean=-1.0, x_std=3.0, eps=1e-5, param_dtype="bf16"),
    _w(wl.RMSNORM, "bf16", 33, 196608, 204, eps=1e-6, param_dtype="bf16"),
    _w(wl.RMSNORM, "f32", 19, 40960, 205, eps=1e-6, param_dtype="f32"),
]


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_pipelined_parity(w):
    inp = w.generate()
    ran = 0
    for P in (1, 2, 3, 5, 8, 9, 16):
        p = _plan(w, P)
        if p is None:
            continue
        assert p.variant == C.CLUSTER_PIPELINED and p.exchange == C.EXCHANGE_ASYNC
        check(w, run(w, inp, p), inp)
        ran += 1
    assert ran >= 4


def test_pipelined_absent_parameters():
    w = _w(wl.LAYERNORM, "bf16", 17, 65536, 206, x_mean=0.5, x_std=2.0, eps=1e-5,
           param_dtype="f32")
    inp = {"x": w.generate()["x"]}
    r = _w(wl.RMSNORM, "bf16", 17, 65536, 207, eps=1e-6, param_dtype="bf16")
    rin = {"x": r.generate()["x"]}
    for P in (2, 4):
        check(w, run(w, inp, _plan(w, P)), inp)
        check(r, run(r, rin, _plan(r, P)), rin)


@pytest.mark.parametrize("rows", [1, 3, 150])
def test_pipelined_row_counts_and_role_splits(rows):
    # fewer rows than clusters, a few, and many rows per cluster; threads
    # from one reducer + one storer warp up to sixteen consumer warps; one
    # and two CTAs per SM
    w = _w(wl.LAYERNORM, "bf16", rows, 32768, 208, x_mean=0.5, x_std=2.0, eps=1e-5,
           param_dtype="f32")
    s = _w(wl.SOFTMAX, "bf16", rows, 32768, 209)
    ran = 0
    for wk in (w, s):
        inp = wk.generate()
        for P, threads, cps in itertools.product((1, 2, 4, 8), (96, 288, 544), (1, 2)):
            if cps == 2 and threads > 288:
                continue
            p = _plan(wk, P, threads=threads, ctas_per_sm=cps)
            if p is None:
                continue
            assert p.threads == threads
            check(wk, run(wk, inp, p), inp)
            ran += 1
    assert ran >= 24


def test_pipelined_chunked_ring_one_row_slot():
    # a slice of many chunk slots with a ring that holds one row: the next
    # row's chunks land only as the storers release them
    w = _w(wl.SOFTMAX, "bf16", 40, 1 << 20, 210)
    inp = w.generate()
    p = _plan(w, 10)
    assert p is not None
    assert p.ring_slots * p.chunk_elems < 2 * p.slice_elems  # one row slot
    check(w, run(w, inp, p), inp)


def test_pipelined_requests_and_operators_not_offered():
    dev = torch.cuda.current_device()
    with pytest.raises(C.CreditError) as e:
        C.credit_plan_with(C.SOFTMAX, 8, 65536, C.F32, dev, C.CLUSTER_PIPELINED, 4,
                           exchange=C.EXCHANGE_BARRIER)
    assert e.value.status == C.ERR_INVALID_ARG
    with pytest.raises(C.CreditError) as e:  # a producer, a reducer and a storer warp at least
        C.credit_plan_with(C.SOFTMAX, 8, 65536, C.F32, dev, C.CLUSTER_PIPELINED, 4, threads=64)
    assert e.value.status == C.ERR_INVALID_ARG
    for op in (C.QUANTIZE, C.WEIGHTED_STD, C.PEARSON):
        with pytest.raises(C.CreditError) as e:
            C.credit_plan_for(op, 8, 65536, C.F32, dev, C.CLUSTER_PIPELINED, 4)
        assert e.value.status == C.ERR_NO_LEGAL_PLAN


def test_pipelined_misaligned_falls_back_to_element_path():
    # x one element past a 16-byte boundary: bulk copies cannot stage it, so
    # the call runs the one-row-per-cluster element path with the same P
    w = _w(wl.SOFTMAX, "f32", 5, 16384, 211, x_std=3.0)
    inp = w.generate()
    p = _plan(w, 4)
    dx = torch.from_numpy(np.concatenate([np.zeros(1, np.float32), inp["x"].reshape(-1)])).cuda()[1:]
    dy = torch.empty(dx.numel() + 1, device="cuda")[1:]
    assert call(w, dx, dy, {}, p) == C.OK
    torch.cuda.synchronize()
    check(w, to_host(dy).reshape(w.rows, w.cols), inp)
    assert C.credit_get_device_error(torch.cuda.current_device()) == C.OK


def test_pipelined_in_place():
    w = _w(wl.RMSNORM, "bf16", 12, 131072, 212, eps=1e-6, param_dtype="bf16")
    inp = w.generate()
    check(w, run(w, inp, _plan(w, 4), in_place=True), inp)


def test_pipelined_staged_parameters():
    # the storers copy each CTA's parameter slice into shared memory once:
    # slices whose parameter bytes start 8 bytes past a 16-byte boundary
    # (fp32 data, bf16 parameters, slice = 4 mod 8) take the element copy;
    # gamma without beta; many rows per cluster reuse the staged copy
    dev = torch.cuda.current_device()
    w = _w(wl.LAYERNORM, "f32", 64, 8200, 213, x_mean=-1.0, x_std=3.0, eps=1e-5,
           param_dtype="bf16")
    inp = w.generate()
    g_only = {k: v for k, v in inp.items() if k != "beta"}
    ran = 0
    for P in (2, 3, 6):
        p = _plan(w, P)
        if p is None:
            continue
        ring = p.ring_slots * p.chunk_elems * 4
        assert p.smem_bytes > ring  # a parameter room follows the ring
        check(w, run(w, inp, p), inp)
        check(w, run(w, g_only, p), g_only)
        ran += 1
    assert ran >= 2
    assert C.credit_get_device_error(dev) == C.OK
