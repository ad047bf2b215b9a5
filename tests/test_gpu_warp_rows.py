"""GPU parity of the warp-per-row kernel (CREDIT_WARP_ROWS): a warp holds a
whole row in registers, reduces it with shuffles and writes it.  Softmax
(fp32 with spikes, bf16), LayerNorm and RMSNorm with fp32, bf16 or absent
parameters against the oracle; row widths from one vector per lane to the
4 KiB limit, rows that leave lanes idle, row counts below and far above one
warp per resident slot (the grid strides), in place, constant rows; the
misaligned fallback and the shapes it does not take; the cost model and the
static rule choosing it for narrow rows."""
import numpy as np
import pytest
import torch

from dsmem_thread_block_gb300 import _credit as C
from dsmem_thread_block_gb300 import workloads as wl

from gpu_helpers import DT, OPS, call, check, run, to_host

pytestmark = pytest.mark.gpu


def _w(op, dtype, rows, cols, seed, **kw):
    return wl.Workload(f"{op}_{dtype}_{rows}x{cols}", op, dtype, rows, cols, seed, **kw)


def _plan(w):
    return C.credit_plan_for(OPS[w.op], w.rows, w.cols, DT[w.dtype],
                             torch.cuda.current_device(), C.WARP_ROWS, 1)


CASES = [
    _w(wl.SOFTMAX, "f32", 3001, 1024, 400, x_std=4.0, spike_frac=0.01),
    _w(wl.SOFTMAX, "bf16", 2000, 2048, 401),
    _w(wl.SOFTMAX, "bf16", 777, 8, 402),          # one vector per row: 31 idle lanes
    _w(wl.SOFTMAX, "f32", 513, 100, 403),         # 25 vectors: a partial first pass
    _w(wl.LAYERNORM, "bf16", 1500, 1024, 404, x_mean=0.5, x_std=2.0, eps=1e-5, param_dtype="f32"),
    _w(wl.LAYERNORM, "f32", 700, 1000, 405, x_mean=-1.0, x_std=3.0, eps=1e-5, param_dtype="bf16"),
    _w(wl.RMSNORM, "bf16", 1300, 2048, 406, eps=1e-6, param_dtype="bf16"),
    _w(wl.RMSNORM, "f32", 900, 512, 407, eps=1e-6, param_dtype="f32"),
]


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_warp_rows_parity(w):
    inp = w.generate()
    p = _plan(w)
    assert p.variant == C.WARP_ROWS and p.cluster_size == 1 and p.smem_bytes == 0
    check(w, run(w, inp, p), inp)


def test_warp_rows_absent_parameters_in_place_and_constant_rows():
    w = _w(wl.LAYERNORM, "bf16", 300, 1024, 408, x_mean=0.5, x_std=2.0, eps=1e-5,
           param_dtype="f32")
    inp = {"x": w.generate()["x"]}
    check(w, run(w, inp, _plan(w)), inp)
    r = _w(wl.RMSNORM, "f32", 300, 1024, 409, eps=1e-6, param_dtype="f32")
    rin = r.generate()
    check(r, run(r, rin, _plan(r), in_place=True), rin)
    s = _w(wl.SOFTMAX, "f32", 64, 1024, 410)
    sin = s.generate()
    sin["x"][:8] = 3.25  # constant rows: a uniform softmax
    got = run(s, sin, _plan(s))
    assert np.allclose(got[:8], 1.0 / 1024, rtol=1e-6)
    check(s, got, sin)


def test_warp_rows_many_rows_per_warp():
    # far more rows than resident warps: each warp strides over many rows
    w = _w(wl.SOFTMAX, "bf16", 300000, 128, 411)
    inp = w.generate()
    p = _plan(w)
    assert p.waves > 4
    check(w, run(w, inp, p), inp, rows=np.arange(0, w.rows, 997))


def test_warp_rows_limits_and_fallback():
    dev = torch.cuda.current_device()
    # wider than 4 KiB, and operators the kernel does not run
    with pytest.raises(C.CreditError) as e:
        C.credit_plan_for(C.SOFTMAX, 8, 2048 + 4, C.F32, dev, C.WARP_ROWS, 1)
    assert e.value.status == C.ERR_NO_LEGAL_PLAN
    for op in (C.QUANTIZE, C.WEIGHTED_STD, C.PEARSON):
        with pytest.raises(C.CreditError) as e:
            C.credit_plan_for(op, 8, 1024, C.F32, dev, C.WARP_ROWS, 1)
        assert e.value.status == C.ERR_NO_LEGAL_PLAN
    with pytest.raises(C.CreditError) as e:  # no exchange to choose
        C.credit_plan_with(C.SOFTMAX, 8, 1024, C.F32, dev, C.WARP_ROWS, 1,
                           exchange=C.EXCHANGE_ASYNC)
    assert e.value.status == C.ERR_INVALID_ARG
    # a misaligned row runs the one-CTA element path instead
    w = _w(wl.SOFTMAX, "f32", 33, 1024, 412, x_std=3.0)
    inp = w.generate()
    dx = torch.from_numpy(np.concatenate([np.zeros(1, np.float32), inp["x"].reshape(-1)])).cuda()[1:]
    dy = torch.empty(dx.numel() + 1, device="cuda")[1:]
    assert call(w, dx, dy, {}, _plan(w)) == C.OK
    torch.cuda.synchronize()
    check(w, to_host(dy).reshape(w.rows, w.cols), inp)
    assert C.credit_get_device_error(dev) == C.OK


def test_cost_model_and_static_plan_take_warp_rows_for_narrow_rows():
    # 2 KiB bf16 rows: the cost model times the warp-per-row kernel as a
    # baseline candidate (measured 1.5x the one-CTA staging kernel there),
    # and the static rule picks it without a profile
    dev = torch.cuda.current_device()
    plan, rep = C.credit_plan_profiled(C.SOFTMAX, 65536, 1024, C.BF16, -1, dev, 5, 0)
    assert rep.baseline_variant == C.WARP_ROWS
    assert rep.b_base_bytes == rep.b_credit_bytes  # one read, one write
    assert plan.variant == C.WARP_ROWS  # no clustered candidate beats it
    auto = C.credit_plan(C.LAYERNORM, 1001, 1024, C.BF16, dev)
    assert auto.variant == C.WARP_ROWS
    wide = C.credit_plan(C.LAYERNORM, 1001, 4096, C.BF16, dev)
    assert wide.variant == C.CLUSTER
