"""GPU parity of the Pearson correlation operator (two staged operands):
every legal cluster size with both exchanges, the two-pass baseline, the
element path for ragged rows, in-place calls on either operand, constant
operands, more rows than one two-pass grid holds, argument checks, and the
full-size workload on sampled rows in the benchmark's launch configuration."""
import numpy as np
import pytest
import torch

from dsmem_thread_block_gb300 import _credit as C
from dsmem_thread_block_gb300 import workloads as wl

from gpu_helpers import DT, OPS, check_pearson, make_plan, run

pytestmark = pytest.mark.gpu


def _w(dtype, rows, cols, seed, **kw):
    kw.setdefault("x_mean", 0.5)
    kw.setdefault("x_std", 2.0)
    kw.setdefault("eps", 1e-5)
    return wl.Workload(f"pearson_{dtype}_{rows}x{cols}", wl.PEARSON, dtype, rows, cols, seed, **kw)


def _plans(w, sizes=(1, 2, 3, 4, 5, 8, 16)):
    dev = torch.cuda.current_device()
    out = []
    for P in sizes:
        for xc in (C.EXCHANGE_BARRIER, C.EXCHANGE_ASYNC):
            try:
                out.append(C.credit_plan_with(OPS[w.op], w.rows, w.cols, DT[w.dtype], dev,
                                              C.CLUSTER, P, exchange=xc))
            except C.CreditError as e:
                assert e.status == C.ERR_NO_LEGAL_PLAN
    out.append(make_plan(w, C.TWO_PASS))
    return out


CASES = [wl.PEARSON_F32_4096x65536.with_rows(5),
         _w("bf16", 4, 131072, 70),
         _w("f32", 3, 4096, 71, u_corr=-0.3),
         _w("f32", 3, 10001, 72),            # ragged: element path
         _w("bf16", 2, 1001, 73),
         _w("bf16", 3, 1000, 74)]            # 16-byte rows, ragged slices


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_pearson_parity(w):
    inp = w.generate()
    plans = _plans(w)
    assert len(plans) >= 4
    for p in plans:
        check_pearson(w, run(w, inp, p), inp)


def test_pearson_in_place_on_either_operand():
    w = _w("f32", 3, 32768, 75)
    inp = w.generate()
    for p in (make_plan(w, C.CLUSTER, 4), make_plan(w, C.TWO_PASS)):
        check_pearson(w, run(w, inp, p, in_place="x"), inp)
        check_pearson(w, run(w, inp, p, in_place="u"), inp)


def test_pearson_constant_operand_and_perfect_correlation():
    w = _w("f32", 3, 16384, 76)
    inp = w.generate()
    inp["u"][0] = 2.0                                   # constant: y = 0, r = 0
    inp["u"][1] = 3.0 * inp["x"][1] + 1.0               # linear: r = 1
    inp["u"][2] = -inp["x"][2]                          # r = -1 exactly
    for p in (make_plan(w, C.CLUSTER, 2), make_plan(w, C.CLUSTER, 8), make_plan(w, C.TWO_PASS)):
        y, r = run(w, inp, p)
        assert (y[0] == 0).all() and r[0] == 0.0
        assert abs(r[1] - 1.0) < 1e-5 and abs(r[2] + 1.0) < 1e-5
        check_pearson(w, (y, r), inp)


def test_pearson_more_rows_than_one_two_pass_grid():
    # the two-pass grid holds 65535 rows: later batches offset x, u, y, r
    # and the 8-float workspace partials
    w = _w("f32", 70000, 16, 77)
    inp = w.generate()
    check_pearson(w, run(w, inp, make_plan(w, C.TWO_PASS)), inp)
    check_pearson(w, run(w, inp, make_plan(w, C.CLUSTER, 1)), inp)


def test_pearson_argument_checks():
    dev = torch.cuda.current_device()
    x = torch.zeros(4, 4096, device="cuda")
    u = torch.zeros(4, 4096, device="cuda")
    y = torch.zeros(4, 4096, device="cuda")
    r = torch.zeros(4, device="cuda")
    ok = C.credit_pearson(x.data_ptr(), u.data_ptr(), y.data_ptr(), r.data_ptr(), 4, 4096, C.F32,
                          1e-5)
    assert ok == C.OK
    # missing u or r
    assert C.credit_pearson(x.data_ptr(), 0, y.data_ptr(), r.data_ptr(), 4, 4096, C.F32,
                            1e-5) == C.ERR_INVALID_ARG
    assert C.credit_pearson(x.data_ptr(), u.data_ptr(), y.data_ptr(), 0, 4, 4096, C.F32,
                            1e-5) == C.ERR_INVALID_ARG
    # y partially overlapping u; r inside y
    assert C.credit_pearson(x.data_ptr(), u.data_ptr(), u.data_ptr() + 64, r.data_ptr(), 3, 4096,
                            C.F32, 1e-5) == C.ERR_INVALID_ARG
    assert C.credit_pearson(x.data_ptr(), u.data_ptr(), y.data_ptr(), y.data_ptr(), 4, 4096,
                            C.F32, 1e-5) == C.ERR_INVALID_ARG
    assert C.credit_pearson(x.data_ptr(), u.data_ptr(), y.data_ptr(), r.data_ptr(), 4, 4096,
                            C.F32, -1.0) == C.ERR_INVALID_ARG
    # several rows per cluster and the persistent kernel are not offered
    with pytest.raises(C.CreditError) as e:
        C.credit_plan_with(C.PEARSON, 4, 4096, C.F32, dev, C.CLUSTER, 2, rows_per_cluster=2)
    assert e.value.status == C.ERR_INVALID_ARG
    with pytest.raises(C.CreditError) as e:
        C.credit_plan_for(C.PEARSON, 4, 4096, C.F32, dev, C.CLUSTER_PERSISTENT, 2)
    assert e.value.status == C.ERR_NO_LEGAL_PLAN
    torch.cuda.synchronize()
    assert C.credit_get_device_error(dev) == C.OK


def test_pearson_full_size_sampled_rows():
    # the benchmark's workload and launch plan (static choice), all rows run,
    # sampled rows compared with the oracle; every row's output mean is its r
    w = wl.PEARSON_F32_4096x65536
    inp = w.generate()
    p = make_plan(w)
    y, r = run(w, inp, p)
    rows = np.array([0, 1, 2, 1000, 2047, 3001, 4094, 4095])
    check_pearson(w, (y, r), inp, rows=rows)
    means = y.astype(np.float64).mean(axis=1)
    assert np.abs(means - r).max() < 1e-4
    assert np.all(np.abs(r - 1.2 / np.sqrt(2.08)) < 0.02)


@pytest.mark.parametrize("variant,P", [(C.CLUSTER, 1), (C.CLUSTER, 4), (C.TWO_PASS, 1)])
def test_pearson_misaligned_operands(variant, P):
    # x, u and y one element past a 16-byte boundary: the element path
    w = _w("f32", 3, 8192, 78)
    inp = w.generate()
    dev = torch.cuda.current_device()

    def shifted(a):
        t = torch.from_numpy(np.concatenate([np.zeros(1, np.float32), a.reshape(-1)])).cuda()
        return t[1:]
    dx, du = shifted(inp["x"]), shifted(inp["u"])
    dy = torch.empty(dx.numel() + 1, device="cuda")[1:]
    r = torch.empty(w.rows, device="cuda")
    p = C.credit_plan_for(C.PEARSON, w.rows, w.cols, C.F32, dev, variant, P)
    ws = torch.empty(max(1, int(p.workspace_bytes)), dtype=torch.uint8, device="cuda")
    assert C.credit_pearson(dx.data_ptr(), du.data_ptr(), dy.data_ptr(), r.data_ptr(), w.rows,
                            w.cols, C.F32, w.eps, p, ws.data_ptr(), int(p.workspace_bytes)) == C.OK
    torch.cuda.synchronize()
    check_pearson(w, (dy.cpu().numpy().reshape(w.rows, w.cols), r.cpu().numpy()), inp)
