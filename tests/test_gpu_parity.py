"""GPU parity: the CUDA path (called through the C ABI) against the fp64
oracle on the same seeded inputs, element by element.

Covers the five workloads' shapes at reduced row counts for every legal
cluster size and the two-pass baseline, the full-size workloads on sampled
rows in the launch configuration the benchmark uses, cluster-size invariance,
and the edge cases: ragged widths (element-wise staging path), slices that are
empty, a single row, in-place calls, misaligned pointers, absent parameters,
bf16 parameters and constant rows.
"""
import itertools

import numpy as np
import pytest
import torch

from dsmem_thread_block_gb300 import _credit as C
from dsmem_thread_block_gb300 import workloads as wl

from gpu_helpers import (DT, OPS, bounds, call, check, check_quant, make_plan, oracle_rows, run,
                         to_device, to_host)

pytestmark = pytest.mark.gpu

TWO = ("two_pass", 0)


def _try_plan(w, variant, P, rows=None):
    try:
        return make_plan(w, variant, P, rows=rows)
    except C.CreditError as e:
        assert e.status == C.ERR_NO_LEGAL_PLAN
        return None


def _plans(w, cluster_sizes, rows=None):
    """One-row-per-cluster plans for `cluster_sizes` (must be legal), the
    persistent plans of those sizes that are legal, and the two-pass plan."""
    out = []
    for P in cluster_sizes:
        out.append(make_plan(w, C.CLUSTER, P, rows=rows))
        p = _try_plan(w, C.CLUSTER_PERSISTENT, P, rows=rows)
        if p is not None:
            out.append(p)
    out.append(make_plan(w, C.TWO_PASS, rows=rows))
    return out


# ----------------------------------------------------------- workload shapes
def test_softmax_f32_64x4096_all_cluster_sizes():
    w = wl.SOFTMAX_F32_64x4096
    inp = w.generate()
    for P in (1, 2, 3, 4, 8, 16):
        got = run(w, inp, make_plan(w, C.CLUSTER, P))
        check(w, got, inp)
        got = run(w, inp, make_plan(w, C.CLUSTER_PERSISTENT, P))
        check(w, got, inp)
    got = run(w, inp, make_plan(w, C.TWO_PASS))
    check(w, got, inp)


@pytest.mark.parametrize("w,sizes", [
    (wl.LAYERNORM_BF16_1024x262144.with_rows(3), (4, 5, 8, 16)),
    (wl.SOFTMAX_F32_512x131072_SPIKES.with_rows(3), (4, 6, 8, 16)),
    (wl.RMSNORM_BF16_2048x786432.with_rows(2), (8, 12, 16)),
])
def test_wide_rows_every_legal_cluster_size(w, sizes):
    inp = w.generate()
    outs = []
    for p in _plans(w, sizes):
        got = run(w, inp, p)
        check(w, got, inp)
        outs.append(oracle_widen(got))
    # cluster-size invariance: variants agree pairwise within twice the
    # per-element bound against the oracle
    _, bound, _ = bounds(w, inp)
    ref = outs[0]
    for o in outs[1:]:
        assert (np.abs(o - ref) <= 2 * bound).all()


def oracle_widen(a):
    import oracle
    return oracle.widen(a)


@pytest.mark.parametrize("cols", [1 << k for k in range(10, 21, 2)])
def test_bf16_softmax_sweep_shapes(cols):
    w = wl.sweep_point(cols).with_rows(2)
    inp = w.generate()
    # every power-of-two cluster size that is legal at this width, and two-pass
    for P in (1, 2, 4, 8, 16):
        for variant in (C.CLUSTER, C.CLUSTER_PERSISTENT):
            p = _try_plan(w, variant, P)
            if p is not None:
                check(w, run(w, inp, p), inp)
    check(w, run(w, inp, make_plan(w, C.TWO_PASS)), inp)


# ---------------------------------------------------------------- edge cases
def _custom(op, dtype, rows, cols, seed, **kw):
    return wl.Workload(f"{op}_{dtype}_{rows}x{cols}", op, dtype, rows, cols, seed, **kw)


EDGE = [
    _custom(wl.SOFTMAX, "f32", 3, 4099, 5, x_std=3.0),            # ragged: element path
    _custom(wl.SOFTMAX, "bf16", 2, 1001, 6),                       # ragged bf16
    _custom(wl.SOFTMAX, "bf16", 2, 1000, 7),                       # 16B rows, ragged slices
    _custom(wl.SOFTMAX, "f32", 2, 8, 8),                           # empty CTAs, bulk path
    _custom(wl.SOFTMAX, "f32", 2, 5, 9),                           # cols < P*vec, element path
    _custom(wl.SOFTMAX, "f32", 1, 1, 10),                          # one element
    _custom(wl.LAYERNORM, "f32", 2, 3001, 11, x_mean=1.0, x_std=2.0, eps=1e-5, param_dtype="f32"),
    _custom(wl.LAYERNORM, "bf16", 2, 4096, 12, x_mean=0.5, x_std=2.0, eps=1e-5, param_dtype="bf16"),
    _custom(wl.LAYERNORM, "f32", 2, 4096, 13, x_mean=-3.0, x_std=0.5, eps=1e-5),  # no params
    _custom(wl.RMSNORM, "f32", 2, 5003, 14, eps=1e-6, param_dtype="f32"),
    _custom(wl.RMSNORM, "bf16", 2, 777, 15, eps=1e-6),                            # no weight
    _custom(wl.RMSNORM, "bf16", 1, 65536, 16, eps=1e-6, param_dtype="f32"),
]


@pytest.mark.parametrize("w", EDGE, ids=[w.name for w in EDGE])
def test_edge_shapes(w):
    inp = w.generate()
    for P in (1, 2, 3, 4, 7, 16):
        for variant in (C.CLUSTER, C.CLUSTER_PERSISTENT):
            p = _try_plan(w, variant, P)
            if p is not None:  # persistent plans of ragged rows run the element path
                check(w, run(w, inp, p), inp)
    check(w, run(w, inp, make_plan(w, C.TWO_PASS)), inp)
    check(w, run(w, inp, None), inp)  # automatic plan


@pytest.mark.parametrize("variant,P", [(C.CLUSTER, 1), (C.CLUSTER, 4), (C.TWO_PASS, 1),
                                       (C.CLUSTER_PERSISTENT, 1), (C.CLUSTER_PERSISTENT, 4)])
def test_in_place(variant, P):
    for w in (_custom(wl.SOFTMAX, "f32", 4, 16384, 20, x_std=2.0),
              _custom(wl.LAYERNORM, "bf16", 4, 16384, 21, eps=1e-5, param_dtype="f32"),
              _custom(wl.RMSNORM, "f32", 4, 16387, 22, eps=1e-6, param_dtype="bf16")):
        inp = w.generate()
        got = run(w, inp, make_plan(w, variant, P), in_place=True)
        check(w, got, inp)


@pytest.mark.parametrize("variant,P", [(C.CLUSTER, 1), (C.CLUSTER, 4), (C.TWO_PASS, 1),
                                       (C.CLUSTER_PERSISTENT, 4)])
def test_misaligned_pointers_take_element_path(variant, P):
    w = _custom(wl.LAYERNORM, "bf16", 3, 8192, 23, eps=1e-5, param_dtype="f32")
    inp = w.generate()
    # place x and y one element past a 16-byte boundary
    xs = to_device(np.concatenate([np.zeros(1, np.uint16), inp["x"].reshape(-1)]))
    dx = xs[1:]
    dy_full = torch.empty(dx.numel() + 1, dtype=dx.dtype, device=dx.device)
    dy = dy_full[1:]
    params = {k: to_device(v) for k, v in inp.items() if k != "x"}
    assert call(w, dx, dy, params, make_plan(w, variant, P)) == C.OK
    torch.cuda.synchronize()
    got = to_host(dy).reshape(w.rows, w.cols)
    check(w, got, inp)


def test_constant_rows():
    # LayerNorm of a constant row is exactly beta (sums of -1.5 are exact)
    w = _custom(wl.LAYERNORM, "f32", 2, 65536, 24, eps=1e-5, param_dtype="f32")
    inp = w.generate()
    inp["x"] = np.full((2, 65536), -1.5, np.float32)
    for p in _plans(w, (2, 4)):  # a 256 KiB fp32 row needs P >= 2
        got = run(w, inp, p)
        assert np.array_equal(got, np.broadcast_to(inp["beta"], got.shape))
    # softmax of a constant row is uniform
    w = _custom(wl.SOFTMAX, "f32", 2, 65536, 25)
    inp = {"x": np.full((2, 65536), 0.25, np.float32)}
    for p in _plans(w, (2, 4)):
        got = run(w, inp, p)
        np.testing.assert_allclose(got, 1.0 / 65536, rtol=1e-6)


def test_auto_plan_is_legal_and_clustered_for_wide_rows():
    for w in (wl.LAYERNORM_BF16_1024x262144, wl.SOFTMAX_F32_512x131072_SPIKES,
              wl.RMSNORM_BF16_2048x786432):
        p = make_plan(w)
        assert p.variant in (C.CLUSTER, C.CLUSTER_PERSISTENT)
        assert p.slice_elems * p.cluster_size >= w.cols
        assert p.smem_bytes <= 232448


# ------------------------------------------------- full size, sampled rows
FULL = [wl.SOFTMAX_F32_64x4096, wl.LAYERNORM_BF16_1024x262144,
        wl.SOFTMAX_F32_512x131072_SPIKES, wl.RMSNORM_BF16_2048x786432]


@pytest.mark.parametrize("w", FULL, ids=[w.name for w in FULL])
def test_full_size_sampled_rows(w):
    inp = w.generate()
    # the launch configuration the benchmark times: the cost model's choice
    # after timing every legal candidate (bench.py plans the same way)
    dev = torch.cuda.current_device()
    pdt = DT[w.param_dtype] if w.param_dtype else -1
    p, _ = C.tuned_plan(OPS[w.op], w.rows, w.cols, DT[w.dtype], pdt, dev)
    dx = to_device(inp["x"])
    dy = torch.empty_like(dx)
    params = {k: to_device(v) for k, v in inp.items() if k != "x"}
    assert call(w, dx, dy, params, p) == C.OK
    torch.cuda.synchronize()
    assert C.credit_get_device_error(torch.cuda.current_device()) == C.OK
    rng = np.random.default_rng(99)
    rows = sorted({0, w.rows - 1, *rng.integers(0, w.rows, 6).tolist()})
    got = to_host(dy[rows])
    sub = dict(inp)
    sub["x"] = inp["x"][rows]
    res = check(w, got, sub)
    print(f"[parity] {w.name} ({C.variant_name(p)}): max_rel {res['max_rel']:.3e}, "
          f"{res['only_cancel']} of {res['n']} through the cancellation term")
    if w.dtype == "bf16":
        assert res["only_cancel_frac"] < 1e-4
    # every row, at any size: finite, and softmax rows sum to one
    yf = dy.float()
    assert bool(torch.isfinite(yf).all())
    if w.op == wl.SOFTMAX:
        tol = 1e-4 if w.dtype == "f32" else 2e-2
        sums = yf.double().sum(dim=1)
        assert float((sums - 1).abs().max()) <= tol


def test_illegal_cluster_sizes_are_rejected():
    # a 256 KiB fp32 row cannot be staged by one CTA (227 KiB limit)
    w = _custom(wl.SOFTMAX, "f32", 2, 65536, 26)
    with pytest.raises(C.CreditError) as e:
        make_plan(w, C.CLUSTER, 1)
    assert e.value.status == C.ERR_NO_LEGAL_PLAN
    with pytest.raises(C.CreditError) as e:
        make_plan(w, C.CLUSTER, 17)
    assert e.value.status == C.ERR_NO_LEGAL_PLAN
    # a forced plan passed to a call is re-derived and checked the same way
    p = make_plan(w, C.CLUSTER, 2)
    p.cluster_size = 1
    inp = w.generate()
    dx = to_device(inp["x"])
    assert call(w, dx, torch.empty_like(dx), {}, p) == C.ERR_NO_LEGAL_PLAN


@pytest.mark.parametrize("rows", [1, 7, 300])
def test_persistent_row_counts(rows):
    # fewer rows than resident clusters, a few rows per cluster, many rows
    # per cluster (slot, ring and mbarrier-phase reuse over many rows); one
    # and two CTAs per SM; both exchanges
    w = _custom(wl.LAYERNORM, "bf16", rows, 32768, 30, x_mean=0.5, x_std=2.0, eps=1e-5,
                param_dtype="f32")
    inp = w.generate()
    ran = 0
    for P, cps, xc in itertools.product((1, 2, 4, 8), (1, 2),
                                        (C.EXCHANGE_BARRIER, C.EXCHANGE_ASYNC)):
        p = _try_plan(w, C.CLUSTER_PERSISTENT, P)
        if p is None:
            continue
        p.exchange = xc
        if True:
            p.ctas_per_sm = cps
            dx = to_device(inp["x"])
            dy = torch.empty_like(dx)
            params = {k: to_device(v) for k, v in inp.items() if k != "x"}
            st = call(w, dx, dy, params, p)
            if st == C.ERR_NO_LEGAL_PLAN:
                continue
            assert st == C.OK
            torch.cuda.synchronize()
            check(w, to_host(dy), inp)
            ran += 1
    assert ran >= 8


def test_persistent_async_exchange_all_ops():
    # the st.async exchange in the persistent ring for every operator it
    # runs, at cluster sizes whose slices leave a ragged last CTA
    dev = torch.cuda.current_device()
    cases = [
        _custom(wl.SOFTMAX, "f32", 37, 65536, 90, x_std=4.0, spike_frac=0.01),
        _custom(wl.SOFTMAX, "bf16", 41, 131072, 91),
        _custom(wl.RMSNORM, "bf16", 33, 196608, 92, eps=1e-6, param_dtype="bf16"),
        _custom(wl.LAYERNORM, "f32", 29, 49152, 93, x_mean=-1.0, x_std=3.0, eps=1e-5,
                param_dtype="f32"),
    ]
    ran = 0
    for w in cases:
        inp = w.generate()
        for P in (2, 3, 5, 9):
            try:
                p = C.credit_plan_with(gh_ops(w), w.rows, w.cols, gh_dt(w), dev,
                                       C.CLUSTER_PERSISTENT, P, exchange=C.EXCHANGE_ASYNC)
            except C.CreditError as e:
                assert e.status == C.ERR_NO_LEGAL_PLAN
                continue
            assert p.exchange == C.EXCHANGE_ASYNC
            check(w, run(w, inp, p), inp)
            ran += 1
    assert ran >= 8
    assert C.credit_get_device_error(dev) == C.OK


@pytest.mark.parametrize("R", [2, 4])
def test_rows_per_cluster(R):
    # several rows per cluster share one exchange and each parameter load;
    # row counts that are not a multiple of R leave a partial last cluster
    cases = [
        _custom(wl.LAYERNORM, "bf16", 7, 65536, 40, x_mean=0.5, x_std=2.0, eps=1e-5,
                param_dtype="f32"),
        _custom(wl.LAYERNORM, "f32", 5, 12288, 41, x_mean=-1.0, x_std=3.0, eps=1e-5,
                param_dtype="bf16"),
        _custom(wl.RMSNORM, "bf16", 6, 98304, 42, eps=1e-6, param_dtype="bf16"),
        _custom(wl.SOFTMAX, "f32", 9, 32768, 43, x_std=4.0, spike_frac=0.01),
        _custom(wl.SOFTMAX, "bf16", 3, 4096, 44),
    ]
    dev = torch.cuda.current_device()
    for w in cases:
        inp = w.generate()
        for P in (1, 2, 4, 8):
            try:
                p = C.credit_plan_with(gh_ops(w), w.rows, w.cols, gh_dt(w), dev, C.CLUSTER, P,
                                       rows_per_cluster=R)
            except C.CreditError as e:
                assert e.status == C.ERR_NO_LEGAL_PLAN
                continue
            assert p.rows_per_cluster == R
            check(w, run(w, inp, p), inp)
            check(w, run(w, inp, p, in_place=True), inp)


@pytest.mark.parametrize("exchange", ["barrier", "async"])
@pytest.mark.parametrize("R", [1, 2, 4])
def test_exchange_modes(R, exchange):
    # st.async deposits counted on each receiver's mbarrier, or remote stores
    # plus the release/acquire cluster barrier: same statistics, same outputs
    xc = C.EXCHANGE_ASYNC if exchange == "async" else C.EXCHANGE_BARRIER
    cases = [
        _custom(wl.LAYERNORM, "bf16", 9, 131072, 50, x_mean=0.5, x_std=2.0, eps=1e-5,
                param_dtype="f32"),
        _custom(wl.RMSNORM, "f32", 5, 65536, 51, eps=1e-6, param_dtype="f32"),
        _custom(wl.SOFTMAX, "f32", 7, 65536, 52, x_std=4.0, spike_frac=0.01),
        _custom(wl.SOFTMAX, "bf16", 6, 262144, 53),
        _custom(wl.WEIGHTED_STD, "f32", 5, 32768, 54, x_mean=0.5, x_std=2.0, eps=1e-5,
                param_dtype="f32", p_uniform=True),
    ]
    dev = torch.cuda.current_device()
    ran = 0
    for w in cases:
        inp = w.generate()
        for P in (2, 3, 4, 8, 16):
            try:
                p = C.credit_plan_with(gh_ops(w), w.rows, w.cols, gh_dt(w), dev, C.CLUSTER, P,
                                       rows_per_cluster=R, exchange=xc)
            except C.CreditError as e:
                assert e.status == C.ERR_NO_LEGAL_PLAN
                continue
            assert p.exchange == xc and p.cluster_size == P
            check(w, run(w, inp, p), inp)
            ran += 1
    assert ran >= 10
    assert C.credit_get_device_error(dev) == C.OK


def test_rmsnorm_bf16_weights_pipelined_output():
    # bf16 data with bf16 weights takes the software-pipelined output pass:
    # slices whose granule count leaves partial warp tiles and odd tile
    # counts per warp
    dev = torch.cuda.current_device()
    for cols in (98312, 24584, 8200):
        w = _custom(wl.RMSNORM, "bf16", 3, cols, 58, eps=1e-6, param_dtype="bf16")
        inp = w.generate()
        for P in (1, 2, 3, 5, 7, 16):
            try:
                p = C.credit_plan_with(gh_ops(w), w.rows, w.cols, gh_dt(w), dev, C.CLUSTER, P)
            except C.CreditError as e:
                assert e.status == C.ERR_NO_LEGAL_PLAN
                continue
            check(w, run(w, inp, p), inp)
    assert C.credit_get_device_error(dev) == C.OK


def test_rmsnorm_bf16_weights_large_slices_deep_kernel():
    # slices too large for three CTAs per SM take the instantiation with the
    # deeper weight prefetch: whole, ragged and partial warp tiles
    dev = torch.cuda.current_device()
    for cols, sizes in ((786432, (8, 12, 16)), (600000, (4, 7, 9)), (300008, (3, 4))):
        w = _custom(wl.RMSNORM, "bf16", 3, cols, 59, eps=1e-6, param_dtype="bf16")
        inp = w.generate()
        ran = 0
        for P in sizes:
            try:
                p = C.credit_plan_with(gh_ops(w), w.rows, w.cols, gh_dt(w), dev, C.CLUSTER, P)
            except C.CreditError as e:
                assert e.status == C.ERR_NO_LEGAL_PLAN
                continue
            assert p.smem_bytes > 64 * 1024  # the deep instantiation's range
            check(w, run(w, inp, p), inp)
            ran += 1
        assert ran >= 1
    assert C.credit_get_device_error(dev) == C.OK


def test_planned_exchange():
    dev = torch.cuda.current_device()
    w = _custom(wl.SOFTMAX, "f32", 4, 65536, 57)
    assert make_plan(w, C.CLUSTER, 4).exchange == C.EXCHANGE_ASYNC
    assert make_plan(w, C.TWO_PASS, 1).exchange == C.EXCHANGE_DEFAULT
    p = _try_plan(w, C.CLUSTER_PERSISTENT, 4)
    if p is not None:
        assert p.exchange == C.EXCHANGE_ASYNC
    assert C.credit_plan_with(C.SOFTMAX, 4, 65536, C.F32, dev, C.CLUSTER, 4,
                              exchange=C.EXCHANGE_BARRIER).exchange == C.EXCHANGE_BARRIER


def test_async_exchange_quantize_and_ragged():
    # int8 codes stay bit-exact; a ragged, misaligned row takes the element
    # path with the same exchange
    dev = torch.cuda.current_device()
    q = _custom(wl.QUANTIZE, "f32", 6, 65536, 55, x_std=3.0)
    inp = q.generate()
    for P in (2, 4, 16):
        p = C.credit_plan_with(gh_ops(q), q.rows, q.cols, gh_dt(q), dev, C.CLUSTER, P,
                               exchange=C.EXCHANGE_ASYNC)
        check_quant(run(q, inp, p), inp)
    w = _custom(wl.LAYERNORM, "bf16", 5, 40001, 56, x_mean=-0.25, x_std=1.5, eps=1e-5,
                param_dtype="bf16")
    inp = w.generate()
    for P in (3, 5):
        p = C.credit_plan_with(gh_ops(w), w.rows, w.cols, gh_dt(w), dev, C.CLUSTER, P,
                               exchange=C.EXCHANGE_ASYNC)
        check(w, run(w, inp, p), inp)
    assert C.credit_get_device_error(dev) == C.OK


def gh_ops(w):
    from gpu_helpers import OPS
    return OPS[w.op]


def gh_dt(w):
    from gpu_helpers import DT
    return DT[w.dtype]


def test_rows_wider_than_any_cluster_fall_back_to_two_pass():
    # 64 MB fp32 rows: no cluster of up to 16 CTAs can stage one, so the
    # automatic plan is the two-pass kernel pair, which still matches
    w = _custom(wl.SOFTMAX, "f32", 2, 1 << 24, 96, x_std=3.0)
    dev = torch.cuda.current_device()
    with pytest.raises(C.CreditError) as e:
        C.credit_plan_for(C.SOFTMAX, w.rows, w.cols, C.F32, dev, C.CLUSTER, 16)
    assert e.value.status == C.ERR_NO_LEGAL_PLAN
    p = make_plan(w)
    assert p.variant == C.TWO_PASS
    inp = w.generate()
    check(w, run(w, inp, p), inp)
