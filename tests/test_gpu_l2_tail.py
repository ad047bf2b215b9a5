"""L2-tail plans of the one-row-per-cluster kernel against the oracle.

An L2-tail plan stages only the first `staged_elems` elements of each CTA's
slice in shared memory; the rest of the slice is read from HBM once (kept
in L2 with an evict-last hint) for the statistics and read again, from L2,
by the output pass -- through registers, or copied by each warp into a ring
of its freed staged tiles (16-byte granules), including warps with too few
staged tiles for a ring and tails several rings long.  The results must match the oracle exactly as a fully
staged plan's do: the workload shapes at reduced row counts for several
cluster sizes and staged lengths (including cluster sizes whose whole slice
does not fit shared memory), unequal last slices, CTAs whose slice ends
before the tail starts, a staged part of a single vector, in-place calls,
absent parameters, fp32 data, the checked build, seeded random shapes, and
two and four rows per cluster, and the argument rules (operators without an
L2-tail form, misaligned pointers falling back to whole-slice staging)."""
import numpy as np
import pytest
import torch

from dsmem_thread_block_gb300 import _credit as C
from dsmem_thread_block_gb300 import workloads as wl

from gpu_helpers import DT, OPS, call, check, run, to_device, to_host

pytestmark = pytest.mark.gpu


def _plan(w, P, staged, rows_per_cluster=0):
    dev = torch.cuda.current_device()
    return C.credit_plan_with(OPS[w.op], w.rows, w.cols, DT[w.dtype], dev, C.CLUSTER, P,
                              rows_per_cluster=rows_per_cluster, staged_elems=staged)


WIDE = [
    (wl.LAYERNORM_BF16_1024x262144.with_rows(3), [(8, 16384), (8, 24576), (16, 12288), (4, 36864)]),
    (wl.RMSNORM_BF16_2048x786432.with_rows(2), [(10, 36864), (12, 28672), (16, 24576), (8, 53248),
                                                 (5, 53248)]),
    (wl.sweep_point(1 << 20).with_rows(2), [(12, 36864), (16, 28672), (10, 53248), (8, 37376),
                                             (8, 18688)]),
    # 28,672 staged elements: warps 0-3 have four full staged tiles for a
    # ring of tail tiles, warps 4-7 read their tail tiles from global memory
    (wl.sweep_point(1 << 19).with_rows(3), [(12, 36864), (8, 36864), (8, 28672), (8, 18688),
                                            (8, 4096)]),
]


@pytest.mark.parametrize("w,cases", WIDE, ids=[c[0].name for c in WIDE])
def test_wide_rows_with_an_l2_tail(w, cases):
    inp = w.generate()
    for P, staged in cases:
        p = _plan(w, P, staged)
        assert p.staged_elems == staged and p.slice_elems > staged, (P, staged, p)
        assert p.smem_bytes == staged * (4 if w.dtype == "f32" else 2)
        check(w, run(w, inp, p), inp)


def _custom(op, dtype, rows, cols, seed, **kw):
    return wl.Workload(f"{op}_{dtype}_{rows}x{cols}", op, dtype, rows, cols, seed, **kw)


EDGES = [
    # unequal last slice: P = 7 over 100008 columns (slices of 14288, the
    # last 14280), a tail in every CTA
    (_custom(wl.LAYERNORM, "bf16", 3, 100008, 60, x_mean=0.5, x_std=2.0, eps=1e-5,
             param_dtype="f32"), 7, 10000),
    # the last CTA's slice (8184) ends before the tail would start (8192)
    (_custom(wl.RMSNORM, "bf16", 3, 24584, 61, eps=1e-6, param_dtype="bf16"), 3, 8192),
    # a staged part of one vector: nearly everything through L2
    (_custom(wl.SOFTMAX, "bf16", 2, 65536, 62, x_std=3.0, spike_frac=0.01), 4, 8),
    # fp32 data, fp32 and bf16 parameters, absent parameters
    (_custom(wl.LAYERNORM, "f32", 3, 98304, 63, x_mean=-1.0, x_std=1.5, eps=1e-5,
             param_dtype="bf16"), 4, 12000),
    (_custom(wl.RMSNORM, "f32", 3, 131072, 64, eps=1e-6, param_dtype="f32"), 4, 20000),
    (_custom(wl.LAYERNORM, "bf16", 2, 262144, 65, x_mean=3.0, x_std=0.5, eps=1e-5), 8, 20480),
    (_custom(wl.RMSNORM, "bf16", 2, 262144, 66, eps=1e-6), 8, 16384),
]


@pytest.mark.parametrize("w,P,staged", EDGES, ids=[e[0].name for e in EDGES])
def test_tail_edges(w, P, staged):
    inp = w.generate()
    p = _plan(w, P, staged)
    check(w, run(w, inp, p), inp)
    check(w, run(w, inp, p, in_place=True), inp)  # y == x: each element read before written


def test_tail_plan_argument_rules():
    dev = torch.cuda.current_device()
    sm = _custom(wl.SOFTMAX, "f32", 2, 65536, 70)
    with pytest.raises(C.CreditError) as e:  # fp32 softmax stashes in place: no tail form
        _plan(sm, 4, 8192)
    assert e.value.status == C.ERR_INVALID_ARG
    q = _custom(wl.QUANTIZE, "bf16", 2, 65536, 71)
    with pytest.raises(C.CreditError) as e:
        _plan(q, 4, 8192)
    assert e.value.status == C.ERR_INVALID_ARG
    ln = _custom(wl.LAYERNORM, "bf16", 4, 65536, 72, eps=1e-5, param_dtype="f32")
    pe = _custom(wl.PEARSON, "f32", 2, 65536, 74)
    with pytest.raises(C.CreditError) as e:  # two staged operands: no tail form
        _plan(pe, 4, 8192)
    assert e.value.status == C.ERR_INVALID_ARG
    with pytest.raises(C.CreditError) as e:
        C.credit_plan_with(OPS[ln.op], ln.rows, ln.cols, DT[ln.dtype], dev, C.CLUSTER, 4,
                           staged_elems=-8)
    assert e.value.status == C.ERR_INVALID_ARG
    # a staged length at or beyond the slice is a whole-slice plan
    p = _plan(ln, 4, 1 << 20)
    assert p.staged_elems == p.slice_elems


MULTI = [
    (wl.LAYERNORM_BF16_1024x262144.with_rows(5), [(8, 2, 18432), (8, 4, 8192), (16, 2, 12288)]),
    (wl.RMSNORM_BF16_2048x786432.with_rows(3), [(12, 2, 18432), (16, 2, 16384)]),
    (wl.sweep_point(1 << 19).with_rows(7), [(8, 2, 18432), (12, 4, 8192)]),
    (_custom(wl.LAYERNORM, "f32", 5, 100004, 75, x_mean=-0.5, x_std=1.5, eps=1e-5,
             param_dtype="bf16"), [(7, 2, 6000), (3, 4, 4000)]),
]


@pytest.mark.parametrize("w,cases", MULTI, ids=[c[0].name for c in MULTI])
def test_tails_with_several_rows_per_cluster(w, cases):
    # R rows per cluster share one parameter load; each row's slice has its
    # staged part at its own pitch and its own L2 tail (row counts that are
    # not a multiple of R leave the last cluster short)
    inp = w.generate()
    for P, R, staged in cases:
        p = _plan(w, P, staged, rows_per_cluster=R)
        assert p.rows_per_cluster == R and p.staged_elems == staged < p.slice_elems
        check(w, run(w, inp, p), inp)
        check(w, run(w, inp, p, in_place=True), inp)


def test_misaligned_pointers_fall_back_to_whole_slice_staging():
    # a tail plan handed misaligned pointers takes the element path, which
    # stages the whole slice (legal here); where the whole slice cannot be
    # staged the call reports that no legal plan exists
    w = _custom(wl.LAYERNORM, "bf16", 2, 65536, 73, x_mean=0.5, x_std=2.0, eps=1e-5,
                param_dtype="f32")
    inp = w.generate()
    xs = to_device(np.concatenate([np.zeros(1, np.uint16), inp["x"].reshape(-1)]))
    dx = xs[1:]
    dy = torch.empty(dx.numel() + 1, dtype=dx.dtype, device=dx.device)[1:]
    params = {k: to_device(v) for k, v in inp.items() if k != "x"}
    assert call(w, dx, dy, params, _plan(w, 4, 8192)) == C.OK
    torch.cuda.synchronize()
    check(w, to_host(dy).reshape(w.rows, w.cols), inp)
    big = wl.RMSNORM_BF16_2048x786432.with_rows(1)
    binp = big.generate()
    bx = to_device(np.concatenate([np.zeros(1, np.uint16), binp["x"].reshape(-1)]))[1:]
    by = torch.empty(bx.numel() + 1, dtype=bx.dtype, device=bx.device)[1:]
    bp = {k: to_device(v) for k, v in binp.items() if k != "x"}
    assert call(big, bx, by, bp, _plan(big, 5, 53248)) == C.ERR_NO_LEGAL_PLAN


def test_tail_plans_in_the_checked_build():
    cases = [(wl.RMSNORM_BF16_2048x786432.with_rows(2), 10, 36864),
             (wl.LAYERNORM_BF16_1024x262144.with_rows(3), 8, 16384),
             (wl.sweep_point(1 << 20).with_rows(2), 12, 36864)]
    with C.use_checked_build():
        for w, P, staged in cases:
            inp = w.generate()
            check(w, run(w, inp, _plan(w, P, staged)), inp)
        assert C.credit_get_device_error(torch.cuda.current_device()) == C.OK


def _random_cases(n=40, seed=20261203):
    rng = np.random.default_rng(seed)
    out = []
    for k in range(n):
        op = str(rng.choice([wl.SOFTMAX, wl.LAYERNORM, wl.RMSNORM]))
        dtype = "bf16" if op == wl.SOFTMAX else str(rng.choice(["f32", "bf16"]))
        vec = 4 if dtype == "f32" else 8
        cols = int(vec * rng.integers(512, 40000))
        rows = int(rng.integers(1, 9))
        kw = {"x_mean": float(rng.normal(0, 1.5)), "x_std": float(rng.uniform(0.2, 3.0)),
              "eps": 1e-5}
        if op != wl.SOFTMAX and rng.random() < 0.8:
            kw["param_dtype"] = str(rng.choice(["f32", "bf16"]))
        w = wl.Workload(f"tail{k}_{op}_{dtype}_{rows}x{cols}", op, dtype, rows, cols,
                        seed=int(rng.integers(1, 1 << 30)), **kw)
        P = int(rng.integers(1, 17))
        slice_ = -(-(-(-cols // P)) // vec) * vec
        staged = int(vec * rng.integers(1, max(2, slice_ // vec)))
        out.append((w, P, staged))
    return out


RANDOM = _random_cases()


@pytest.mark.parametrize("w,P,staged", RANDOM, ids=[c[0].name for c in RANDOM])
def test_random_tail_plans(w, P, staged):
    inp = w.generate()
    # the drawn cluster size, or the next one up that can be resident
    for q in range(P, 17):
        try:
            p = _plan(w, q, staged)
            break
        except C.CreditError as e:
            assert e.status == C.ERR_NO_LEGAL_PLAN, (w.name, q, e)
    else:
        raise AssertionError(f"{w.name}: no legal plan from P = {P}")
    check(w, run(w, inp, p), inp)



LARGE = [
    # footprints that leave room for at most two CTAs per SM: whole slices and
    # L2 tails of LayerNorm (bf16 data, fp32 parameters) with one and two rows
    # per cluster, and RMSNorm's bf16 instantiation bounded to two CTAs per SM
    (wl.LAYERNORM_BF16_1024x262144.with_rows(5), [(12, 2, 0), (10, 2, 0), (8, 2, 24576),
                                                   (4, 1, 45056)]),
    (_custom(wl.LAYERNORM, "bf16", 5, 200008, 76, x_mean=-2.0, x_std=0.7, eps=1e-5,
             param_dtype="f32"), [(9, 2, 0), (5, 2, 20000), (3, 1, 40000)]),
    (wl.RMSNORM_BF16_2048x786432.with_rows(3), [(16, 1, 0), (8, 1, 45056)]),
]


@pytest.mark.parametrize("w,cases", LARGE, ids=[c[0].name for c in LARGE])
def test_footprints_of_two_ctas_per_sm(w, cases):
    inp = w.generate()
    smem_per_sm = torch.cuda.get_device_properties(0).shared_memory_per_multiprocessor
    for P, R, staged in cases:
        p = _plan(w, P, staged, rows_per_cluster=R)
        assert p.rows_per_cluster == R
        assert p.smem_bytes > smem_per_sm // 3, (P, R, staged, p.smem_bytes)
        check(w, run(w, inp, p), inp)
        check(w, run(w, inp, p, in_place=True), inp)


FOUR = [
    # bf16 softmax and LayerNorm (bf16 data, fp32 parameters) L2-tail plans
    # whose footprint leaves room for four CTAs per SM take the instantiation
    # bounded to 64 registers
    (wl.sweep_point(1 << 19).with_rows(5), [8, 4, 16, 5]),
    (wl.sweep_point(1 << 20).with_rows(3), [16, 8, 12]),
    (_custom(wl.SOFTMAX, "bf16", 4, 400008, 77, x_std=2.5, spike_frac=0.02), [7, 12]),
    (wl.LAYERNORM_BF16_1024x262144.with_rows(5), [4, 8, 6]),
    (_custom(wl.LAYERNORM, "bf16", 3, 300008, 78, x_mean=-1.0, x_std=3.0, eps=1e-5,
             param_dtype="f32"), [3, 5]),
    (_custom(wl.LAYERNORM, "bf16", 3, 262144, 79, x_mean=2.0, x_std=0.5, eps=1e-5), [4]),
]


@pytest.mark.parametrize("w,sizes", FOUR, ids=[c[0].name for c in FOUR])
def test_four_ctas_per_sm(w, sizes):
    inp = w.generate()
    dev = torch.cuda.current_device()
    smem_per_sm = torch.cuda.get_device_properties(0).shared_memory_per_multiprocessor
    for P in sizes:
        p = C.credit_plan_tail(OPS[w.op], w.rows, w.cols, DT[w.dtype], dev, P, 4)
        assert p.staged_elems < p.slice_elems and 4 * p.smem_bytes < smem_per_sm, (P, p)
        check(w, run(w, inp, p), inp)
        check(w, run(w, inp, p, in_place=True), inp)
    with C.use_checked_build():
        p = C.credit_plan_tail(OPS[w.op], w.rows, w.cols, DT[w.dtype], dev, sizes[0], 4)
        check(w, run(w, inp, p), inp)
        assert C.credit_get_device_error(dev) == C.OK


SMALL = [
    # 128-thread CTAs staging the length for ten CTAs per SM (the tuner's
    # small-CTA form for the operators with the 64-register instantiation)
    (wl.LAYERNORM_BF16_1024x262144.with_rows(5), [8, 4, 12]),
    (wl.sweep_point(1 << 19).with_rows(3), [8, 16]),
    (_custom(wl.LAYERNORM, "bf16", 3, 200008, 80, x_mean=0.3, x_std=1.7, eps=1e-5,
             param_dtype="f32"), [5, 7]),
]


@pytest.mark.parametrize("w,sizes", SMALL, ids=[c[0].name for c in SMALL])
def test_small_ctas(w, sizes):
    inp = w.generate()
    dev = torch.cuda.current_device()
    for P in sizes:
        t10 = C.credit_plan_tail(OPS[w.op], w.rows, w.cols, DT[w.dtype], dev, P, 10)
        p = C.credit_plan_with(OPS[w.op], w.rows, w.cols, DT[w.dtype], dev, C.CLUSTER, P,
                               threads=128, staged_elems=int(t10.staged_elems))
        assert p.threads == 128 and p.staged_elems < p.slice_elems, (P, p)
        check(w, run(w, inp, p), inp)
        check(w, run(w, inp, p, in_place=True), inp)
