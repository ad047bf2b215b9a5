"""Seeded random shapes through every plan variant, against the oracle.

Each case draws an operator, element and parameter type, row count, width
(aligned, ragged, narrow, a few slices wide), input distribution, a variant
the shape allows (automatic, one row per cluster at a random legal P with
either exchange, several rows per cluster, persistent, pipelined, warp per
row, two-pass), absent parameters and in-place calls; the cases are fixed by
the seed, so a failure names a reproducible shape."""
import numpy as np
import pytest
import torch

from dsmem_thread_block_gb300 import _credit as C
from dsmem_thread_block_gb300 import workloads as wl

from gpu_helpers import DT, OPS, check, check_pearson, check_quant, run

pytestmark = pytest.mark.gpu

N_CASES = 200
SEED = 20261202


def _draw(rng, k):
    op = str(rng.choice([wl.SOFTMAX, wl.LAYERNORM, wl.RMSNORM, wl.QUANTIZE, wl.WEIGHTED_STD,
                     wl.PEARSON]))
    dtype = str(rng.choice(["f32", "bf16"]))
    vec = 4 if dtype == "f32" else 8
    kind = str(rng.choice(["narrow", "mid", "wide", "ragged"]))
    if kind == "narrow":
        cols = int(vec * rng.integers(1, 65))
    elif kind == "mid":
        cols = int(vec * rng.integers(65, 4097))
    elif kind == "wide":
        cols = int(vec * rng.integers(4097, 40001))
    else:
        cols = int(rng.integers(3, 20000)) | 1  # odd: the element path
    rows = int(rng.integers(1, 97 if cols < 50000 else 17))
    kw = {"x_mean": float(rng.normal(0, 2)), "x_std": float(rng.uniform(0.1, 4.0)),
          "eps": float(rng.choice([1e-5, 1e-6]))}
    if op == wl.SOFTMAX and rng.random() < 0.3:
        kw["spike_frac"] = 0.01
    if op in (wl.LAYERNORM, wl.RMSNORM, wl.WEIGHTED_STD):
        kw["param_dtype"] = str(rng.choice(["f32", "bf16"]))
        if op == wl.WEIGHTED_STD:
            kw["p_uniform"] = True
    if op == wl.PEARSON:
        kw["u_corr"] = float(rng.uniform(-0.9, 0.9))
    w = wl.Workload(f"rand{k}_{op}_{dtype}_{rows}x{cols}", op, dtype, rows, cols,
                    seed=int(rng.integers(1, 1 << 30)), **kw)
    return w, rng


def _plan(w, rng):
    dev = torch.cuda.current_device()
    o, d = OPS[w.op], DT[w.dtype]
    choices = ["auto", "cluster", "two_pass"]
    if w.op in (wl.SOFTMAX, wl.LAYERNORM, wl.RMSNORM):
        choices += ["persistent", "pipelined", "warp_rows"]
    if w.op != wl.PEARSON:
        choices += ["rows"]
    for _ in range(20):
        v = str(rng.choice(choices))
        try:
            if v == "auto":
                return v, C.credit_plan(o, w.rows, w.cols, d, dev)
            if v == "two_pass":
                return v, C.credit_plan_for(o, w.rows, w.cols, d, dev, C.TWO_PASS, 1)
            if v == "warp_rows":
                return v, C.credit_plan_for(o, w.rows, w.cols, d, dev, C.WARP_ROWS, 1)
            P = int(rng.integers(1, 17))
            if v == "cluster":
                x = C.EXCHANGE_BARRIER if rng.random() < 0.3 else C.EXCHANGE_ASYNC
                return f"cluster:{P}", C.credit_plan_with(o, w.rows, w.cols, d, dev, C.CLUSTER, P,
                                                          exchange=x)
            if v == "rows":
                R = int(rng.choice([2, 4]))
                return f"cluster:{P}x{R}", C.credit_plan_with(o, w.rows, w.cols, d, dev, C.CLUSTER,
                                                              P, rows_per_cluster=R)
            var = C.CLUSTER_PERSISTENT if v == "persistent" else C.CLUSTER_PIPELINED
            return f"{v}:{P}", C.credit_plan_for(o, w.rows, w.cols, d, dev, var, P)
        except C.CreditError as e:
            assert e.status == C.ERR_NO_LEGAL_PLAN, (w.name, v, e)
    return "auto", C.credit_plan(o, w.rows, w.cols, d, dev)


def _cases():
    rng = np.random.default_rng(SEED)
    out = []
    for k in range(N_CASES):
        w, rng = _draw(rng, k)
        out.append((w, int(rng.integers(0, 1 << 30))))
    return out


CASES = _cases()


@pytest.mark.parametrize("w,pseed", CASES, ids=[c[0].name for c in CASES])
def test_random_shape_matches_oracle(w, pseed):
    rng = np.random.default_rng(pseed)
    inp = w.generate()
    if w.op in (wl.LAYERNORM, wl.RMSNORM) and rng.random() < 0.2:
        inp = {"x": inp["x"]}  # parameters absent
    name, plan = _plan(w, rng)
    in_place = bool(rng.random() < 0.2) and w.op not in (wl.QUANTIZE, wl.PEARSON)
    got = run(w, inp, plan, in_place=in_place)
    if w.op == wl.QUANTIZE:
        check_quant(got, inp)
    elif w.op == wl.PEARSON:
        check_pearson(w, got, inp)
    else:
        check(w, got, inp)
    assert C.credit_get_device_error(torch.cuda.current_device()) == C.OK, name
