"""Shared helpers for the GPU parity tests: move seeded inputs to the device,
call the library through its C ABI, read results back, and compare them with
the fp64 oracle under the stated tolerances.

Tolerances (per element, o = oracle value in fp64, g = GPU value widened):
  fp32 outputs   |g - o| <= 1e-5   * |o|
  bf16 outputs   |g - o| <= 2^-7   * |o|        (one bf16 ulp at a binade top)
LayerNorm adds a cancellation term.  fp32 cannot hold the row mean mu to
better than ~2^-24 |mu|, so z = (x - mu) / sigma carries an absolute error of
order 2^-24 (|z| + |mu| / sigma) however it is computed, and the final
y = z * gamma + beta can cancel to a tiny |o|.  Its bound is therefore
  |g - o| <= rtol * |o| + 1e-5 * (|gamma| (|z| + |mu| / sigma) + |beta|)
with sigma = sqrt(var + eps) of the row (1e-5 is ~170 fp32 ulps: room for
the summation error of the statistics), and the tests report how many
elements pass only through that term.
Pearson's y = zx zu (z the deviations over sqrt(var + eps)) carries that
error in both factors.  A short row's fp32 mean is off by about 2^-24 times
the row's typical magnitude rather than |mean| (a mean near zero of values
near +-2 still errs by ~2^-24 * 2), so the term uses the row's rms:
  |g - o| <= rtol * |o| + 1e-5 * (|zu| (|zx| + rms_x / sx) + |zx| (|zu| + rms_u / su))
and its fp32 correlation r is held to |g - o| <= 1e-5 (r lies in [-1, 1]).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from dsmem_thread_block_gb300 import _credit as C
from dsmem_thread_block_gb300 import workloads as wl

RTOL = {"f32": 1e-5, "bf16": 2.0 ** -7}
LN_CANCEL = 1e-5
OPS = {wl.SOFTMAX: C.SOFTMAX, wl.LAYERNORM: C.LAYERNORM, wl.RMSNORM: C.RMSNORM,
       wl.QUANTIZE: C.QUANTIZE, wl.WEIGHTED_STD: C.WEIGHTED_STD, wl.PEARSON: C.PEARSON}
DT = {"f32": C.F32, "bf16": C.BF16}


def to_device(a: np.ndarray, dev="cuda") -> torch.Tensor:
    """numpy fp32 / uint16(bf16 bits) -> CUDA tensor of the same bytes."""
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(a)
    return t.to(dev)


def to_host(t: torch.Tensor) -> np.ndarray:
    """CUDA tensor -> numpy with the same bytes (bf16 as uint16 bits)."""
    t = t.cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def make_plan(w: wl.Workload, variant=None, P=1, rows=None):
    rows = w.rows if rows is None else rows
    dev = torch.cuda.current_device()
    if variant is None:
        return C.credit_plan(OPS[w.op], rows, w.cols, DT[w.dtype], dev)
    return C.credit_plan_for(OPS[w.op], rows, w.cols, DT[w.dtype], dev, variant, P)


def call(w: wl.Workload, dx: torch.Tensor, dy: torch.Tensor, params: dict, plan,
         rows=None, stream=None) -> int:
    """One library call through the C ABI on device tensors; returns status."""
    rows = w.rows if rows is None else rows
    ws = None
    if plan is not None and plan.workspace_bytes:
        ws = torch.empty(int(plan.workspace_bytes), dtype=torch.uint8, device=dx.device)
    wptr = ws.data_ptr() if ws is not None else 0
    wbytes = int(plan.workspace_bytes) if ws is not None else 0
    s = stream if stream is not None else torch.cuda.current_stream().cuda_stream
    pdt = DT[w.param_dtype] if w.param_dtype else C.F32
    if w.op == wl.SOFTMAX:
        return C.credit_softmax(dx.data_ptr(), dy.data_ptr(), rows, w.cols, DT[w.dtype], plan,
                                wptr, wbytes, s)
    if w.op == wl.LAYERNORM:
        g, b = params.get("gamma"), params.get("beta")
        return C.credit_layernorm(dx.data_ptr(), dy.data_ptr(), rows, w.cols, DT[w.dtype],
                                  g.data_ptr() if g is not None else 0,
                                  b.data_ptr() if b is not None else 0, pdt, w.eps, plan,
                                  wptr, wbytes, s)
    if w.op == wl.QUANTIZE:
        return C.credit_quantize(dx.data_ptr(), dy.data_ptr(), params["scales"].data_ptr(), rows,
                                 w.cols, DT[w.dtype], plan, wptr, wbytes, s)
    if w.op == wl.PEARSON:
        return C.credit_pearson(dx.data_ptr(), params["u"].data_ptr(), dy.data_ptr(),
                                params["r"].data_ptr(), rows, w.cols, DT[w.dtype], w.eps, plan,
                                wptr, wbytes, s)
    wt = params.get("weight")
    if w.op == wl.WEIGHTED_STD:
        return C.credit_weighted_std(dx.data_ptr(), dy.data_ptr(), rows, w.cols, DT[w.dtype],
                                     wt.data_ptr(), pdt, w.eps, plan, wptr, wbytes, s)
    return C.credit_rmsnorm(dx.data_ptr(), dy.data_ptr(), rows, w.cols, DT[w.dtype],
                            wt.data_ptr() if wt is not None else 0, pdt, w.eps, plan, wptr,
                            wbytes, s)


def run(w: wl.Workload, inputs: dict, plan, in_place=False):
    """Run the library on host inputs; return the output bytes (numpy) -- for
    quantization the pair (int8 codes, fp32 scales)."""
    dx = to_device(inputs["x"])
    params = {k: to_device(v) for k, v in inputs.items() if k != "x"}
    if w.op == wl.QUANTIZE:
        rows = inputs["x"].shape[0]
        dq = torch.full(dx.shape, 77, dtype=torch.int8, device=dx.device)
        params["scales"] = torch.full((rows,), -1.0, dtype=torch.float32, device=dx.device)
        st = call(w, dx, dq, params, plan, rows=rows)
        assert st == C.OK, C.status_string(st)
        torch.cuda.synchronize()
        assert C.credit_get_device_error(torch.cuda.current_device()) == C.OK
        return dq.cpu().numpy(), params["scales"].cpu().numpy()
    if w.op == wl.PEARSON:
        rows = inputs["x"].shape[0]
        params["r"] = torch.full((rows,), 7.0, dtype=torch.float32, device=dx.device)
        dy = {False: None, True: dx, "x": dx, "u": params["u"]}[in_place]
        if dy is None:
            dy = torch.empty_like(dx)
        st = call(w, dx, dy, params, plan, rows=rows)
        assert st == C.OK, C.status_string(st)
        torch.cuda.synchronize()
        assert C.credit_get_device_error(torch.cuda.current_device()) == C.OK
        return to_host(dy), params["r"].cpu().numpy()
    dy = dx if in_place else torch.empty_like(dx)
    st = call(w, dx, dy, params, plan, rows=inputs["x"].shape[0])
    assert st == C.OK, C.status_string(st)
    torch.cuda.synchronize()
    assert C.credit_get_device_error(torch.cuda.current_device()) == C.OK
    return to_host(dy)


def oracle_rows(w: wl.Workload, inputs: dict, rows=None, want_z=False):
    """fp64 oracle on all rows (or the listed row indices)."""
    x = inputs["x"] if rows is None else inputs["x"][rows]
    if w.op == wl.SOFTMAX:
        return oracle.softmax(x), None
    if w.op == wl.LAYERNORM:
        y, z = oracle.layernorm(x, inputs.get("gamma"), inputs.get("beta"), eps=w.eps,
                                want_z=True)
        return y, z
    if w.op == wl.WEIGHTED_STD:
        y = oracle.weighted_std(x, inputs["weight"], eps=w.eps)
        return y, y
    return oracle.rmsnorm(x, inputs.get("weight"), eps=w.eps), None


def check(w: wl.Workload, got: np.ndarray, inputs: dict, rows=None, scale=1.0) -> dict:
    """Compare GPU output bytes with the oracle; assert the tolerance."""
    want, z = oracle_rows(w, inputs, rows)
    g = oracle.widen(got if rows is None else got[rows])
    rtol = RTOL[w.dtype] * scale
    err = np.abs(g - want)
    bound = rtol * np.abs(want)
    only_cancel = 0
    if w.op in (wl.LAYERNORM, wl.WEIGHTED_STD):
        gam = oracle.widen(inputs["gamma"]) if "gamma" in inputs else 1.0
        bet = oracle.widen(inputs["beta"]) if "beta" in inputs else 0.0
        xw = oracle.widen(inputs["x"] if rows is None else inputs["x"][rows])
        wts = oracle.widen(inputs["weight"]) if w.op == wl.WEIGHTED_STD else np.ones(xw.shape[1])
        mean = (xw * wts).sum(axis=1, keepdims=True) / wts.sum()
        var = (wts * (xw - mean) ** 2).sum(axis=1, keepdims=True) / wts.sum()
        mu_over_sigma = np.abs(mean) / np.sqrt(var + w.eps)
        extra = LN_CANCEL * scale * (np.abs(gam) * (np.abs(z) + mu_over_sigma) + np.abs(bet))
        only_cancel = int(((err > bound) & (err <= bound + extra)).sum())
        bound = bound + extra
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(
            f"{w.name}: {int(bad.sum())} of {err.size} elements out of tolerance; worst at "
            f"{i}: got {g[i]!r} want {want[i]!r} err {err[i]:.3e} bound {bound[i]:.3e}")
    rel = err / np.maximum(np.abs(want), 1e-300)
    return {"max_rel": float(rel.max()), "only_cancel": only_cancel, "n": int(err.size)}


def check_quant(got, inputs: dict, rows=None):
    """Quantization parity is bit-exact: codes and scales."""
    q, s = got
    x = inputs["x"] if rows is None else inputs["x"][rows]
    qo, so = oracle.quantize(x)
    if rows is not None:
        q, s = q[rows], s[rows]
    assert np.array_equal(s.view(np.uint32), so.view(np.uint32)), "scales differ"
    bad = np.argwhere(q != qo)
    assert bad.size == 0, f"{len(bad)} codes differ, first at {bad[0]}: {q[tuple(bad[0])]} vs {qo[tuple(bad[0])]}"


PEARSON_CANCEL = 1e-5
R_ATOL = 1e-5


def check_pearson(w: wl.Workload, got, inputs: dict, rows=None, scale=1.0) -> dict:
    """Compare GPU (y, r) with the oracle's; assert the stated tolerances."""
    y, r = got
    x = inputs["x"] if rows is None else inputs["x"][rows]
    u = inputs["u"] if rows is None else inputs["u"][rows]
    want, rw = oracle.pearson(x, u, eps=w.eps)
    g = oracle.widen(y if rows is None else y[rows])
    rg = (r if rows is None else r[rows]).astype(np.float64)
    xw, uw = oracle.widen(x), oracle.widen(u)
    mx, mu = xw.mean(axis=1, keepdims=True), uw.mean(axis=1, keepdims=True)
    sx = np.sqrt(((xw - mx) ** 2).mean(axis=1, keepdims=True) + w.eps)
    su = np.sqrt(((uw - mu) ** 2).mean(axis=1, keepdims=True) + w.eps)
    zx, zu = (xw - mx) / sx, (uw - mu) / su
    err = np.abs(g - want)
    rms_x = np.sqrt((xw ** 2).mean(axis=1, keepdims=True))
    rms_u = np.sqrt((uw ** 2).mean(axis=1, keepdims=True))
    bound = RTOL[w.dtype] * scale * np.abs(want) + PEARSON_CANCEL * scale * (
        np.abs(zu) * (np.abs(zx) + rms_x / sx) + np.abs(zx) * (np.abs(zu) + rms_u / su))
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(
            f"{w.name}: {int(bad.sum())} of {err.size} outputs out of tolerance; worst at {i}: "
            f"got {g[i]!r} want {want[i]!r} err {err[i]:.3e} bound {bound[i]:.3e}")
    rerr = np.abs(rg - rw)
    assert (rerr <= R_ATOL * scale).all(), \
        f"{w.name}: r differs by {rerr.max():.3e} at row {int(np.argmax(rerr))}"
    return {"max_r_err": float(rerr.max()), "n": int(err.size)}
