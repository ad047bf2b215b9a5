"""Shared helpers for the GPU parity tests: move seeded inputs to the device,
call the library through its C ABI, read results back, and compare them with
the fp64 oracle under the stated tolerances.

Tolerances (per element, o = oracle value in fp64, g = GPU value widened):
  fp32 outputs   |g - o| <= 1e-5   * |o|
  bf16 outputs   |g - o| <= 2^-7   * |o|        (one bf16 ulp at a binade top)
  quantization   bit-exact codes and scales

Cancellation (LayerNorm, weighted standardization, Pearson).  These outputs
are a difference of O(1) quantities: y = z gamma + beta with z = (x - mu) /
sigma, and z itself is x - mu over sigma.  Any fp32 evaluation rounds its
intermediates at their own magnitude, so its absolute error scales with
  S = |gamma| (|z| + rms / sigma) + |beta|      (rms = sqrt(mean x^2))
and not with |o|, which can be arbitrarily small: |mu| / sigma enters
through the fp32 row mean (its rounding is relative to the summands, i.e.
to rms), |z| through the rounding of z and of 1/sigma, |beta| and the final
rounding through the last fused multiply-add.  An element is therefore held
to the relative bound unless it lies in the cancellation zone, where the
bound becomes the fp32 evaluation error instead:
  |g - o| <= max(rtol |o|,  u_out |o| + C u S),   u = 2^-24,  C = 16,
u_out the output's own rounding (0 for fp32 outputs -- it is part of C u S --
and 2^-8 for bf16).  C counts the roundings after the statistics (the two
fused multiply-adds, the product mu r and the four correctly rounded steps
of r = 1 / sqrt(M2 / N + eps): at most 3.5 u S together, whatever the
kernel) and leaves 12.5 u S for the fp32 mean and M2.  Those are recursive
sums that the kernels split over at most a few hundred terms per thread
before an ordered fold; their worst-case first-order bound grows with the
term count, but their rounding errors are unbiased and cancel (Higham and
Mary's probabilistic bound grows with its square root), and the largest
total error measured over the whole GPU suite is 2.7 u S.  For
Pearson, y = zx zu, S = |zu| (|zx| + rms_x / sx) + |zx| (|zu| + rms_u / su),
and r is held to 1e-5 absolute (r lies in [-1, 1]).
Outside the zone (rtol |o| >= C u S) the bound is exactly rtol |o|.  Each
check reports the elements that pass only through the zone term and the
largest error in units of u S; for fp32 inputs it asserts that they are at
most a quarter of the zone's elements (bf16 inputs take few distinct values
near a large mean, so their zone elements come in clumps and a share means
little).  How many there are depends on the rows: for fp32
outputs a pure relative bound is out of reach for any fp32 evaluation -- even
an ideal one (exact statistics, one rounding per operation) misses 1e-5 |o|
on about 0.2 % of LayerNorm elements of N(0.5, 2) rows (pinned on the CPU in
tests/test_tolerance.py), and on more where the mean is large against sigma
(rms / sigma large); the bf16 workloads' full-size tests also assert that
fewer than 1e-4 of their elements need the zone term.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from dsmem_thread_block_gb300 import _credit as C
from dsmem_thread_block_gb300 import workloads as wl

RTOL = {"f32": 1e-5, "bf16": 2.0 ** -7}
U32 = 2.0 ** -24       # fp32 unit roundoff
C_ZONE = 16            # fp32 evaluation error in units of u S (see above)
U_OUT = {"f32": 0.0, "bf16": 2.0 ** -8}
ZONE_SHARE = 0.25      # elements passing only through the zone term, share of the zone
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


def cancel_scale(w: wl.Workload, inputs: dict, z: np.ndarray, rows=None) -> np.ndarray:
    """S of the cancellation bound for LayerNorm / weighted standardization:
    |gamma| (|z| + rms / sigma) + |beta|, rms and sigma (weighted for the
    weighted standardization) of each row."""
    gam = oracle.widen(inputs["gamma"]) if "gamma" in inputs else 1.0
    bet = oracle.widen(inputs["beta"]) if "beta" in inputs else 0.0
    xw = oracle.widen(inputs["x"] if rows is None else inputs["x"][rows])
    wts = oracle.widen(inputs["weight"]) if w.op == wl.WEIGHTED_STD else np.ones(xw.shape[1])
    W = wts.sum()
    mean = (xw * wts).sum(axis=1, keepdims=True) / W
    var = (wts * (xw - mean) ** 2).sum(axis=1, keepdims=True) / W
    rms = np.sqrt((wts * xw * xw).sum(axis=1, keepdims=True) / W)
    return np.abs(gam) * (np.abs(z) + rms / np.sqrt(var + w.eps)) + np.abs(bet)


def bounds(w: wl.Workload, inputs: dict, rows=None, scale=1.0, with_scale=False):
    """(oracle values, per-element bound, strict relative bound[, u S or None])."""
    want, z = oracle_rows(w, inputs, rows)
    strict = RTOL[w.dtype] * scale * np.abs(want)
    if w.op in (wl.LAYERNORM, wl.WEIGHTED_STD):
        uS = U32 * cancel_scale(w, inputs, z, rows)
        zone = U_OUT[w.dtype] * np.abs(want) + C_ZONE * scale * uS
        out = (want, np.maximum(strict, zone), strict, uS)
    else:
        out = (want, strict, strict, None)
    return out if with_scale else out[:3]


def _report(name: str, err, bound, strict, want, dtype: str, uS=None,
            in_dtype: str = "f32") -> dict:
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(
            f"{name}: {int(bad.sum())} of {err.size} elements out of tolerance; worst at "
            f"{i}: want {want[i]!r} err {err[i]:.3e} bound {bound[i]:.3e}")
    only_zone = int((err > strict).sum())
    in_zone = bound > strict
    rel = err / np.maximum(np.abs(want), 1e-300)
    res = {"max_rel": float(rel[~in_zone].max()) if (~in_zone).any() else 0.0,
           "only_cancel": only_zone, "zone": int(in_zone.sum()), "n": int(err.size),
           "only_cancel_frac": only_zone / max(1, err.size)}
    if uS is not None:
        res["max_c"] = float((np.maximum(err - U_OUT[dtype] * np.abs(want), 0) / uS).max())
    if in_dtype == "f32":
        assert only_zone <= ZONE_SHARE * res["zone"], \
            f"{name}: {only_zone} of the zone's {res['zone']} elements need the cancellation term"
    if only_zone:
        print(f"[parity] {name}: max_rel {res['max_rel']:.3e} outside the zone; "
              f"{only_zone} of {err.size} ({100 * res['only_cancel_frac']:.4f} %; zone "
              f"{res['zone']}) pass only through the cancellation term; "
              f"max err {res.get('max_c', float('nan')):.2f} u S")
    return res


def check(w: wl.Workload, got: np.ndarray, inputs: dict, rows=None, scale=1.0) -> dict:
    """Compare GPU output bytes with the oracle; assert the tolerance."""
    want, bound, strict, uS = bounds(w, inputs, rows, scale, with_scale=True)
    g = oracle.widen(got if rows is None else got[rows])
    return _report(w.name, np.abs(g - want), bound, strict, want, w.dtype, uS, w.dtype)


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
    rms_x = np.sqrt((xw ** 2).mean(axis=1, keepdims=True))
    rms_u = np.sqrt((uw ** 2).mean(axis=1, keepdims=True))
    S = np.abs(zu) * (np.abs(zx) + rms_x / sx) + np.abs(zx) * (np.abs(zu) + rms_u / su)
    strict = RTOL[w.dtype] * scale * np.abs(want)
    bound = np.maximum(strict, U_OUT[w.dtype] * np.abs(want) + C_ZONE * U32 * scale * S)
    res = _report(w.name, np.abs(g - want), bound, strict, want, w.dtype, U32 * S, w.dtype)
    rerr = np.abs(rg - rw)
    assert (rerr <= R_ATOL * scale).all(), \
        f"{w.name}: r differs by {rerr.max():.3e} at row {int(np.argmax(rerr))}"
    res["max_r_err"] = float(rerr.max())
    return res
