"""The allocation-free two-pass entry point (for callers that cannot call
cudaMalloc: memory already handed to their own pool, hot loops that must not
synchronise the device, plug-in hosts without an allocator) gives the same
results as the regular two-pass call with a caller-provided workspace, on two
calls in a row that share the library's fixed scratch array, and both match
the fp64 oracle within the parity tolerances.

This file is collected last on purpose."""
import numpy as np
import pytest
import torch

from dsmem_thread_block_gb300 import _credit as C
from dsmem_thread_block_gb300 import workloads as wl

from gpu_helpers import DT, OPS, RTOL, call, check, make_plan, to_device, to_host

pytestmark = pytest.mark.gpu


def _noalloc(w, dx, dy, params):
    p0 = params.get("gamma", params.get("weight"))
    p1 = params.get("beta")
    pdt = DT[w.param_dtype] if w.param_dtype else C.F32
    return C.credit_two_pass_noalloc(OPS[w.op], dx.data_ptr(), dy.data_ptr(), w.rows, w.cols,
                                     DT[w.dtype], p0.data_ptr() if p0 is not None else 0,
                                     p1.data_ptr() if p1 is not None else 0, pdt, w.eps,
                                     torch.cuda.current_stream().cuda_stream)


CASES = [wl.LAYERNORM_BF16_1024x262144.with_rows(8), wl.SOFTMAX_F32_64x4096,
         wl.RMSNORM_BF16_2048x786432.with_rows(4)]


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_noalloc_matches_workspace_two_pass(w):
    plan = make_plan(w, C.TWO_PASS)
    for seed_shift in (0, 1):  # two calls in a row, different data
        w2 = wl.Workload(**{**w.__dict__, "seed": w.seed + 100 * seed_shift})
        inp = w2.generate()
        dx = to_device(inp["x"])
        params = {k: to_device(v) for k, v in inp.items() if k != "x"}
        ref = torch.empty_like(dx)
        assert call(w2, dx, ref, params, plan) == C.OK
        got = torch.full_like(dx, float("nan"))
        assert _noalloc(w2, dx, got, params) == C.OK
        torch.cuda.synchronize()
        a = to_host(got).astype(np.float64) if w.dtype == "f32" else \
            wl.bf16_bits_to_f32(to_host(got)).astype(np.float64)
        b = to_host(ref).astype(np.float64) if w.dtype == "f32" else \
            wl.bf16_bits_to_f32(to_host(ref)).astype(np.float64)
        assert np.isfinite(a).all()
        assert (np.abs(a - b) <= RTOL[w.dtype] * np.abs(b) + 1e-30).all()
        # and against the oracle itself, not only the other CUDA path
        check(w2, to_host(got), inp)


def test_noalloc_size_limit():
    # softmax fp32 with 128 columns: one 16-byte partial per row, so the
    # 2 MiB array holds exactly 131072 rows.  That many run (and match the
    # workspace path); one more row is rejected on the host.  Both buffers
    # are real, so even a wrong check could not touch foreign memory.
    w = wl.Workload("softmax_f32_131073x128", wl.SOFTMAX, "f32", 131073, 128, seed=3)
    inp = w.generate()
    dx = to_device(inp["x"])
    dy = torch.empty_like(dx)
    s = torch.cuda.current_stream().cuda_stream
    st = C.credit_two_pass_noalloc(C.SOFTMAX, dx.data_ptr(), dy.data_ptr(), 131073, 128,
                                   C.F32, 0, 0, C.F32, 0.0, s)
    assert st == C.ERR_INVALID_ARG
    w1 = w.with_rows(131072)
    st = C.credit_two_pass_noalloc(C.SOFTMAX, dx.data_ptr(), dy.data_ptr(), 131072, 128,
                                   C.F32, 0, 0, C.F32, 0.0, s)
    assert st == C.OK
    ref = torch.empty_like(dx)
    assert call(w1, dx, ref, {}, make_plan(w1, C.TWO_PASS)) == C.OK
    torch.cuda.synchronize()
    a = dy[:131072].double().cpu().numpy()
    b = ref[:131072].double().cpu().numpy()
    assert (np.abs(a - b) <= RTOL["f32"] * np.abs(b)).all()
    check(w1, to_host(dy)[:131072], {"x": inp["x"][:131072]})
