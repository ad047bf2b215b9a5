"""Host-buffer calls (credit_run_host): chunked copies and kernels on the
library's pipeline streams give byte-identical results to the device-buffer
calls with the same plan, for every chunking of the rows (one chunk, ragged
last chunk, one row per chunk), and the oracle agrees."""
import numpy as np
import pytest
import torch

from dsmem_thread_block_gb300 import _credit as C
from dsmem_thread_block_gb300 import workloads as wl

from gpu_helpers import DT, OPS, check, check_pearson, check_quant, run, to_device

pytestmark = pytest.mark.gpu


def _pinned(a: np.ndarray) -> torch.Tensor:
    t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
    return t.pin_memory()


def _host_run(w, inp, plan, rpc):
    """Run through credit_run_host; return (y bytes, row results or None)."""
    hx = _pinned(inp["x"])
    quant, pearson = w.op == wl.QUANTIZE, w.op == wl.PEARSON
    hy = torch.empty(inp["x"].shape, dtype=torch.int8 if quant else hx.dtype).pin_memory()
    hu = _pinned(inp["u"]) if pearson else None
    hr = torch.full((w.rows,), 7.0, dtype=torch.float32).pin_memory() if (quant or pearson) else None
    params = {k: to_device(v) for k, v in inp.items() if k not in ("x", "u")}
    g = params.get("gamma", params.get("weight"))
    b = params.get("beta")
    pdt = DT[w.param_dtype] if w.param_dtype else C.F32
    call = C.host_call(OPS[w.op], DT[w.dtype], w.rows, w.cols, hx.data_ptr(), hy.data_ptr(),
                       u=hu.data_ptr() if hu is not None else 0,
                       row_out=hr.data_ptr() if hr is not None else 0,
                       p0=g.data_ptr() if g is not None else 0,
                       p1=b.data_ptr() if b is not None else 0, param_dtype=pdt, eps=w.eps)
    nbytes = C.credit_host_buffer_bytes(call, plan, rpc)
    buf = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    st = C.credit_run_host(call, plan, buf.data_ptr(), nbytes, rpc, stream)
    assert st == C.OK, C.status_string(st)
    torch.cuda.current_stream().synchronize()
    assert C.credit_get_device_error(torch.cuda.current_device()) == C.OK
    y = hy.numpy()
    if y.dtype == np.int16:
        y = y.view(np.uint16)
    return y, (hr.numpy().copy() if hr is not None else None)


CASES = [
    wl.LAYERNORM_BF16_1024x262144.with_rows(10),
    wl.Workload("softmax_f32_37x8192", wl.SOFTMAX, "f32", 37, 8192, seed=80, x_std=3.0),
    wl.QUANTIZE_F32_4096x65536.with_rows(9),
    wl.PEARSON_F32_4096x65536.with_rows(7),
    wl.Workload("rmsnorm_bf16_13x24576", wl.RMSNORM, "bf16", 13, 24576, seed=81, eps=1e-6,
                param_dtype="bf16"),
]


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_host_pipeline_matches_device_calls(w):
    inp = w.generate()
    dev = torch.cuda.current_device()
    plans = [C.credit_plan(OPS[w.op], w.rows, w.cols, DT[w.dtype], dev),
             C.credit_plan_for(OPS[w.op], w.rows, w.cols, DT[w.dtype], dev, C.TWO_PASS, 1)]
    for plan in plans:
        ref = run(w, inp, plan)  # the device-buffer call
        for rpc in (w.rows, 4, 1):
            y, r = _host_run(w, inp, plan, rpc)
            if w.op == wl.QUANTIZE:
                assert np.array_equal(y, ref[0]) and np.array_equal(r, ref[1])
                check_quant((y, r), inp)
            elif w.op == wl.PEARSON:
                assert np.array_equal(y, ref[0]) and np.array_equal(r, ref[1])
                check_pearson(w, (y, r), inp)
            else:
                assert np.array_equal(y, ref)
                check(w, y, inp)


def test_host_pipeline_orders_after_the_callers_stream():
    # the caller writes the parameters on its stream just before the call:
    # the pipeline must see them
    w = wl.Workload("rmsnorm_f32_6x4096", wl.RMSNORM, "f32", 6, 4096, seed=82, eps=1e-6,
                    param_dtype="f32")
    inp = w.generate()
    dev = torch.cuda.current_device()
    plan = C.credit_plan(C.RMSNORM, w.rows, w.cols, C.F32, dev)
    wt = torch.zeros(w.cols, device="cuda")
    hx = _pinned(inp["x"])
    hy = torch.empty(hx.shape, dtype=torch.float32).pin_memory()
    call = C.host_call(C.RMSNORM, C.F32, w.rows, w.cols, hx.data_ptr(), hy.data_ptr(),
                       p0=wt.data_ptr(), param_dtype=C.F32, eps=w.eps)
    nbytes = C.credit_host_buffer_bytes(call, plan, 2)
    buf = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        torch.cuda._sleep(2_000_000)  # keep the stream busy before the write
        wt.copy_(to_device(inp["weight"]), non_blocking=True)
        assert C.credit_run_host(call, plan, buf.data_ptr(), nbytes, 2, s.cuda_stream) == C.OK
    s.synchronize()
    check(w, hy.numpy(), inp)
