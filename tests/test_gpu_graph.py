"""The library's calls are stream-ordered, allocate nothing and never wait
on the host, so a sequence of them captures into a CUDA graph and replays
with the same results as the eager calls."""
import numpy as np
import pytest
import torch

from dsmem_thread_block_gb300 import _credit as C
from dsmem_thread_block_gb300 import workloads as wl

from gpu_helpers import DT, OPS, to_device, to_host

pytestmark = pytest.mark.gpu


def test_calls_capture_into_a_cuda_graph_and_replay():
    dev = torch.cuda.current_device()
    ln = wl.LAYERNORM_BF16_1024x262144.with_rows(6)
    q = wl.QUANTIZE_F32_4096x65536.with_rows(5)
    pe = wl.PEARSON_F32_4096x65536.with_rows(4)
    li, qi, pi = ln.generate(), q.generate(), pe.generate()
    lx, lg, lb = to_device(li["x"]), to_device(li["gamma"]), to_device(li["beta"])
    qx, px, pu = to_device(qi["x"]), to_device(pi["x"]), to_device(pi["u"])
    ly = torch.empty_like(lx)
    qq = torch.empty(qx.shape, dtype=torch.int8, device="cuda")
    qs = torch.empty(q.rows, device="cuda")
    py = torch.empty_like(px)
    pr = torch.empty(pe.rows, device="cuda")
    plans = {
        "ln": C.credit_plan_for(C.LAYERNORM, ln.rows, ln.cols, C.BF16, dev, C.CLUSTER, 8),
        "q": C.credit_plan_for(C.QUANTIZE, q.rows, q.cols, C.F32, dev, C.CLUSTER, 4),
        "pe_tp": C.credit_plan_for(C.PEARSON, pe.rows, pe.cols, C.F32, dev, C.TWO_PASS, 1),
    }
    ws = torch.empty(int(plans["pe_tp"].workspace_bytes), dtype=torch.uint8, device="cuda")

    def calls(stream):
        assert C.credit_layernorm(lx.data_ptr(), ly.data_ptr(), ln.rows, ln.cols, C.BF16,
                                  lg.data_ptr(), lb.data_ptr(), C.F32, ln.eps, plans["ln"], 0, 0,
                                  stream) == C.OK
        assert C.credit_quantize(qx.data_ptr(), qq.data_ptr(), qs.data_ptr(), q.rows, q.cols,
                                 C.F32, plans["q"], 0, 0, stream) == C.OK
        assert C.credit_pearson(px.data_ptr(), pu.data_ptr(), py.data_ptr(), pr.data_ptr(),
                                pe.rows, pe.cols, C.F32, pe.eps, plans["pe_tp"], ws.data_ptr(),
                                ws.numel(), stream) == C.OK

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):  # eager run (also sets each kernel's attributes once)
        calls(s.cuda_stream)
    s.synchronize()
    eager = [to_host(ly).copy(), qq.cpu().numpy().copy(), qs.cpu().numpy().copy(),
             py.cpu().numpy().copy(), pr.cpu().numpy().copy()]
    for t in (ly, py, pr, qs):
        t.zero_()
    qq.zero_()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        calls(s.cuda_stream)
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        got = [to_host(ly), qq.cpu().numpy(), qs.cpu().numpy(), py.cpu().numpy(), pr.cpu().numpy()]
        for a, b in zip(got, eager):
            assert np.array_equal(a, b)
    assert C.credit_get_device_error(dev) == C.OK
