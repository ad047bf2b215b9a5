"""The torch layer (package functions) on CUDA tensors: automatic plans,
forced plans from `plan()`, workspaces from torch's allocator, and the
per-row outputs of quantization and Pearson."""
import numpy as np
import pytest
import torch

import dsmem_thread_block_gb300 as credit
from dsmem_thread_block_gb300 import workloads as wl

from gpu_helpers import check, check_pearson, check_quant, to_device, to_host

pytestmark = pytest.mark.gpu


def test_torch_layer_every_operator():
    ln = wl.LAYERNORM_BF16_1024x262144.with_rows(3)
    i = ln.generate()
    x, g, b = to_device(i["x"]), to_device(i["gamma"]), to_device(i["beta"])
    check(ln, to_host(credit.layernorm(x, g, b, eps=ln.eps)), i)
    for p in (credit.plan("layernorm", ln.rows, ln.cols, torch.bfloat16, variant="cluster",
                          cluster_size=8, exchange="barrier"),
              credit.plan("layernorm", ln.rows, ln.cols, torch.bfloat16, variant="persistent",
                          cluster_size=4),
              credit.plan("layernorm", ln.rows, ln.cols, torch.bfloat16, variant="two_pass")):
        check(ln, to_host(credit.layernorm(x, g, b, eps=ln.eps, plan=p)), i)

    sm = wl.SOFTMAX_F32_64x4096
    i = sm.generate()
    check(sm, to_host(credit.softmax(to_device(i["x"]))), i)

    rms = wl.Workload("rmsnorm_bf16_4x65536", wl.RMSNORM, "bf16", 4, 65536, seed=95, eps=1e-6,
                      param_dtype="bf16")
    i = rms.generate()
    check(rms, to_host(credit.rmsnorm(to_device(i["x"]), to_device(i["weight"]), eps=rms.eps)), i)

    q = wl.QUANTIZE_F32_4096x65536.with_rows(3)
    i = q.generate()
    codes, scales = credit.quantize(to_device(i["x"]))
    check_quant((codes.cpu().numpy(), scales.cpu().numpy()), i)

    ws = wl.WEIGHTED_STD_F32_4096x65536.with_rows(3)
    i = ws.generate()
    check(ws, to_host(credit.weighted_std(to_device(i["x"]), to_device(i["weight"]), eps=ws.eps)), i)

    pe = wl.PEARSON_F32_4096x65536.with_rows(3)
    i = pe.generate()
    y, r = credit.pearson(to_device(i["x"]), to_device(i["u"]), eps=pe.eps)
    check_pearson(pe, (to_host(y), r.cpu().numpy()), i)
    assert credit.device_error() == 0


def test_torch_layer_rejects_bad_tensors():
    x = torch.zeros(4, 64, device="cuda")
    with pytest.raises(ValueError):
        credit.softmax(x.t())                      # not contiguous
    with pytest.raises(ValueError):
        credit.layernorm(x, torch.ones(63, device="cuda"))
    with pytest.raises(ValueError):
        credit.pearson(x, torch.zeros(4, 32, device="cuda"))
    with pytest.raises(TypeError):
        credit.softmax(torch.zeros(4, 64, device="cuda", dtype=torch.float16))
