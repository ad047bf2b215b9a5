"""GPU parity of the quantization (bit-exact codes and scales) and weighted
standardization operators: every legal cluster size, 1/2/4 rows per cluster,
the two-pass baseline, the element path, zero rows, and the full-size
workloads on sampled rows."""
import numpy as np
import pytest
import torch

from dsmem_thread_block_gb300 import _credit as C
from dsmem_thread_block_gb300 import workloads as wl

from gpu_helpers import DT, OPS, call, check, check_quant, make_plan, run, to_device, to_host

pytestmark = pytest.mark.gpu


def _plans(w):
    dev = torch.cuda.current_device()
    out = []
    for P in (1, 2, 3, 4, 8, 16):
        for R in (1, 2, 4):
            try:
                out.append(C.credit_plan_with(OPS[w.op], w.rows, w.cols, DT[w.dtype], dev,
                                              C.CLUSTER, P, rows_per_cluster=R))
            except C.CreditError as e:
                assert e.status == C.ERR_NO_LEGAL_PLAN
    out.append(make_plan(w, C.TWO_PASS))
    return out


QUANT = [wl.QUANTIZE_F32_4096x65536.with_rows(5),
         wl.Workload("quantize_bf16_3x131072", wl.QUANTIZE, "bf16", 3, 131072, seed=60, x_std=3.0),
         wl.Workload("quantize_f32_4x4104", wl.QUANTIZE, "f32", 4, 4104, seed=61),  # element path
         wl.Workload("quantize_bf16_2x1000", wl.QUANTIZE, "bf16", 2, 1000, seed=62)]


@pytest.mark.parametrize("w", QUANT, ids=[w.name for w in QUANT])
def test_quantize_bit_exact(w):
    inp = w.generate()
    for p in _plans(w):
        check_quant(run(w, inp, p), inp)


def test_quantize_zero_rows_and_constant_rows():
    w = wl.Workload("quantize_f32_4x8192", wl.QUANTIZE, "f32", 4, 8192, seed=63)
    inp = w.generate()
    inp["x"][1] = 0.0
    inp["x"][2] = -2.5
    for p in _plans(w):
        q, s = run(w, inp, p)
        assert s[1] == 0.0 and (q[1] == 0).all()
        assert (q[2] == -127).all()
        check_quant((q, s), inp)


def _near_half_row(amax, cols, rng):
    """A row whose maximum is `amax` and whose other entries sit on and next
    to the products b * s for half-integers b (s = amax / 127 in IEEE
    single): the values where rounding x / s to an integer is decided by the
    last bit of the quotient."""
    f32 = np.float32
    s = f32(f32(amax) / f32(127.0))
    vals = [f32(amax)]
    for b in np.arange(-126, 127) + 0.5:
        v = f32(f32(b) * s)
        vals.append(v)
        up = dn = v
        for _ in range(3):
            up = np.nextafter(up, f32(np.inf))
            dn = np.nextafter(dn, f32(-np.inf))
            vals += [up, dn]
    row = np.array(vals, np.float32)
    row = row[np.abs(row) <= f32(amax)]
    out = rng.uniform(-amax, amax, cols).astype(np.float32)
    out[:len(row)] = row[:cols]
    return out


def test_quantize_codes_decided_by_the_last_quotient_bit():
    # every near-half-integer quotient must round exactly as the IEEE
    # division does (including ties to even at s = 1), on both kernel arms
    rng = np.random.default_rng(65)
    amaxes = [1.0, 3.7, 127.0, 1e-20, 2.5e30, 0.01, 1e-30, 6.1e-34]
    x = np.stack([_near_half_row(a, 2048, rng) for a in amaxes])
    w = wl.Workload("quantize_f32_8x2048_near_half", wl.QUANTIZE, "f32", len(amaxes), 2048, seed=66)
    inp = {"x": x}
    for p in _plans(w):
        check_quant(run(w, inp, p), inp)


def test_quantize_more_rows_than_one_launch_grid():
    # the two-pass grid holds 65535 rows: later batches offset the int8 codes
    # by one byte per element and the scales by one per row
    w = wl.Workload("quantize_f32_70000x16", wl.QUANTIZE, "f32", 70000, 16, seed=64)
    inp = w.generate()
    check_quant(run(w, inp, make_plan(w, C.TWO_PASS)), inp)
    check_quant(run(w, inp, make_plan(w, C.CLUSTER, 1)), inp)


def test_quantize_rejects_overlap():
    x = torch.zeros(4, 4096, device="cuda")
    s = torch.zeros(4, device="cuda")
    # codes written over the input
    assert C.credit_quantize(x.data_ptr(), x.data_ptr(), s.data_ptr(), 4, 4096, C.F32) == \
        C.ERR_INVALID_ARG
    # scales inside the input
    q = torch.zeros(4, 4096, dtype=torch.int8, device="cuda")
    assert C.credit_quantize(x.data_ptr(), q.data_ptr(), x.data_ptr() + 64, 4, 4096, C.F32) == \
        C.ERR_INVALID_ARG
    assert C.credit_quantize(x.data_ptr(), q.data_ptr(), 0, 4, 4096, C.F32) == C.ERR_INVALID_ARG


WSTD = [wl.WEIGHTED_STD_F32_4096x65536.with_rows(5),
        wl.Workload("weighted_std_bf16_3x262144", wl.WEIGHTED_STD, "bf16", 3, 262144, seed=64,
                    x_mean=-1.0, x_std=0.5, eps=1e-5, param_dtype="bf16", p_uniform=True),
        wl.Workload("weighted_std_f32_3x5003", wl.WEIGHTED_STD, "f32", 3, 5003, seed=65,
                    eps=1e-5, param_dtype="f32", p_uniform=True)]  # element path


@pytest.mark.parametrize("w", WSTD, ids=[w.name for w in WSTD])
def test_weighted_std_parity(w):
    inp = w.generate()
    for p in _plans(w):
        check(w, run(w, inp, p), inp)
    check(w, run(w, inp, make_plan(w, C.CLUSTER, 4), in_place=True), inp)


def test_weighted_std_requires_weights():
    x = torch.zeros(2, 4096, device="cuda")
    assert C.credit_weighted_std(x.data_ptr(), x.data_ptr(), 2, 4096, C.F32, 0, C.F32, 1e-5) == \
        C.ERR_INVALID_ARG


@pytest.mark.parametrize("w", [wl.QUANTIZE_F32_4096x65536, wl.WEIGHTED_STD_F32_4096x65536],
                         ids=["quantize", "weighted_std"])
def test_full_size_sampled_rows(w):
    inp = w.generate()
    p = make_plan(w)
    rng = np.random.default_rng(7)
    rows = sorted({0, w.rows - 1, *rng.integers(0, w.rows, 6).tolist()})
    if w.op == wl.QUANTIZE:
        q, s = run(w, inp, p)
        sub = {"x": inp["x"][rows]}
        check_quant((q[rows], s[rows]), sub)
    else:
        got = run(w, inp, p)
        sub = dict(inp)
        sub["x"] = inp["x"][rows]
        check(w, got[rows], sub)


@pytest.mark.parametrize("variant,P", [(C.CLUSTER, 1), (C.CLUSTER, 4), (C.TWO_PASS, 1)])
def test_quantize_misaligned_codes(variant, P):
    # int8 codes starting one byte past a 16-byte boundary: the element path
    w = wl.Workload("quantize_f32_3x8192", wl.QUANTIZE, "f32", 3, 8192, seed=67)
    inp = w.generate()
    dev = torch.cuda.current_device()
    dx = to_device(inp["x"])
    dq = torch.empty(dx.numel() + 1, dtype=torch.int8, device="cuda")[1:]
    s = torch.empty(w.rows, device="cuda")
    p = C.credit_plan_for(C.QUANTIZE, w.rows, w.cols, C.F32, dev, variant, P)
    ws = torch.empty(max(1, int(p.workspace_bytes)), dtype=torch.uint8, device="cuda")
    assert C.credit_quantize(dx.data_ptr(), dq.data_ptr(), s.data_ptr(), w.rows, w.cols, C.F32, p,
                             ws.data_ptr(), int(p.workspace_bytes)) == C.OK
    torch.cuda.synchronize()
    check_quant((dq.cpu().numpy().reshape(w.rows, w.cols), s.cpu().numpy()), inp)
