"""The C ABI library builds, loads and exports every symbol include/credit.h
declares, and its host-side argument checks behave (no GPU needed: nothing
here launches a kernel)."""
import ctypes
import os
import re
import subprocess

import pytest

from dsmem_thread_block_gb300 import _credit as C
from dsmem_thread_block_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        text = open(os.path.join(inc, f)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(credit_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    B.build()
    return C.load()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "credit_softmax" in names and "credit_plan" in names
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (credit_[a-z0-9_]+)\b", out))
    missing = [n for n in names if n not in exported]
    assert not missing, f"declared but not exported: {missing}"
    for n in names:
        getattr(lib, n)


def test_binding_covers_the_abi(lib):
    for n in declared_functions():
        assert n in C.SIGNATURES, f"{n} has no ctypes signature"


def test_plan_struct_layout_matches_header():
    # int32 x4, int64 x3, int32 x6, float x2 -> 72 bytes, no padding surprises
    assert ctypes.sizeof(C.Plan) == 80
    assert C.Plan.smem_bytes.offset == 16 and C.Plan.pred_us.offset == 64
    assert C.Plan.exchange.offset == 60


def test_struct_mirrors_match_the_header(tmp_path):
    # sizes and field offsets of the plan, candidate and report structs as
    # the C compiler lays them out from include/credit.h, against the ctypes
    # mirrors the binding passes to the library
    src = tmp_path / "layout.c"
    src.write_text("""
#include <stddef.h>
#include <stdio.h>
#include "credit.h"
int main(void) {
    printf("%zu %zu %zu %zu %zu %zu %zu\\n", sizeof(credit_plan_t), sizeof(credit_candidate_t),
           sizeof(credit_model_report_t), offsetof(credit_candidate_t, persistent_us),
           offsetof(credit_candidate_t, pipelined_us), offsetof(credit_model_report_t, cand),
           sizeof(credit_host_call_t));
    return 0;
}
""")
    exe = tmp_path / "layout"
    cuda_inc = "/usr/local/cuda/include"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), "-I", cuda_inc, str(src), "-o",
                    str(exe)], check=True)
    got = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    assert got == [ctypes.sizeof(C.Plan), ctypes.sizeof(C.Candidate),
                   ctypes.sizeof(C.ModelReport), C.Candidate.persistent_us.offset,
                   C.Candidate.pipelined_us.offset, C.ModelReport.cand.offset,
                   ctypes.sizeof(C.HostCall)]


def test_status_strings(lib):
    for s in range(8):
        assert C.status_string(s) != "unknown status"
    assert C.status_string(C.ERR_NO_LEGAL_PLAN).startswith("no legal plan")
    assert C.credit_version() == "0.5.0"


def test_host_side_argument_checks_need_no_gpu(lib):
    # null pointers and bad shapes are rejected before any CUDA call
    assert C.credit_softmax(0, 0, 4, 4, C.F32) == C.ERR_INVALID_ARG
    assert C.credit_softmax(16, 32, 0, 4, C.F32) == C.ERR_INVALID_ARG
    assert C.credit_softmax(16, 32, 4, 0, C.F32) == C.ERR_INVALID_ARG
    assert C.credit_softmax(16, 32, 4, 4, 7) == C.ERR_UNSUPPORTED
    assert C.credit_layernorm(16, 1024, 1, 4, C.F32, 0, 0, C.F32, -1.0) == C.ERR_INVALID_ARG
    # partial overlap of x and y (in place x == y is allowed)
    assert C.credit_rmsnorm(4096, 4100, 1, 64, C.F32, 0, C.F32, 1e-6) == C.ERR_INVALID_ARG
    assert lib.credit_plan(C.SOFTMAX, 4, 4, C.F32, 0, None) == C.ERR_INVALID_ARG
    assert lib.credit_plan_for(C.SOFTMAX, 4, 4, C.F32, 0, 9, 1, None) == C.ERR_INVALID_ARG
    # exchanges exist only for the clustered kernels
    out = C.Plan()
    for variant, exchange in ((C.TWO_PASS, C.EXCHANGE_ASYNC), (C.TWO_PASS, C.EXCHANGE_BARRIER),
                              (C.CLUSTER_PERSISTENT, 3), (C.CLUSTER, 3), (C.CLUSTER, -1),
                              (C.WARP_ROWS, C.EXCHANGE_ASYNC), (C.WARP_ROWS, C.EXCHANGE_BARRIER),
                              # the warp-specialised kernel exchanges with st.async only
                              (C.CLUSTER_PIPELINED, C.EXCHANGE_BARRIER)):
        req = C.Plan(variant=variant, cluster_size=2, exchange=exchange)
        assert lib.credit_plan_with(C.SOFTMAX, 4, 4, C.F32, 0, ctypes.byref(req),
                                    ctypes.byref(out)) == C.ERR_INVALID_ARG
    # unknown variants, in a request and in a forced plan
    for variant in (C.AUTO, 6, -1):
        req = C.Plan(variant=variant, cluster_size=2)
        assert lib.credit_plan_with(C.SOFTMAX, 4, 4, C.F32, 0, ctypes.byref(req),
                                    ctypes.byref(out)) == C.ERR_INVALID_ARG
        assert lib.credit_plan_for(C.SOFTMAX, 4, 4, C.F32, 0, variant, 2,
                                   ctypes.byref(out)) == C.ERR_INVALID_ARG


def test_library_fails_loudly_when_missing(monkeypatch, tmp_path):
    monkeypatch.setattr(B, "LIB", str(tmp_path / "nope.so"))
    monkeypatch.setattr(C, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        C.load()


def test_host_buffer_layout_needs_no_gpu(lib):
    # two slots of (x, y) rounded to 256 bytes; Pearson adds u and r, and
    # quantization's output is int8 plus a scale per row
    ln = C.host_call(C.LAYERNORM, C.BF16, 1000, 4096, x=16, y=32)
    assert C.credit_host_buffer_bytes(ln, None, 128) == 2 * (2 * 128 * 4096 * 2)
    pe = C.host_call(C.PEARSON, C.F32, 1000, 100, x=16, y=32, u=48, row_out=64)
    slot = 3 * (((10 * 100 * 4) + 255) // 256 * 256) + ((10 * 4 + 255) // 256 * 256)
    assert C.credit_host_buffer_bytes(pe, None, 10) == 2 * slot
    q = C.host_call(C.QUANTIZE, C.F32, 8, 4096, x=16, y=32, row_out=64)
    assert C.credit_host_buffer_bytes(q, None, 8) == 2 * (8 * 4096 * 4 + 8 * 4096 + 256)
    # argument checks before any CUDA call
    plan = C.Plan(variant=C.CLUSTER, cluster_size=1)
    assert C.credit_run_host(ln, None, 4096, 1 << 30, 128) == C.ERR_INVALID_ARG   # no plan
    assert C.credit_run_host(ln, plan, 4096, 1024, 128) == C.ERR_INVALID_ARG      # short buffer
    assert C.credit_run_host(ln, plan, 4096 + 16, 1 << 30, 128) == C.ERR_INVALID_ARG  # unaligned
    assert C.credit_run_host(ln, plan, 4096, 1 << 30, 0) == C.ERR_INVALID_ARG     # no chunk
    assert C.credit_run_host(C.host_call(C.PEARSON, C.F32, 4, 8, x=16, y=32, row_out=64), plan,
                             4096, 1 << 30, 4) == C.ERR_INVALID_ARG                # no u


def test_checked_build_exports_the_same_abi_and_reports_itself(lib):
    # the checked build (-DCREDIT_DEBUG) carries every declared symbol; the
    # debug entry points answer without a GPU: which build this is, and
    # UNSUPPORTED / INVALID_ARG before any CUDA call
    path = B.build(checked=True)
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT (credit_[a-z0-9_]+)\b", out))
    assert not [n for n in declared_functions() if n not in exported]
    chk = C._open(path)
    assert chk.credit_debug_build() == 1
    assert lib.credit_debug_build() == 0
    assert lib.credit_selftest_bounds(0) == C.ERR_UNSUPPORTED
    assert lib.credit_debug_trace(None, 1) == C.ERR_UNSUPPORTED
    assert chk.credit_debug_trace(None, 1) == C.ERR_INVALID_ARG
    assert chk.credit_debug_trace(None, C.TRACE_CTAS + 1) == C.ERR_INVALID_ARG
    assert C.status_string(C.ERR_DEVICE_BOUNDS).startswith("a device index check failed")
