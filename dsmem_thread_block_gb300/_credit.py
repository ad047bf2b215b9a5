"""ctypes binding of libcredit.so -- argument marshalling only.

The functions here carry the C ABI's names and arguments (include/credit.h):
raw device pointers as ints, sizes, dtype codes, a ``Plan`` structure and a
stream handle.  Every step of the computation runs in the library's CUDA
kernels; if the library is missing this module raises instead of falling
back to anything else.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_NO_LEGAL_PLAN, ERR_CUDA, \
    ERR_DEVICE_TIMEOUT, ERR_NOT_CALIBRATED, ERR_DEVICE_BOUNDS = range(8)
TRACE_CTAS = 8192  # CREDIT_TRACE_CTAS
F32, BF16 = 0, 1
SOFTMAX, LAYERNORM, RMSNORM, QUANTIZE, WEIGHTED_STD, PEARSON = 0, 1, 2, 3, 4, 5
AUTO, CLUSTER, TWO_PASS, CLUSTER_PERSISTENT, CLUSTER_PIPELINED, WARP_ROWS = 0, 1, 2, 3, 4, 5
EXCHANGE_DEFAULT, EXCHANGE_BARRIER, EXCHANGE_ASYNC = 0, 1, 2

_vp, _i64, _i32, _f32, _sz = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                              ctypes.c_float, ctypes.c_size_t)


class Plan(ctypes.Structure):
    """Mirror of credit_plan_t."""
    _fields_ = [("variant", ctypes.c_int32), ("cluster_size", ctypes.c_int32),
                ("threads", ctypes.c_int32), ("waves", ctypes.c_int32),
                ("smem_bytes", ctypes.c_int64), ("workspace_bytes", ctypes.c_int64),
                ("slice_elems", ctypes.c_int64), ("active_clusters", ctypes.c_int32),
                ("ctas_per_sm", ctypes.c_int32), ("chunk_elems", ctypes.c_int32),
                ("ring_slots", ctypes.c_int32), ("rows_per_cluster", ctypes.c_int32),
                ("exchange", ctypes.c_int32), ("pred_us", ctypes.c_float),
                ("pred_two_pass_us", ctypes.c_float), ("staged_elems", ctypes.c_int64)]

    def as_dict(self) -> dict:
        return {f: getattr(self, f) for f, _ in self._fields_}

    def __repr__(self):
        return f"Plan({self.as_dict()})"


class BenchResult(ctypes.Structure):
    """Mirror of credit_bench_result_t."""
    _fields_ = [("kind", ctypes.c_int32), ("cluster_size", ctypes.c_int32),
                ("runs", ctypes.c_int32), ("smids", ctypes.c_int32 * 16),
                ("median_cycles", ctypes.c_double), ("median_ns", ctypes.c_double),
                ("iqr_cycles", ctypes.c_double), ("bytes_per_cycle", ctypes.c_double),
                ("gbps", ctypes.c_double)]

    def as_dict(self) -> dict:
        d = {f: getattr(self, f) for f, _ in self._fields_ if f != "smids"}
        d["smids"] = list(self.smids)[: self.cluster_size]
        return d


class Candidate(ctypes.Structure):
    """Mirror of credit_candidate_t."""
    _fields_ = [("cluster_size", ctypes.c_int32), ("legal", ctypes.c_int32), ("plan", Plan),
                ("t_ctrl_us", ctypes.c_double), ("t_comm_us", ctypes.c_double),
                ("pred_us", ctypes.c_double), ("measured_us", ctypes.c_double),
                ("persistent_us", ctypes.c_double),
                ("pipelined_us", ctypes.c_double), ("tail_us", ctypes.c_double),
                ("tail_staged_elems", ctypes.c_int64)]


class DeviceKey(ctypes.Structure):
    """Mirror of credit_device_key_t."""
    _fields_ = [("gpu_name", ctypes.c_char * 96), ("sms", ctypes.c_int32),
                ("sm_clock_mhz", ctypes.c_int32), ("mem_clock_mhz", ctypes.c_int32),
                ("cc_major", ctypes.c_int32), ("cc_minor", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class HostCall(ctypes.Structure):
    """Mirror of credit_host_call_t."""
    _fields_ = [("op", ctypes.c_int32), ("dtype", ctypes.c_int32), ("rows", ctypes.c_int64),
                ("cols", ctypes.c_int64), ("x", ctypes.c_void_p), ("u", ctypes.c_void_p),
                ("y", ctypes.c_void_p), ("row_out", ctypes.c_void_p), ("p0", ctypes.c_void_p),
                ("p1", ctypes.c_void_p), ("param_dtype", ctypes.c_int32), ("eps", ctypes.c_float)]


class ModelReport(ctypes.Structure):
    """Mirror of credit_model_report_t."""
    _fields_ = [("baseline_variant", ctypes.c_int32), ("model_cluster_size", ctypes.c_int32),
                ("profitable", ctypes.c_int32), ("chosen_cluster_size", ctypes.c_int32),
                ("chosen_variant", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("t_base_us", ctypes.c_double), ("b_base_bytes", ctypes.c_double),
                ("b_credit_bytes", ctypes.c_double), ("t_ctrl_base_us", ctypes.c_double),
                ("cand", Candidate * 16)]

    def as_dict(self) -> dict:
        d = {f: getattr(self, f) for f, _ in self._fields_ if f not in ("cand", "reserved")}
        d["candidates"] = [{"P": c.cluster_size, "t_ctrl_us": c.t_ctrl_us, "t_comm_us": c.t_comm_us,
                            "pred_us": c.pred_us, "measured_us": c.measured_us,
                            "persistent_us": c.persistent_us, "pipelined_us": c.pipelined_us,
                            "plan": c.plan.as_dict()}
                           for c in self.cand if c.legal]
        return d


BENCH_BARRIER, BENCH_EXCHANGE, BENCH_REMOTE_LOAD_LATENCY, BENCH_LOCAL_LOAD_LATENCY, \
    BENCH_REMOTE_STORE_BW, BENCH_REMOTE_LOAD_BW, BENCH_LOCAL_STORE_BW, \
    BENCH_LOCAL_LOAD_BW, BENCH_ASYNC_EXCHANGE = range(9)


class CreditError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


# C signatures: name -> (restype, argtypes)
SIGNATURES = {
    "credit_plan": (_i32, [_i32, _i64, _i64, _i32, _i32, ctypes.POINTER(Plan)]),
    "credit_plan_for": (_i32, [_i32, _i64, _i64, _i32, _i32, _i32, _i32, ctypes.POINTER(Plan)]),
    "credit_plan_with": (_i32, [_i32, _i64, _i64, _i32, _i32, ctypes.POINTER(Plan),
                                ctypes.POINTER(Plan)]),
    "credit_softmax": (_i32, [_vp, _vp, _i64, _i64, _i32, ctypes.POINTER(Plan), _vp, _sz, _vp]),
    "credit_layernorm": (_i32, [_vp, _vp, _i64, _i64, _i32, _vp, _vp, _i32, _f32,
                                ctypes.POINTER(Plan), _vp, _sz, _vp]),
    "credit_rmsnorm": (_i32, [_vp, _vp, _i64, _i64, _i32, _vp, _i32, _f32,
                              ctypes.POINTER(Plan), _vp, _sz, _vp]),
    "credit_quantize": (_i32, [_vp, _vp, _vp, _i64, _i64, _i32, ctypes.POINTER(Plan), _vp, _sz,
                               _vp]),
    "credit_weighted_std": (_i32, [_vp, _vp, _i64, _i64, _i32, _vp, _i32, _f32,
                                   ctypes.POINTER(Plan), _vp, _sz, _vp]),
    "credit_pearson": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i32, _f32, ctypes.POINTER(Plan),
                              _vp, _sz, _vp]),
    "credit_two_pass_noalloc": (_i32, [_i32, _vp, _vp, _i64, _i64, _i32, _vp, _vp, _i32, _f32,
                                       _vp]),
    "credit_bench_dsmem": (_i32, [_i32, _i32, _i32, _i32, _i32, ctypes.POINTER(BenchResult)]),
    "credit_control_time": (_i32, [_i32, _i64, _i32, _i32, _i64, _i32, _i32, _i32,
                                   ctypes.POINTER(ctypes.c_double)]),
    "credit_calibrate": (_i32, [_i32, _i32, ctypes.c_char_p]),
    "credit_plan_profiled": (_i32, [_i32, _i64, _i64, _i32, _i32, _i32, _i32, _i32,
                                    ctypes.POINTER(Plan), ctypes.POINTER(ModelReport)]),
    "credit_status_string": (ctypes.c_char_p, [_i32]),
    "credit_l2_read_rate": (_i32, [_i32, _i64, _i32, ctypes.POINTER(ctypes.c_double)]),
    "credit_device_key": (_i32, [_i32, ctypes.POINTER(DeviceKey)]),
    "credit_plan_tail": (_i32, [_i32, _i64, _i64, _i32, _i32, _i32, _i32, ctypes.POINTER(Plan)]),
    "credit_save_profile": (_i32, [_i32, ctypes.c_char_p]),
    "credit_load_profile": (_i32, [_i32, ctypes.c_char_p]),
    "credit_profile_check": (_i32, [ctypes.c_char_p, ctypes.POINTER(DeviceKey)]),
    "credit_stage_copy_rate": (_i32, [_i32, _i32, _i32, ctypes.POINTER(ctypes.c_double),
                                      ctypes.POINTER(ctypes.c_int32)]),
    "credit_host_buffer_bytes": (_i32, [ctypes.POINTER(HostCall), ctypes.POINTER(Plan), _i64,
                                        ctypes.POINTER(ctypes.c_size_t)]),
    "credit_run_host": (_i32, [ctypes.POINTER(HostCall), ctypes.POINTER(Plan), _vp, _sz, _i64,
                               _vp]),
    "credit_get_device_error": (_i32, [_i32]),
    "credit_selftest_wait_timeout": (_i32, [_i32, _i64]),
    "credit_debug_build": (_i32, []),
    "credit_selftest_bounds": (_i32, [_i32]),
    "credit_debug_trace": (_i32, [_vp, _i64]),
    "credit_debug_stats": (_i32, [_vp, _i64]),
    "credit_version": (ctypes.c_char_p, []),
}

_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def _open(path: str) -> ctypes.CDLL:
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(lib, name)
        f.restype, f.argtypes = res, args
    return lib


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libcredit.so (building it first only if asked)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if not os.path.exists(path):
                if not build_if_missing:
                    raise RuntimeError(
                        f"libcredit.so is not built ({path}); run "
                        "`python -c 'import __graft_entry__ as g; g.build()'`")
                _build.build()
            _lib = _open(path)
    return _lib


class use_checked_build:
    """Context manager: route every call of this module to the checked
    build (libcredit_checked.so: index checks and the phase trace) and back
    to the regular library on exit."""

    def __enter__(self):
        global _lib
        path = _build.CHECKED_LIB
        if not os.path.exists(path):
            raise RuntimeError(f"the checked build is missing ({path}); run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        with _lock:
            self._saved = _lib
            _lib = _open(path)
        return _lib

    def __exit__(self, *exc):
        global _lib
        with _lock:
            _lib = self._saved
        return False


def status_string(status: int) -> str:
    try:
        return load().credit_status_string(status).decode()
    except Exception:  # library not loadable: still give a readable message
        return f"status {status}"


def _check(status: int, where: str) -> None:
    if status != OK:
        raise CreditError(status, where)


def _plan_ptr(plan):
    return None if plan is None else ctypes.byref(plan)


def credit_plan(op: int, rows: int, cols: int, dtype: int, device: int) -> Plan:
    p = Plan()
    _check(load().credit_plan(op, rows, cols, dtype, device, ctypes.byref(p)), "credit_plan")
    return p


def credit_plan_for(op: int, rows: int, cols: int, dtype: int, device: int,
                    variant: int, cluster_size: int = 1) -> Plan:
    p = Plan()
    _check(load().credit_plan_for(op, rows, cols, dtype, device, variant, cluster_size,
                                  ctypes.byref(p)), "credit_plan_for")
    return p


def credit_plan_tail(op: int, rows: int, cols: int, dtype: int, device: int, cluster_size: int,
                     ctas_per_sm: int) -> Plan:
    """The L2-tail plan of cluster size P whose staged part lets ctas_per_sm
    CTAs share an SM (raises ERR_NO_LEGAL_PLAN where there is none)."""
    p = Plan()
    _check(load().credit_plan_tail(op, rows, cols, dtype, device, cluster_size, ctas_per_sm,
                                   ctypes.byref(p)), "credit_plan_tail")
    return p


def credit_plan_with(op: int, rows: int, cols: int, dtype: int, device: int, variant: int,
                     cluster_size: int = 1, threads: int = 0, ctas_per_sm: int = 0,
                     chunk_elems: int = 0, rows_per_cluster: int = 0,
                     exchange: int = EXCHANGE_DEFAULT, staged_elems: int = 0) -> Plan:
    req = Plan(variant=variant, cluster_size=cluster_size, threads=threads,
               ctas_per_sm=ctas_per_sm, chunk_elems=chunk_elems,
               rows_per_cluster=rows_per_cluster, exchange=exchange,
               staged_elems=staged_elems)
    p = Plan()
    _check(load().credit_plan_with(op, rows, cols, dtype, device, ctypes.byref(req),
                                   ctypes.byref(p)), "credit_plan_with")
    return p


def credit_softmax(x: int, y: int, rows: int, cols: int, dtype: int, plan=None,
                   workspace: int = 0, workspace_bytes: int = 0, stream: int = 0) -> int:
    return load().credit_softmax(x, y, rows, cols, dtype, _plan_ptr(plan), workspace or None,
                                 workspace_bytes, stream or None)


def credit_layernorm(x: int, y: int, rows: int, cols: int, dtype: int, gamma: int, beta: int,
                     param_dtype: int, eps: float, plan=None, workspace: int = 0,
                     workspace_bytes: int = 0, stream: int = 0) -> int:
    return load().credit_layernorm(x, y, rows, cols, dtype, gamma or None, beta or None,
                                   param_dtype, eps, _plan_ptr(plan), workspace or None,
                                   workspace_bytes, stream or None)


def credit_rmsnorm(x: int, y: int, rows: int, cols: int, dtype: int, weight: int,
                   param_dtype: int, eps: float, plan=None, workspace: int = 0,
                   workspace_bytes: int = 0, stream: int = 0) -> int:
    return load().credit_rmsnorm(x, y, rows, cols, dtype, weight or None, param_dtype, eps,
                                 _plan_ptr(plan), workspace or None, workspace_bytes,
                                 stream or None)


def credit_quantize(x: int, q: int, scales: int, rows: int, cols: int, dtype: int, plan=None,
                    workspace: int = 0, workspace_bytes: int = 0, stream: int = 0) -> int:
    return load().credit_quantize(x, q, scales, rows, cols, dtype, _plan_ptr(plan),
                                  workspace or None, workspace_bytes, stream or None)


def credit_weighted_std(x: int, y: int, rows: int, cols: int, dtype: int, weights: int,
                        weight_dtype: int, eps: float, plan=None, workspace: int = 0,
                        workspace_bytes: int = 0, stream: int = 0) -> int:
    return load().credit_weighted_std(x, y, rows, cols, dtype, weights or None, weight_dtype,
                                      eps, _plan_ptr(plan), workspace or None, workspace_bytes,
                                      stream or None)


def credit_pearson(x: int, u: int, y: int, r: int, rows: int, cols: int, dtype: int,
                   eps: float, plan=None, workspace: int = 0, workspace_bytes: int = 0,
                   stream: int = 0) -> int:
    return load().credit_pearson(x or None, u or None, y or None, r or None, rows, cols, dtype,
                                 eps, _plan_ptr(plan), workspace or None, workspace_bytes,
                                 stream or None)


def credit_two_pass_noalloc(op: int, x: int, y: int, rows: int, cols: int, dtype: int,
                            p0: int = 0, p1: int = 0, param_dtype: int = F32, eps: float = 0.0,
                            stream: int = 0) -> int:
    """Two-pass call for callers that cannot allocate device memory: the
    partials live in the library's own fixed 2 MiB device array."""
    return load().credit_two_pass_noalloc(op, x, y, rows, cols, dtype, p0 or None, p1 or None,
                                          param_dtype, eps, stream or None)


def credit_bench_dsmem(device: int, kind: int, cluster_size: int = 2, iters: int = 1000,
                       runs: int = 15) -> BenchResult:
    r = BenchResult()
    _check(load().credit_bench_dsmem(device, kind, cluster_size, iters, runs, ctypes.byref(r)),
           "credit_bench_dsmem")
    return r


def credit_control_time(device: int, nclusters: int, cluster_size: int, threads: int,
                        smem_bytes: int, rows_per_cluster: int, barriers_per_row: int,
                        runs: int = 15) -> float:
    t = ctypes.c_double()
    _check(load().credit_control_time(device, nclusters, cluster_size, threads, smem_bytes,
                                      rows_per_cluster, barriers_per_row, runs, ctypes.byref(t)),
           "credit_control_time")
    return t.value


def credit_calibrate(device: int = 0, runs: int = 7, profile_path: str | None = None) -> None:
    _check(load().credit_calibrate(device, runs, profile_path.encode() if profile_path else None),
           "credit_calibrate")


def credit_plan_profiled(op: int, rows: int, cols: int, dtype: int, param_dtype: int = -1,
                         device: int = 0, runs: int = 7, tune: int = 0):
    p, r = Plan(), ModelReport()
    _check(load().credit_plan_profiled(op, rows, cols, dtype, param_dtype, device, runs, tune,
                                       ctypes.byref(p), ctypes.byref(r)), "credit_plan_profiled")
    return p, r


def variant_name(plan) -> str:
    """Short name of a plan's kernel and cluster size, as the benchmark
    prints it: cluster:P[xR][:sSTAGED][:tTHREADS][:barrier], persist:P,
    pipe:P, warp_rows, two_pass (sSTAGED: an L2-tail plan staging STAGED
    elements per CTA; tTHREADS: an L2-tail plan with other than 256 threads
    per CTA)."""
    if plan.variant == TWO_PASS:
        return "two_pass"
    if plan.variant == WARP_ROWS:
        return "warp_rows"
    kind = {CLUSTER: "cluster", CLUSTER_PERSISTENT: "persist", CLUSTER_PIPELINED: "pipe"}[plan.variant]
    s = f"{kind}:{plan.cluster_size}"
    if plan.variant == CLUSTER and plan.rows_per_cluster > 1:
        s += f"x{plan.rows_per_cluster}"
    if plan.variant == CLUSTER and 0 < plan.staged_elems < plan.slice_elems:
        s += f":s{plan.staged_elems}"
        if plan.threads != 256:
            s += f":t{plan.threads}"
    if plan.variant == CLUSTER and plan.exchange == EXCHANGE_BARRIER:
        s += ":barrier"
    return s


TUNE_RUNS = 15  # timed runs per candidate
TUNE_ALL = 16   # best-predicted candidates to time: every legal cluster size


def tuned_plan(op: int, rows: int, cols: int, dtype: int, param_dtype: int = -1,
               device: int = 0):
    """The plan the benchmark times for a shape: credit_plan_profiled with
    every legal candidate timed; (plan, report)."""
    return credit_plan_profiled(op, rows, cols, dtype, param_dtype, device, TUNE_RUNS, TUNE_ALL)


def credit_device_key(device: int = 0) -> DeviceKey:
    k = DeviceKey()
    _check(load().credit_device_key(device, ctypes.byref(k)), "credit_device_key")
    return k


def credit_save_profile(device: int, path: str) -> int:
    return load().credit_save_profile(device, path.encode())


def credit_load_profile(device: int, path: str) -> int:
    """Status: OK, ERR_NOT_CALIBRATED (stale profile) or ERR_INVALID_ARG."""
    return load().credit_load_profile(device, path.encode())


def credit_profile_check(path: str, key: DeviceKey) -> int:
    """Status: OK, ERR_NOT_CALIBRATED (stale for `key`) or ERR_INVALID_ARG."""
    return load().credit_profile_check(path.encode(), ctypes.byref(key))


def credit_l2_read_rate(device: int, window_bytes: int, runs: int = 7) -> float:
    """GB/s at which all SMs read a window of `window_bytes` from L2."""
    g = ctypes.c_double()
    _check(load().credit_l2_read_rate(device, window_bytes, runs, ctypes.byref(g)),
           "credit_l2_read_rate")
    return g.value


def credit_stage_copy_rate(device: int, ctas_per_sm: int, runs: int = 7):
    """(GB/s, resident CTAs per SM) of the staged-copy primitive."""
    g, k = ctypes.c_double(), ctypes.c_int32()
    _check(load().credit_stage_copy_rate(device, ctas_per_sm, runs, ctypes.byref(g),
                                         ctypes.byref(k)), "credit_stage_copy_rate")
    return g.value, k.value


def host_call(op: int, dtype: int, rows: int, cols: int, x: int, y: int, u: int = 0,
              row_out: int = 0, p0: int = 0, p1: int = 0, param_dtype: int = F32,
              eps: float = 0.0) -> HostCall:
    return HostCall(op=op, dtype=dtype, rows=rows, cols=cols, x=x or None, u=u or None,
                    y=y or None, row_out=row_out or None, p0=p0 or None, p1=p1 or None,
                    param_dtype=param_dtype, eps=eps)


def credit_host_buffer_bytes(call: HostCall, plan=None, rows_per_chunk: int = 1) -> int:
    n = ctypes.c_size_t()
    _check(load().credit_host_buffer_bytes(ctypes.byref(call), _plan_ptr(plan), rows_per_chunk,
                                           ctypes.byref(n)), "credit_host_buffer_bytes")
    return n.value


def credit_run_host(call: HostCall, plan, device_buffer: int, device_buffer_bytes: int,
                    rows_per_chunk: int, stream: int = 0) -> int:
    return load().credit_run_host(ctypes.byref(call), _plan_ptr(plan), device_buffer or None,
                                  device_buffer_bytes, rows_per_chunk, stream or None)


def credit_get_device_error(device: int) -> int:
    return load().credit_get_device_error(device)


def credit_selftest_wait_timeout(device: int = 0, limit_ns: int = 2_000_000) -> int:
    return load().credit_selftest_wait_timeout(device, limit_ns)


def credit_debug_build() -> int:
    return load().credit_debug_build()


def credit_selftest_bounds(device: int = 0) -> int:
    return load().credit_selftest_bounds(device)


def credit_debug_trace(ctas: int):
    """The checked build's phase trace of the first `ctas` CTAs: an int64
    array [ctas, 8] (seven %globaltimer stamps in ns, then the SM id)."""
    import numpy as np
    out = np.zeros((ctas, 8), dtype=np.uint64)
    _check(load().credit_debug_trace(out.ctypes.data, ctas), "credit_debug_trace")
    return out.astype(np.int64)


DEBUG_STATS_ROWS = 64


def credit_debug_stats(rows: int = DEBUG_STATS_ROWS):
    """The checked build's record of the combined statistics each CTA rebuilt:
    a float32 array [rows, 16 ranks, 8] (the statistics, then P in the last
    slot; NaN where no CTA wrote).  Reading resets the record."""
    import numpy as np
    out = np.zeros((rows, 16, 8), dtype=np.float32)
    _check(load().credit_debug_stats(out.ctypes.data, rows), "credit_debug_stats")
    return out


def credit_version() -> str:
    return load().credit_version().decode()
