#!/usr/bin/env python3
"""Benchmark of the clustered DSMEM reduce-reuse path on one GB300.

A step is one library call over the whole workload.  The default workload is
the widest one: bf16 RMSNorm with a bf16 weight, 2048 rows x 786432 columns
(1.5 MiB per row, a slice of 96-192 KiB per CTA for clusters of 8-16),
eps 1e-6, x drawn from N(0, 1) with seed 3.  `value` is the algorithmic HBM
rate of the timed steps: one read plus one write of the matrix, the weight
once, divided by the device time per step (CUDA events on the launching
stream).  The input (3.2 GB) is far larger than the 129 MB L2, so no flush
is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--workload NAME]

Prints ONE JSON line.  Under torchrun (N > 1) every rank runs its own replica
of the workload on its own GPU (rows are independent: weak scaling, no
collective on the data path); the time is the max over ranks.
`--impl reference` times the fp64 CPU oracle on this host's cores instead.
Other workloads (`--workload`) and forced plans (`--variant`) are for local
studies; the default is the headline line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "wide-row reduce-reuse HBM GB/s and % of GB300 peak; DRAM bytes vs 1R+1W ideal"
FALLBACK_HBM_GBS = 6800.0


def _workloads():
    from dsmem_thread_block_gb300 import workloads as wl
    table = {w.name: w for w in wl.ALL}
    for c in wl.SWEEP_COLS:
        w = wl.sweep_point(c)
        table[w.name] = w
    return wl, table


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# The sources that define the kernels and how they are launched (device code,
# launch arguments, plan geometry); the cost model, microbenchmarks, profile
# file and host pipeline do not change what a launch of a given plan moves.
KERNEL_SOURCES = ("api.cu", "cluster.cu", "common.cuh", "internal.h", "pearson.cu",
                  "persistent.cu", "plan.cu", "ptx.cuh", "rowops.cuh", "two_pass.cu",
                  "warp_rows.cu")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dsmem_thread_block_gb300", "csrc")
    for f in KERNEL_SOURCES:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()[:16]


def stored_traffic(workload: str, variant_key: str):
    """Per-launch DRAM bytes from the committed ncu summary, or None if the
    kernels changed since it was taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except Exception:
        return None
    if d.get("kernel_source_hash") != kernel_source_hash():
        return None
    e = d.get("entries", {}).get(f"{workload}|{variant_key}")
    return None if e is None else e.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ clocks
# NVML clock-event reason bits (nvml.h, nvmlClocksEventReason*)
_NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                 0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


class NvmlClockSampler:
    """SM clock, maximum SM clock, power and clock-event reasons, polled every
    `period_ms` through NVML (read-only queries) from a host thread, with
    host timestamps: fine enough for a timed region of a few milliseconds."""

    def __init__(self, uuid: str | None, period_ms: float = 1.0):
        import ctypes
        self.samples = []
        self.error = None
        self._stop = threading.Event()
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                raise RuntimeError("nvmlInit failed")
            h = ctypes.c_void_p()
            if uuid:
                rc = lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h))
            else:
                rc = lib.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(h))
            if rc != 0:
                raise RuntimeError(f"no NVML handle (rc {rc})")
            reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                lib.nvmlDeviceGetCurrentClocksThrottleReasons
        except Exception as e:  # no NVML: the caller falls back to nvidia-smi
            self.error = str(e)
            return
        self.lib, self.h, self.reasons_fn = lib, h, reasons
        self.period = period_ms / 1e3
        self.t = threading.Thread(target=self._poll, daemon=True)
        self.t.start()

    def _poll(self):
        import ctypes
        sm, mx, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            t = time.time()
            ok = (self.lib.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(sm)) == 0 and
                  self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0 and
                  self.reasons_fn(self.h, ctypes.byref(rs)) == 0)
            if ok:
                p = pw.value if self.lib.nvmlDeviceGetPowerUsage(self.h, ctypes.byref(pw)) == 0 else 0
                self.samples.append((t, sm.value, mx.value, rs.value, p / 1e3))
            time.sleep(self.period)

    def stop(self):
        self._stop.set()
        if self.error is None:
            self.t.join(timeout=2)

    def summary(self, t0: float, t1: float) -> dict:
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": "no samples"}
        reasons = sorted({name for s in inside for bit, name in _NVML_REASONS.items()
                          if s[3] & bit})
        return {"sm_mhz": statistics.median(s[1] for s in inside),
                "sm_max_mhz": max(s[2] for s in inside), "reasons": reasons,
                "samples": len(inside), "power_w_max": max(s[4] for s in inside),
                "note": "NVML, polled every ~1 ms during the timed region"}


class ClockSampler:
    """nvidia-smi SM clock and throttle-reason samples, host-timestamped
    (used when NVML cannot be loaded)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_id: str | None, period_ms: int = 50):
        self.samples = []
        self.proc = None
        self.error = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", str(period_ms)]
        if device_id:
            cmd += ["-i", device_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception as e:  # no nvidia-smi
            self.error = str(e)
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        if self.error or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "note": self.error or "no samples"}
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        note = "sampled during the timed region"
        if not inside:  # timed region shorter than the sampling period
            inside = sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:2]
            note = "nearest samples to a short timed region"

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None

        sm = [num(p[0]) for _, p in inside if num(p[0]) is not None]
        mx = [num(p[1]) for _, p in inside if num(p[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, p in inside for i in range(4)
                          if p[4 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside), "note": note}


def clock_sampler(uuid: str | None):
    s = NvmlClockSampler(uuid)
    return s if s.error is None else ClockSampler(uuid)


# ------------------------------------------------------------ CPU oracle
def cpu_oracle_rate(w, inputs, rows: int, threads: int):
    """Time the oracle (as it stands) over the first `rows` rows; return
    (GB/s of algorithmic bytes, seconds)."""
    import oracle
    sub = dict(inputs)
    sub["x"] = inputs["x"][:rows]
    t0 = time.perf_counter()
    if w.op == "quantize":
        bounds = np.linspace(0, rows, min(threads, rows) + 1, dtype=np.int64)
        import concurrent.futures as cf
        with cf.ThreadPoolExecutor(len(bounds) - 1) as ex:
            list(ex.map(lambda i: oracle.quantize(sub["x"][bounds[i]:bounds[i + 1]]),
                        range(len(bounds) - 1)))
    elif w.op == "pearson":
        bounds = np.linspace(0, rows, min(threads, rows) + 1, dtype=np.int64)
        import concurrent.futures as cf
        u = inputs["u"][:rows]
        with cf.ThreadPoolExecutor(len(bounds) - 1) as ex:
            list(ex.map(lambda i: oracle.pearson(sub["x"][bounds[i]:bounds[i + 1]],
                                                 u[bounds[i]:bounds[i + 1]], eps=w.eps),
                        range(len(bounds) - 1)))
    elif w.op == "weighted_std":
        oracle.run_rows(oracle.weighted_std, sub["x"], sub["weight"], threads=threads, eps=w.eps)
    elif w.op == "softmax":
        oracle.run_rows(oracle.softmax, sub["x"], threads=threads)
    elif w.op == "layernorm":
        oracle.run_rows(oracle.layernorm, sub["x"], sub.get("gamma"), sub.get("beta"),
                        threads=threads, eps=w.eps)
    else:
        oracle.run_rows(oracle.rmsnorm, sub["x"], sub.get("weight"), threads=threads, eps=w.eps)
    dt = time.perf_counter() - t0
    return w.with_rows(rows).ideal_bytes() / dt / 1e9, dt


def cpu_sample_rows(w, inputs, threads: int, budget_s: float) -> int:
    """Rows of the workload the oracle finishes in about `budget_s`."""
    _, dt1 = cpu_oracle_rate(w, inputs, min(threads, w.rows), threads)
    per_row = dt1 / min(threads, w.rows) * 1.0
    return int(max(1, min(w.rows, budget_s / max(per_row, 1e-9))))


def run_reference(args, w, rank: int):
    """--impl reference: the fp64 oracle on the host cores, same metric."""
    if rank != 0:
        return
    cores = len(os.sched_getaffinity(0))
    inputs = w.generate()
    total_budget = 90.0
    per_step = total_budget / max(1, args.steps + args.warmup)
    rows = cpu_sample_rows(w, inputs, cores, per_step)
    for _ in range(args.warmup):
        cpu_oracle_rate(w, inputs, rows, cores)
    times = [cpu_oracle_rate(w, inputs, rows, cores)[1] for _ in range(args.steps)]
    tot = sum(times)
    value = w.with_rows(rows).ideal_bytes() * len(times) / tot / 1e9
    sample = f"first {rows} of {w.rows} rows per step (full width {w.cols})"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot / len(times), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "rows": w.rows, "cols": w.cols, "rows_per_step": rows},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------ plans
def parse_variant(spec: str) -> dict:
    """kind:P[xR][:sSTAGED][:tTHREADS] (the plan names variant_name prints)
    -> {kind, P, R, staged, threads}; 0 leaves a field to the planner."""
    kind, rest = spec.split(":", 1)
    if kind not in ("cluster", "persist", "pipe"):
        raise ValueError(f"unknown plan kind in {spec!r}")
    head, *opts = rest.split(":")
    P, R = (head.split("x") + ["0"])[:2] if "x" in head else (head, "0")
    out = {"kind": kind, "P": int(P), "R": int(R), "staged": 0, "threads": 0}
    for q in opts:
        if q.startswith("s"):
            out["staged"] = int(q[1:])
        elif q.startswith("t"):
            out["threads"] = int(q[1:])
        elif q != "barrier":
            raise ValueError(f"unknown plan option {q!r} in {spec!r}")
    return out


# ------------------------------------------------------------ ranks
def max_over_ranks(x: float, world: int, device) -> float:
    """The largest of every rank's `x` (every rank calls this)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(bytes_per_rank_step: float, ms_per_step_max: float, world: int) -> float:
    """Whole-job GB/s: every rank's bytes over the slowest rank's step time
    (replicas: each rank runs the full workload on its own GPU)."""
    return bytes_per_rank_step * world / (ms_per_step_max * 1e-3) / 1e9


# ------------------------------------------------------------------ main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="rmsnorm_bf16_2048x786432")
    ap.add_argument("--variant", default="auto",
                    help="auto (cost model + tuning) | static | cluster:P[xR][:sSTAGED][:tTHREADS] | "
                         "persist:P | pipe:P | warp_rows | two_pass")
    ap.add_argument("--cps", type=int, default=0, help="persistent CTAs per SM (0 = planner)")
    ap.add_argument("--exchange", default="plan", choices=["plan", "barrier", "async"],
                    help="partial exchange of a one-pass clustered plan (plan = as planned)")
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--e2e-chunks", type=int, default=16,
                    help="row chunks of the host-buffer pipeline")
    ap.add_argument("--cpu-budget", type=float, default=20.0,
                    help="seconds of oracle work for the cpu_baseline sample")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--rows", type=int, default=0,
                    help="run the workload's first ROWS rows (0 = all; for profiling captures)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    wl, table = _workloads()
    w = table[args.workload]
    if args.rows:
        w = w.with_rows(args.rows)  # a smaller case of the same shape (profiling)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, w, rank)
        return

    import torch
    import torch.distributed as dist
    from dsmem_thread_block_gb300 import _credit as C

    torch.cuda.set_device(local)
    dev = torch.cuda.current_device()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    C.load(build_if_missing=True)

    inputs = w.generate()
    DT = {"f32": C.F32, "bf16": C.BF16}
    OPS = {"softmax": C.SOFTMAX, "layernorm": C.LAYERNORM, "rmsnorm": C.RMSNORM,
           "quantize": C.QUANTIZE, "weighted_std": C.WEIGHTED_STD, "pearson": C.PEARSON}

    def to_device(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to("cuda")
        return torch.from_numpy(a).to("cuda")
    dx = to_device(inputs["x"])
    quant = w.op == "quantize"
    row_out = quant or w.op == "pearson"  # a per-row fp32 result: scales or r
    dy = torch.empty(dx.shape, dtype=torch.int8, device=dx.device) if quant else torch.empty_like(dx)
    dscales = torch.empty(w.rows, dtype=torch.float32, device=dx.device) if row_out else None
    params = {k: to_device(v) for k, v in inputs.items() if k != "x"}

    tuning = None
    if args.variant == "auto":
        # the cost model screens profitability and ranks the candidates (to
        # within a few percent at the wide end), and the tuning step times
        # every legal candidate; planning and tuning happen once, before
        # (and outside) the timed region
        pdt_model = DT[w.param_dtype] if w.param_dtype else -1
        plan, report = C.tuned_plan(OPS[w.op], w.rows, w.cols, DT[w.dtype], pdt_model, dev)
        tuning = {"model_P": report.model_cluster_size, "baseline_us": round(report.t_base_us, 2)}
        for c in report.cand:
            if c.legal and c.measured_us > 0 and c.cluster_size > 1:
                tuning[C.variant_name(c.plan)] = round(c.measured_us, 2)
            if c.legal and c.tail_us > 0:
                tuning[f"cluster:{c.cluster_size}:s{c.tail_staged_elems}"] = round(c.tail_us, 2)
            if c.legal and c.persistent_us > 0:
                tuning[f"persist:{c.cluster_size}"] = round(c.persistent_us, 2)
            if c.legal and c.pipelined_us > 0:
                tuning[f"pipe:{c.cluster_size}"] = round(c.pipelined_us, 2)
    elif args.variant == "static":
        plan = C.credit_plan(OPS[w.op], w.rows, w.cols, DT[w.dtype], dev)
    elif args.variant == "two_pass":
        plan = C.credit_plan_for(OPS[w.op], w.rows, w.cols, DT[w.dtype], dev, C.TWO_PASS, 1)
    elif args.variant == "warp_rows":
        plan = C.credit_plan_for(OPS[w.op], w.rows, w.cols, DT[w.dtype], dev, C.WARP_ROWS, 1)
    else:
        v = parse_variant(args.variant)
        var = {"cluster": C.CLUSTER, "persist": C.CLUSTER_PERSISTENT,
               "pipe": C.CLUSTER_PIPELINED}[v["kind"]]
        plan = C.credit_plan_with(OPS[w.op], w.rows, w.cols, DT[w.dtype], dev, var, v["P"],
                                  threads=v["threads"], rows_per_cluster=v["R"],
                                  staged_elems=v["staged"])
    if args.cps:
        plan.ctas_per_sm = args.cps
        plan = C.Plan.from_buffer_copy(plan)
    if args.exchange != "plan" and plan.variant == C.CLUSTER:
        plan.exchange = C.EXCHANGE_ASYNC if args.exchange == "async" else C.EXCHANGE_BARRIER
    ws = None
    if plan.workspace_bytes:
        ws = torch.empty(int(plan.workspace_bytes), dtype=torch.uint8, device=dx.device)
    wptr, wbytes = (ws.data_ptr(), int(plan.workspace_bytes)) if ws is not None else (0, 0)
    stream = torch.cuda.Stream()
    sptr = stream.cuda_stream
    pdt = DT[w.param_dtype] if w.param_dtype else C.F32
    lib = C.load()
    pp = C._plan_ptr(plan)

    def launch(xp, yp):
        if quant:
            return lib.credit_quantize(xp, yp, dscales.data_ptr(), w.rows, w.cols, DT[w.dtype], pp,
                                       wptr or None, wbytes, sptr)
        if w.op == "pearson":
            return lib.credit_pearson(xp, params["u"].data_ptr(), yp, dscales.data_ptr(), w.rows,
                                      w.cols, DT[w.dtype], w.eps, pp, wptr or None, wbytes, sptr)
        if w.op == "weighted_std":
            return lib.credit_weighted_std(xp, yp, w.rows, w.cols, DT[w.dtype],
                                           params["weight"].data_ptr(), pdt, w.eps, pp,
                                           wptr or None, wbytes, sptr)
        if w.op == "softmax":
            return lib.credit_softmax(xp, yp, w.rows, w.cols, DT[w.dtype], pp, wptr or None,
                                      wbytes, sptr)
        if w.op == "layernorm":
            g, b = params.get("gamma"), params.get("beta")
            return lib.credit_layernorm(xp, yp, w.rows, w.cols, DT[w.dtype],
                                        g.data_ptr() if g is not None else None,
                                        b.data_ptr() if b is not None else None, pdt, w.eps,
                                        pp, wptr or None, wbytes, sptr)
        wt = params.get("weight")
        return lib.credit_rmsnorm(xp, yp, w.rows, w.cols, DT[w.dtype],
                                  wt.data_ptr() if wt is not None else None, pdt, w.eps, pp,
                                  wptr or None, wbytes, sptr)

    xp, yp = dx.data_ptr(), dy.data_ptr()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            st = launch(xp, yp)
            if st != C.OK:
                raise C.CreditError(st, "warmup launch")
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = clock_sampler(uuid)
    time.sleep(0.3)  # let the sampler start before the timed region
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t_host0 = time.time()
    e0.record(stream)
    for _ in range(args.steps):
        launch(xp, yp)
    e1.record(stream)
    torch.cuda.synchronize()
    t_host1 = time.time()
    if world > 1:
        dist.barrier()
    ms_total = e0.elapsed_time(e1)
    time.sleep(0.1)
    sampler.stop()
    clocks = sampler.summary(t_host0, t_host1)
    assert C.credit_get_device_error(dev) == C.OK

    ms_max = max_over_ranks(ms_total, world, "cuda")
    ms_step = ms_max / args.steps
    bytes_step = w.ideal_bytes()
    value = job_rate(bytes_step, ms_step, world)

    # ---- end to end: pinned host buffers through credit_run_host, which
    # pipelines H2D copies, kernels and D2H copies over row chunks; the
    # parameter vectors are copied from the host every step too
    hx = torch.empty(dx.shape, dtype=dx.dtype, pin_memory=True)
    hx.copy_(dx)
    hin = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True).copy_(v)
           for k, v in params.items()}
    hu = hin.pop("u", None)           # Pearson's second operand travels in the pipeline
    hparams = hin
    hy = torch.empty(dy.shape, dtype=dy.dtype, pin_memory=True)
    hs = torch.empty(w.rows, dtype=torch.float32, pin_memory=True) if row_out else None
    e2e_steps = max(1, min(args.e2e_steps, args.steps))
    h2d = hx.numel() * hx.element_size() + sum(v.numel() * v.element_size()
                                               for v in hin.values())
    if hu is not None:
        h2d += hu.numel() * hu.element_size()
    d2h = hy.numel() * hy.element_size() + (hs.numel() * 4 if row_out else 0)
    dparams = {k: params[k] for k in hparams}
    g = dparams.get("gamma", dparams.get("weight"))
    b = dparams.get("beta")
    call = C.host_call(OPS[w.op], DT[w.dtype], w.rows, w.cols, hx.data_ptr(), hy.data_ptr(),
                       u=hu.data_ptr() if hu is not None else 0,
                       row_out=hs.data_ptr() if hs is not None else 0,
                       p0=g.data_ptr() if g is not None else 0,
                       p1=b.data_ptr() if b is not None else 0, param_dtype=pdt, eps=w.eps)
    rpc = max(1, -(-w.rows // args.e2e_chunks))
    hbytes = C.credit_host_buffer_bytes(call, plan, rpc)
    hbuf = torch.empty(hbytes, dtype=torch.uint8, device=dx.device)
    with torch.cuda.stream(stream):  # untimed: creates the pipeline streams, touches the buffers
        for _ in range(2):
            st = C.credit_run_host(call, plan, hbuf.data_ptr(), hbytes, rpc, sptr)
            if st != C.OK:
                raise C.CreditError(st, "credit_run_host")
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    # an event after every step (no synchronisation in between) shows how
    # the steps spread: the host link stalls now and then for everyone
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps + 1)]
    with torch.cuda.stream(stream):
        marks[0].record(stream)
        for i in range(e2e_steps):
            for k, v in hparams.items():
                dparams[k].copy_(v, non_blocking=True)
            st = C.credit_run_host(call, plan, hbuf.data_ptr(), hbytes, rpc, sptr)
            if st != C.OK:
                raise C.CreditError(st, "credit_run_host")
            marks[i + 1].record(stream)
    torch.cuda.synchronize()
    te = max_over_ranks(marks[0].elapsed_time(marks[-1]), world, "cuda")
    e2e_value = job_rate(bytes_step, te / e2e_steps, world)
    step_ms = [marks[i].elapsed_time(marks[i + 1]) for i in range(e2e_steps)]

    peak, peak_kind = measured_peak()
    variant_key = C.variant_name(plan)
    launches_per_step = 2 if plan.variant == C.TWO_PASS else 1
    traffic = stored_traffic(w.name, variant_key)
    # the dominant kernel is the only kernel of a clustered step
    achieved = bytes_step / (ms_step * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "peak_kind": peak_kind, "traffic": traffic,
                "ideal_bytes": bytes_step}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cores = len(os.sched_getaffinity(0))
        rows = cpu_sample_rows(w, inputs, cores, args.cpu_budget)
        rate, dt = cpu_oracle_rate(w, inputs, rows, cores)
        cpu = {"value": rate, "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": f"first {rows} of {w.rows} rows (full width {w.cols}), "
                         f"{dt:.1f} s on {cores} threads"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "rows": w.rows, "cols": w.cols, "io_dtype": w.dtype,
                       "param_dtype": w.param_dtype, "variant": variant_key,
                       "threads": plan.threads, "smem_bytes": int(plan.smem_bytes),
                       "ctas_per_sm": plan.ctas_per_sm, "clusters": plan.active_clusters,
                       "tuning_us": tuning,
                       "e2e_pipeline": f"credit_run_host, {-(-w.rows // rpc)} chunks of {rpc} rows",
                       "parallelism": f"replicas x{world}",
                       "l2": "input larger than L2 (no flush)",
                       "pct_of_nominal_8TBps": 100 * achieved / 8000.0},
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                    "step_ms_median": statistics.median(step_ms),
                    "step_ms_max": max(step_ms)},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
