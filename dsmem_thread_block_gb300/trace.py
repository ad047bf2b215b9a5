"""Phase trace of the one-row-per-cluster kernel (command line).

Runs one workload through the checked build (libcredit_checked.so), whose
kernel stamps %globaltimer at seven points of every CTA's life -- entry, bulk
copies issued, statistics folded, CTA partial, exchange and combine done,
output written, exit -- and records its SM id.  Prints one JSON object: per
phase the median and 90th percentile over CTAs, the median CTA lifetime, the
idle gap between consecutive CTAs on one SM, and the share of time each SM
holds at least one CTA.  The checked build also runs its index checks, so the
phase times include them; use it for where the time goes, not for rates.

    python -m dsmem_thread_block_gb300.trace --workload softmax_bf16_sweep_1048576 --cluster-size 10

`--rows R` traces the workload's first R rows (the trace holds 8192 CTAs).
"""
from __future__ import annotations

import argparse
import json

import numpy as np

from . import _credit as C
from . import workloads as wl

PHASES = ["setup_and_copy_issue", "stage_and_fold", "cta_partial", "exchange_and_combine",
          "output", "exit_wait"]


def _table():
    t = {w.name: w for w in wl.ALL}
    for c in wl.SWEEP_COLS:
        w = wl.sweep_point(c)
        t[w.name] = w
    return t


def summarize(stamps: np.ndarray) -> dict:
    """Per-phase statistics of trace rows [ctas, 8] (7 stamps + SM id)."""
    t = stamps[:, :7].astype(np.int64)
    sm = stamps[:, 7]
    t = t - t[:, 0].min()
    ph = np.diff(t, axis=1) / 1e3  # us
    out = {"ctas": int(len(t)), "sms": int(len(np.unique(sm))),
           "span_us": round(float(t[:, 6].max()) / 1e3, 2),
           "phase_median_us": {n: round(float(np.median(ph[:, j])), 3) for j, n in enumerate(PHASES)},
           "phase_p90_us": {n: round(float(np.percentile(ph[:, j], 90)), 3)
                            for j, n in enumerate(PHASES)},
           "cta_life_median_us": round(float(np.median(t[:, 6] - t[:, 0])) / 1e3, 3)}
    gaps, busy = [], []
    for s in np.unique(sm):
        life = sorted(zip(t[sm == s, 0], t[sm == s, 6]))
        covered, end, first = 0, None, life[0][0]
        for a, b in life:
            if end is None or a > end:
                if end is not None:
                    gaps.append(a - end)
                covered += b - a
                end = b
            elif b > end:
                covered += b - end
                end = b
        busy.append(covered / max(1, end - first))
    out["sm_gap_median_us"] = round(float(np.median(gaps)) / 1e3, 3) if gaps else None
    out["sm_busy_share_median"] = round(float(np.median(busy)), 4)
    return out


def run(workload: str, cluster_size: int, device: int = 0, warmup: int = 3,
        rows: int = 0) -> dict:
    import torch

    w = _table()[workload]
    if rows:
        w = w.with_rows(rows)
    torch.cuda.set_device(device)
    inp = w.generate()

    def dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
        return torch.from_numpy(a).cuda()

    x = dev(inp["x"])
    y = torch.empty_like(x)
    params = {k: dev(v) for k, v in inp.items() if k != "x"}
    dt = C.F32 if w.dtype == "f32" else C.BF16
    pdt = (C.F32 if w.param_dtype == "f32" else C.BF16) if w.param_dtype else C.F32
    op = {wl.SOFTMAX: C.SOFTMAX, wl.LAYERNORM: C.LAYERNORM, wl.RMSNORM: C.RMSNORM}[w.op]
    with C.use_checked_build():
        assert C.credit_debug_build() == 1
        plan = C.credit_plan_for(op, w.rows, w.cols, dt, device, C.CLUSTER, cluster_size)
        ctas = w.rows * cluster_size
        if ctas > C.TRACE_CTAS:
            raise ValueError(f"{ctas} CTAs: the trace holds {C.TRACE_CTAS}")
        s = torch.cuda.current_stream().cuda_stream

        def go():
            if w.op == wl.SOFTMAX:
                st = C.credit_softmax(x.data_ptr(), y.data_ptr(), w.rows, w.cols, dt, plan, 0, 0, s)
            elif w.op == wl.LAYERNORM:
                g, b = params.get("gamma"), params.get("beta")
                st = C.credit_layernorm(x.data_ptr(), y.data_ptr(), w.rows, w.cols, dt,
                                        g.data_ptr() if g is not None else 0,
                                        b.data_ptr() if b is not None else 0, pdt, w.eps, plan,
                                        0, 0, s)
            else:
                wt = params.get("weight")
                st = C.credit_rmsnorm(x.data_ptr(), y.data_ptr(), w.rows, w.cols, dt,
                                      wt.data_ptr() if wt is not None else 0, pdt, w.eps, plan,
                                      0, 0, s)
            if st != C.OK:
                raise C.CreditError(st, "trace launch")

        for _ in range(warmup + 1):
            go()
        stamps = C.credit_debug_trace(ctas)
        err = C.credit_get_device_error(device)
    out = {"workload": w.name, "cluster_size": cluster_size, "threads": plan.threads,
           "active_clusters": plan.active_clusters, "smem_bytes": plan.smem_bytes,
           "device_error": C.status_string(err)}
    out.update(summarize(stamps))
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", required=True)
    ap.add_argument("--cluster-size", type=int, required=True)
    ap.add_argument("--device", type=int, default=0)
    ap.add_argument("--rows", type=int, default=0, help="trace the first ROWS rows (0 = all)")
    a = ap.parse_args()
    print(json.dumps(run(a.workload, a.cluster_size, a.device, rows=a.rows)))


if __name__ == "__main__":
    main()
