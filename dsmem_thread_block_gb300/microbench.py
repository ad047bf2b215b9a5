"""DSMEM microbenchmark suite (command line).

Measures, on one GPU, the cluster-barrier round trip, the replicated-push
exchange and the st.async exchange (deposits counted on each receiver's
mbarrier, no cluster barrier) for every cluster size 2..16, the staged-copy
rate (HBM -> shared memory -> HBM, bulk copies) at 1..8 CTAs per SM, the L2
read rate of every SM re-reading a 2, 8 and 32 MiB window, remote and local shared-memory load
latency (pointer chase), and remote / local 16-byte load and store throughput
of one CTA, each as the median of 15 launches (CREDIT summary page, "C.
Positioning": latency, throughput and repeated cluster-synchronisation
microbenchmarks with the CTAs on different SMs).  Prints one JSON object.

    python -m dsmem_thread_block_gb300.microbench [--device 0] [--runs 15]
"""
from __future__ import annotations

import argparse
import json

from . import _credit as C


def run_suite(device: int = 0, runs: int = 15, sizes=range(2, 17)) -> dict:
    out = {"device": device, "runs": runs, "barrier": {}, "exchange": {}, "async_exchange": {}}
    for P in sizes:
        out["barrier"][P] = C.credit_bench_dsmem(device, C.BENCH_BARRIER, P, 2000, runs).as_dict()
        out["exchange"][P] = C.credit_bench_dsmem(device, C.BENCH_EXCHANGE, P, 2000, runs).as_dict()
        out["async_exchange"][P] = C.credit_bench_dsmem(device, C.BENCH_ASYNC_EXCHANGE, P, 2000,
                                                        runs).as_dict()
    for name, kind, iters in (("remote_load_latency", C.BENCH_REMOTE_LOAD_LATENCY, 20000),
                              ("local_load_latency", C.BENCH_LOCAL_LOAD_LATENCY, 20000),
                              ("remote_store_bw", C.BENCH_REMOTE_STORE_BW, 64),
                              ("remote_load_bw", C.BENCH_REMOTE_LOAD_BW, 64),
                              ("local_store_bw", C.BENCH_LOCAL_STORE_BW, 64),
                              ("local_load_bw", C.BENCH_LOCAL_LOAD_BW, 64)):
        out[name] = C.credit_bench_dsmem(device, kind, 2, iters, runs).as_dict()
    out["stage_copy"] = {}
    for k in (1, 2, 3, 4, 6, 8):
        g, res = C.credit_stage_copy_rate(device, k, min(runs, 7))
        out["stage_copy"][k] = {"gbps": g, "resident": res}
    out["l2_read_gbps"] = {str(b): C.credit_l2_read_rate(device, b, min(runs, 7))
                           for b in (1 << 21, 1 << 23, 1 << 25)}
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--device", type=int, default=0)
    ap.add_argument("--runs", type=int, default=15)
    a = ap.parse_args()
    print(json.dumps(run_suite(a.device, a.runs)))


if __name__ == "__main__":
    main()
