"""Host logic of the benchmark's evidence fields (no GPU): the roofline
denominator comes from the measured peaks file, else the stated fallback;
stored ncu traffic is reported only while the kernel sources still hash to
the value recorded with it; the whole-job rate divides all ranks' bytes by
the slowest rank's time."""
import json
import os

import bench


def test_traffic_is_reported_only_for_matching_kernel_sources(monkeypatch):
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        d = json.load(f)
    key = next(iter(d["entries"]))
    workload, variant = key.split("|")
    if d["kernel_source_hash"] == bench.kernel_source_hash():
        assert bench.stored_traffic(workload, variant) == d["entries"][key]["dram_bytes_per_launch"]
    assert bench.stored_traffic(workload, "cluster:99") is None  # never captured
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)
    assert bench.stored_traffic(workload, variant) is None  # sources changed since the capture


def test_kernel_source_hash_covers_the_kernel_sources(tmp_path, monkeypatch):
    # every file that defines a kernel or its launch changes the hash; the
    # cost model, microbenchmarks and host pipeline do not
    csrc = tmp_path / "dsmem_thread_block_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in bench.KERNEL_SOURCES + ("costmodel.cu", "microbench.cu", "host.cu"):
        (csrc / f).write_text(f)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    seen = {bench.kernel_source_hash()}
    for f in bench.KERNEL_SOURCES:
        (csrc / f).write_text(f + " edited")
        seen.add(bench.kernel_source_hash())
    assert len(seen) == len(bench.KERNEL_SOURCES) + 1
    h = bench.kernel_source_hash()
    for f in ("costmodel.cu", "microbench.cu", "host.cu"):
        (csrc / f).write_text(f + " edited")
    assert bench.kernel_source_hash() == h
    real = set(os.listdir(os.path.join(os.path.dirname(os.path.dirname(__file__)),
                                       "dsmem_thread_block_gb300", "csrc")))
    assert set(bench.KERNEL_SOURCES) <= real


def test_peak_from_the_measured_file_else_the_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_peak() == (bench.FALLBACK_HBM_GBS, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6781.4}))
    assert bench.measured_peak() == (6781.4, "measured")


def test_job_rate_uses_the_slowest_rank():
    # 2 ranks, 1 GB each per step, the slowest rank 2 ms per step: 1000 GB/s
    assert abs(bench.job_rate(1e9, 2.0, 2) - 1000.0) < 1e-9


def test_plan_names_round_trip():
    # the names the library's plans print are the names --variant accepts
    from dsmem_thread_block_gb300 import _credit as C
    p = C.Plan(variant=C.CLUSTER, cluster_size=8, threads=128, slice_elems=32768,
               staged_elems=9728, rows_per_cluster=1)
    assert C.variant_name(p) == "cluster:8:s9728:t128"
    assert bench.parse_variant(C.variant_name(p)) == {
        "kind": "cluster", "P": 8, "R": 0, "staged": 9728, "threads": 128}
    p = C.Plan(variant=C.CLUSTER, cluster_size=12, threads=256, slice_elems=65536,
               staged_elems=37376, rows_per_cluster=1)
    assert C.variant_name(p) == "cluster:12:s37376"
    p = C.Plan(variant=C.CLUSTER, cluster_size=8, threads=256, slice_elems=32768,
               staged_elems=18432, rows_per_cluster=2)
    assert bench.parse_variant(C.variant_name(p)) == {
        "kind": "cluster", "P": 8, "R": 2, "staged": 18432, "threads": 0}
    p = C.Plan(variant=C.CLUSTER, cluster_size=8, threads=128, slice_elems=16384,
               staged_elems=16384, rows_per_cluster=1)
    assert C.variant_name(p) == "cluster:8"  # whole slice staged: the threads are the planner's
    assert bench.parse_variant("persist:9")["kind"] == "persist"
    for bad in ("cluster:8:q5", "warp:3"):
        try:
            bench.parse_variant(bad)
        except ValueError:
            continue
        raise AssertionError(bad)
