"""DSMEM microbenchmarks and the control kernel: sanity invariants (there is
no GB300 reference value to compare with, so these numbers are judged by
properties that must hold)."""
import pytest
import torch

from dsmem_thread_block_gb300 import _credit as C

pytestmark = pytest.mark.gpu


def test_pair_kinds_run_on_two_sms_and_remote_is_slower():
    rem = C.credit_bench_dsmem(0, C.BENCH_REMOTE_LOAD_LATENCY, 2, 5000, 5)
    loc = C.credit_bench_dsmem(0, C.BENCH_LOCAL_LOAD_LATENCY, 2, 5000, 5)
    assert rem.smids[0] != rem.smids[1]
    assert 0 < loc.median_cycles < rem.median_cycles
    for kind in (C.BENCH_REMOTE_STORE_BW, C.BENCH_REMOTE_LOAD_BW, C.BENCH_LOCAL_STORE_BW,
                 C.BENCH_LOCAL_LOAD_BW):
        r = C.credit_bench_dsmem(0, kind, 2, 16, 5)
        assert r.bytes_per_cycle > 0 and r.gbps > 0


@pytest.mark.parametrize("P", [2, 4, 8, 16])
def test_barrier_and_exchange_costs(P):
    b = C.credit_bench_dsmem(0, C.BENCH_BARRIER, P, 500, 5)
    e = C.credit_bench_dsmem(0, C.BENCH_EXCHANGE, P, 500, 5)
    assert len(set(b.smids[:P])) == P  # one CTA per SM
    assert 0 < b.median_cycles < 1e5
    assert e.median_cycles >= 0.8 * b.median_cycles  # the push adds to the barrier


@pytest.mark.parametrize("P", [2, 4, 8, 16])
def test_async_exchange_runs_on_distinct_sms(P):
    # st.async deposits + a wait on the own mbarrier: no cluster barrier per
    # exchange, so one exchange should cost no more than push + barrier
    a = C.credit_bench_dsmem(0, C.BENCH_ASYNC_EXCHANGE, P, 500, 5)
    e = C.credit_bench_dsmem(0, C.BENCH_EXCHANGE, P, 500, 5)
    assert len(set(a.smids[:P])) == P
    assert 0 < a.median_cycles < 1e5
    assert a.median_cycles <= 1.5 * e.median_cycles


def test_barrier_cost_grows_with_cluster_size():
    c2 = C.credit_bench_dsmem(0, C.BENCH_BARRIER, 2, 1000, 7).median_cycles
    c16 = C.credit_bench_dsmem(0, C.BENCH_BARRIER, 16, 1000, 7).median_cycles
    assert c16 >= 0.8 * c2


def test_control_kernel_excess_over_one_cta():
    t1 = C.credit_control_time(0, 1024, 1, 256, 65536, 1, 2, 5)
    t8 = C.credit_control_time(0, 1024, 8, 256, 65536, 1, 2, 5)
    assert t1 > 0 and t8 > 0
    # clustered control: P times the CTAs and 2 cluster barriers each
    assert t8 >= 0.5 * t1


def test_microbench_argument_checks():
    with pytest.raises(C.CreditError):
        C.credit_bench_dsmem(0, 99, 2, 10, 3)
    with pytest.raises(C.CreditError):
        C.credit_bench_dsmem(0, C.BENCH_BARRIER, 17, 10, 3)
    torch.cuda.synchronize()


def test_l2_read_rate_exceeds_the_hbm_copy_rate():
    # a 2 MiB window stays in L2: all SMs read it faster than the staged
    # copy streams HBM (read + write)
    small = C.credit_l2_read_rate(0, 1 << 21, 5)
    hbm, _ = C.credit_stage_copy_rate(0, 2, 3)
    assert small > 1.5 * hbm > 0
    with pytest.raises(C.CreditError):
        C.credit_l2_read_rate(0, 1000, 3)  # below 64 KiB
    with pytest.raises(C.CreditError):
        C.credit_l2_read_rate(0, 1 << 30, 3)  # beyond 64 MiB: no longer an L2 window
