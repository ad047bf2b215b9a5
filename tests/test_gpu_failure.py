"""Failure detection without a GPU fault: a bounded device-side wait that
nothing completes gives up, records the timeout in the device error word, the
host reads CREDIT_ERR_DEVICE_TIMEOUT, and the context stays usable."""
import numpy as np
import pytest
import torch

from dsmem_thread_block_gb300 import _credit as C
from dsmem_thread_block_gb300 import workloads as wl

from gpu_helpers import check, make_plan, run

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    assert C.credit_get_device_error(0) == C.OK  # clean before
    assert C.credit_selftest_wait_timeout(0, 2_000_000) == C.ERR_DEVICE_TIMEOUT
    assert C.credit_get_device_error(0) == C.OK  # read-and-clear
    # the library still computes correctly afterwards
    w = wl.SOFTMAX_F32_64x4096
    inp = w.generate()
    check(w, run(w, inp, make_plan(w, C.CLUSTER, 4)), inp)


def test_selftest_argument_checks():
    assert C.credit_selftest_wait_timeout(0, 10) == C.ERR_INVALID_ARG
    assert C.credit_selftest_wait_timeout(0, 10 ** 10) == C.ERR_INVALID_ARG
    torch.cuda.synchronize()
