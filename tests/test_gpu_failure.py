"""Failure detection on the GPU without a fault: a pipeline wait that nothing completes gives
up after its limit, the kernel returns, the device error word says where, and the context
stays usable for the next call."""
import time

import numpy as np
import pytest
import torch

import workloads as W
from pkv_testutil import GpuBatch, assert_attention_close, expect_no_device_error

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_reports_and_returns(pkv):
    expect_no_device_error(pkv)
    t0 = time.perf_counter()
    pkv.pkv_check_wait_timeout()
    code, info = pkv.pkv_get_device_error(clear=True)   # synchronises: the kernel has returned
    waited = time.perf_counter() - t0
    assert code == 5 and pkv.DEVERR[code] == "pipeline wait timed out"   # PKV_DEVERR_TIMEOUT
    assert info == pkv.WAIT_CHECK_INFO
    assert 1.5 < waited < 30, waited                     # it waited out its limit, then returned
    # the context is still usable: a decode right after matches the oracle
    wl = W.tiny_decode()
    b = GpuBatch(wl, W.paged_values(wl))
    b.run_slots_and_store(pkv, decode=True)
    assert_attention_close(b.run_decode(pkv), b.oracle_decode(), "decode after a timeout")
    expect_no_device_error(pkv)
