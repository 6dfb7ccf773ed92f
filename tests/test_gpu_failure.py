"""Failure handling on the GPU without a fault: a bounded wait that nothing
satisfies gives up, the host reads HSWA_ERR_TIMEOUT from the device error
word, and the same context then runs a decode step that matches the oracle."""
import time

import pytest

import hswa_workloads as wl
import hybrid_sliding_window_dual_gb300 as H
from scenario import Scenario


@pytest.mark.gpu
def test_bounded_wait_times_out_and_context_stays_usable():
    assert H.hswa_check() == 0
    t0 = time.time()
    H.hswa_selftest_bounded_wait()
    assert H.hswa_check() == H.HSWA_ERR_TIMEOUT
    assert time.time() - t0 < 30
    assert H.hswa_check() == 0  # cleared
    from test_gpu_decode import run_decode_step
    sc = Scenario(64, 8, 128, 64, 128, wl.DTYPE_BF16, [100, 2000], seed=51)
    run_decode_step(sc, [0, 1], seed=3, expect_kernel="decode_mma_bf16_d128")
