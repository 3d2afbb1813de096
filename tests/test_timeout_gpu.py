"""The bounded-wait failure path on the GPU, without a fault.

A test-only kernel waits on barriers that nothing completes (include/fa_selftest.h,
fa_selftest_wait_timeout): one warp with a short limit, the other with the
kernels' own two-second limit. The first must run out, raise the abort flag and
record the timeout bit; the second must leave as soon as it sees the flag; the
CTA frees its tensor memory and returns. The library then reports
FA_ERR_DEVICE_TIMEOUT exactly once, and attention calls that follow on the same
context are still correct.
"""
import time

import pytest
import torch

import exact_io_aware_27_gb300 as fa
from exact_io_aware_27_gb300.inputs import SINGLE_HEAD_128, workload_inputs
from tests import parity

pytestmark = pytest.mark.gpu

LIMIT_CYCLES = 2_000_000  # about 1 ms at 2 GHz


def test_wait_runs_out_and_reports_once():
    fa.build()
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.api.FA_OK  # clear anything left before
    t0 = time.perf_counter()
    ok = fa.fa_selftest_wait_timeout(LIMIT_CYCLES)  # copies `out` back: synchronises
    elapsed = time.perf_counter() - t0
    assert ok == [0, 0], f"both waits must give up, got {ok}"
    # Warp 1's own limit is about two seconds: returning well before it shows that
    # the abort flag ended its wait.
    assert elapsed < 1.0, f"the kernel took {elapsed:.3f} s"
    assert fa.fa_get_device_status() == fa.api.FA_ERR_DEVICE_TIMEOUT
    assert fa.fa_get_device_status() == fa.api.FA_OK  # read-and-clear


def test_attention_correct_after_a_timeout():
    fa.build()
    assert fa.fa_selftest_wait_timeout(LIMIT_CYCLES) == [0, 0]
    assert fa.fa_get_device_status() == fa.api.FA_ERR_DEVICE_TIMEOUT
    w = SINGLE_HEAD_128
    Q, K, V, dO = workload_inputs(w)
    for causal in (False, True):
        got = parity.run_gpu(Q, K, V, dO, causal)
        parity.check_heads(Q, K, V, dO, causal, got)
    assert fa.fa_get_device_status() == fa.api.FA_OK
