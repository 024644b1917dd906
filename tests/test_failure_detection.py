"""Failure detection without a GPU fault: a bounded device wait that runs out reports
FA_ERR_TIMEOUT through the error word, and the context stays usable afterwards."""
import pytest
import torch

from exact_io_aware_28_gb300 import fa
from exact_io_aware_28_gb300 import workloads as W

from _parity import compare, run_library, run_oracle


def test_selftest_rejects_bad_limits():
    lib = fa.load()
    assert lib.fa_selftest_wait_timeout(0, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_selftest_wait_timeout(20000, None) == fa.FA_ERR_INVALID_ARG


@pytest.mark.gpu
def test_bounded_wait_times_out_and_context_survives():
    assert fa.fa_device_error() == fa.FA_OK
    fa.fa_selftest_wait_timeout(50)
    assert fa.fa_device_error() == fa.FA_ERR_TIMEOUT   # reported ...
    assert fa.fa_device_error() == fa.FA_OK            # ... and cleared
    x = W.make_inputs(W.custom("after", 1, 2, 200, 64, "bf16", causal=True), seed=3,
                      device="cuda")
    compare(run_library(x), run_oracle(x), "bf16")
