"""Failure detection without a GPU fault: a bounded in-kernel wait that can
never complete gives up, reports through the device error flags, and leaves
the context usable for the next forward."""
import numpy as np
import pytest
import torch

import block_sparse_masked_gb300 as fa
from block_sparse_masked_gb300 import runner
from block_sparse_masked_gb300 import workloads as W

import parity as PT

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    PT.ensure_built()


def test_bounded_wait_times_out_and_context_survives():
    assert fa.fa_device_error_flags() == 0
    fa.fa_selftest_wait_timeout(1_000_000)          # 1 ms
    torch.cuda.synchronize()
    assert fa.fa_device_error_flags() & 1           # the wait gave up and said so
    assert fa.fa_device_error_flags() == 0          # reading clears the bits
    w = W.tiny_causal(0)
    dp = runner.to_device(w)
    plan = runner.build_plan(dp)
    runner.forward(dp, plan)
    torch.cuda.synchronize()
    assert fa.fa_device_error_flags() == 0
    rows = {(0, h): list(range(256)) for h in range(2)}
    PT.check_rows(w, dp.o, dp.lse, rows)
    plan.free()


def test_selftest_argument_range():
    with pytest.raises(fa.FaError) as ei:
        fa.fa_selftest_wait_timeout(10)
    assert ei.value.code == fa.FA_ERR_INVALID_ARG
