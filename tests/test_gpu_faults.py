"""Failure detection without a GPU fault: a bounded device-side wait is made to
give up on purpose (an mbarrier armed for bulk-copy bytes that no copy
delivers, waited on with the kernels' own bounded wait and a 2 ms limit).  The
kernel must return, the device error word must read RR_ERR_DEVICE_TIMEOUT, and
the context must stay usable: a normal call afterwards matches the oracle and
leaves the error word clear."""
import time

import pytest
import torch

import row_reduction_pass_gb300 as rr
from row_reduction_pass_gb300 import synth

from parity import check_softmax

pytestmark = pytest.mark.gpu

RR_ERR_DEVICE_TIMEOUT = 6


def test_bounded_wait_gives_up_and_context_stays_usable():
    dev = torch.cuda.current_device()
    assert rr.rr_read_device_error(dev, reset=True) == 0
    t0 = time.perf_counter()
    rr.rr_selftest_bounded_wait(2_000_000)        # 2 ms
    torch.cuda.synchronize()                       # the kernel has returned
    elapsed = time.perf_counter() - t0
    assert rr.rr_read_device_error(dev, reset=True) == RR_ERR_DEVICE_TIMEOUT
    assert elapsed < 5.0, f"the 2 ms wait took {elapsed:.3f} s to give up"
    assert rr.rr_read_device_error(dev, reset=False) == 0    # cleared by the read
    x, _ = synth.xent_inputs(300, 1000, "bf16", 3.0, 77, ignore_frac=0.0, outlier_frac=0.01,
                             masked_row_every=37)
    check_softmax(x, "bf16")
    assert rr.rr_read_device_error(dev, reset=True) == 0


def test_bounded_wait_rejects_bad_limits():
    for bad in (0, -5, 2_000_000_000):
        with pytest.raises(rr.RRError, match="INVALID_ARG"):
            rr.rr_selftest_bounded_wait(bad)
