"""Failure detection without a GPU fault: every wait in the tensor-core kernels is bounded.  The
test hook makes the forward's producer withhold its first K/V tile, so the consumers' waits run
out; the kernel records FA_ERR_TIMEOUT in the device error word and returns normally, the host
reads it, and the context stays usable for the next (correct) call."""
import pytest
import torch

from gpu_helpers import compare_fwd, run_gpu
from workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu

FA_OK, FA_ERR_TIMEOUT = 0, 4


def test_bounded_wait_reports_timeout_and_recovers():
    import exact_io_aware_23_gb300 as fa
    x = make_inputs(Workload("wd", 1, 2, 300, 64, "bf16"), seed=3)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    assert fa.check_device_status() == FA_OK
    try:
        fa.set_wait_limit_ms(100)
        fa.set_fault_injection(1)
        fa.forward(q, k, v)                       # launches; the kernel gives up after ~100 ms
        assert fa.check_device_status() == FA_ERR_TIMEOUT
        assert fa.check_device_status() == FA_OK  # reading the word clears it
    finally:
        fa.set_fault_injection(0)
        fa.set_wait_limit_ms(0)
    compare_fwd(x, run_gpu(x, backward=False))    # the context is still good
