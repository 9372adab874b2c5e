"""Failure detection on the GPU without a fault: a bounded barrier wait that
nothing satisfies must give up after about a second, report
TM_ERR_DEVICE_TIMEOUT through tm_device_error, and leave the context usable."""
import time

import pytest
import torch

from tests.gpu_util import TOL, run_and_compare
from w4a16_quantized_gemm_gb300 import binding

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)


def test_bounded_wait_times_out_and_context_survives():
    binding.device_error(clear=True)
    t0 = time.perf_counter()
    binding.selftest_wait_timeout()
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert 0.5 < dt < 30.0, dt                      # it waited about the limit, then returned
    assert binding.device_error(clear=True) == 1    # timeout bit, reported (status 5) and cleared
    assert binding.device_error(clear=False) == 0
    err, _ = run_and_compare(8, 1024, 384, 128)     # the context still computes correctly
    assert err <= TOL
