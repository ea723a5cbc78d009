"""Failure detection without a GPU fault: a pipeline wait that can never complete gives
up after its bound, the kernel flags DEV_WAIT_TIMEOUT in the device status word and
returns, and the context stays usable for the next launch."""
import time

import pytest
import torch

from paged_kv_cache_87_gb300 import binding, inputs
from tests.test_gpu_decode import _full_parity

pytestmark = pytest.mark.gpu


def test_a_wait_that_never_completes_flags_a_timeout_and_the_context_survives():
    binding.pkv_get_device_status()                       # clear
    torch.cuda.synchronize()
    t0 = time.monotonic()
    binding.pkv_selftest_wait_bound()
    status = binding.pkv_get_device_status()              # synchronises
    dt = time.monotonic() - t0
    assert status & binding.DEV_WAIT_TIMEOUT
    assert status & ~binding.DEV_WAIT_TIMEOUT == 0
    assert 1.5 < dt < 60                                   # the bound is 2 s of device time
    # the same context still runs a decode to the oracle's tolerance, with a clean status
    _full_parity(inputs.make_config(0))
    assert binding.pkv_get_device_status() == 0
