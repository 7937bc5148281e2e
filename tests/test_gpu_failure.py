"""The failure path of the kernels' bounded waits, exercised without a fault,
trap or hang: a self-test kernel waits on a barrier that nothing completes;
its wait gives up after the iteration limit, the event is recorded and read
back on the host, and the same context then runs a product that matches the
oracle."""
import time

import numpy as np
import pytest
import torch

import bit_weight_gemv_sign_b300 as b1
from bit_weight_gemv_sign_b300 import synth
from tests.helpers import abs_bound, assert_gemv_close, dev_bf16, dev_u8, dev_u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    b1.load()


def test_bounded_wait_gives_up_and_the_context_survives(orc):
    b1.bit1_device_wait_timeouts()                  # clear earlier events
    done = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    b1.bit1_selftest_wait_timeout(done)
    torch.cuda.synchronize()
    seconds = time.perf_counter() - t0
    assert int(done.item()) == 1                    # the kernel ran to its end
    assert b1.bit1_device_wait_timeouts() & 16      # and recorded the timeout
    assert seconds < 2, seconds                     # the self-test's own short bound
    print(f"bounded wait gave up after {seconds:.3f} s")
    N, K = 512, 4096
    bits, scales = synth.matrix(N, K, 4242)
    x = synth.x_for(1, K, 4242)
    y = b1.bit1_gemv_ex(dev_u8(bits), dev_u16(scales), dev_bf16(x).view(1, K), variant=b1.LUT6)
    torch.cuda.synchronize()
    assert_gemv_close(y, orc.gemv(bits, scales, x, 1, N, K), abs_bound(scales, x, K), "after the self-test")
    assert b1.bit1_device_wait_timeouts() == 0
