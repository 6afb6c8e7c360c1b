"""GPU failure detection without a fault: a kernel whose bounded wait runs
out.  bigemm_selftest_timeout launches the split-K partial kernel with a
producer that issues no loads; the MMA issuer's wait on the first stage gives
up after its 2 s limit, every role leaves its wait, and the kernel ends with
a bit in the device error word.  The host reads it with bigemm_device_status,
and the context keeps working."""
import time

import pytest
import torch

import deterministic_invariant_gemm_gb300 as dig
import workloads
from gemm_check import bits_equal

pytestmark = pytest.mark.gpu

ERR_TIMEOUT = 6


def test_expired_wait_is_reported_and_the_context_survives(cuda_device):
    dig.load()
    assert dig.bigemm_device_status(reset=True) == 0
    A, B = workloads.pair(16, 256, 512, 3)
    A, B = A.cuda(), B.cuda()
    before = dig.matmul(A, B, split_k=1)
    torch.cuda.synchronize()

    t0 = time.time()
    assert dig.bigemm_selftest_timeout() == 0
    assert dig.bigemm_last_launch_count() == 1
    st = dig.bigemm_device_status(reset=True)          # synchronises
    elapsed = time.time() - t0
    assert st == ERR_TIMEOUT, st
    assert 1.5 < elapsed < 30.0, elapsed               # the 2 s limit, not a hang
    assert dig.bigemm_device_status(reset=False) == 0  # the reset cleared it

    # the context still works and gives the same bits as before
    after = dig.matmul(A, B, split_k=1)
    torch.cuda.synchronize()
    assert bits_equal(after, before)
    assert dig.bigemm_device_status(reset=False) == 0
