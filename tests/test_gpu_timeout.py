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


def test_expired_wait_is_reported_and_the_context_survives(builtin_scratch):
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


@pytest.mark.parametrize("pair_mode", [None, "always"])
def test_ozaki_order_wait_gives_up_once_for_the_whole_grid(builtin_scratch, pair_mode):
    """The Ozaki kernel's epilogues wait for the previous slice pair of their
    tile, possibly on another CTA.  bigemm_selftest_ozaki_order_timeout starts
    every tile's count far below zero, so no such wait is ever met: the first
    to give up (after 2 s) sets the launch's abort word and every other CTA
    leaves at once -- one 2 s limit for the grid, not one per CTA or per pair
    in turn.  The error word reports the timeout, and a later product is
    still right.  Run on single CTAs (the default rule at this size) and on CTA
    pairs, whose drains also end after one limit."""
    dig.load()
    assert dig.bigemm_device_status(reset=True) == 0
    g = workloads.generator(5)
    A = torch.randn(200, 300, generator=g, dtype=torch.float64).cuda()
    B = torch.randn(300, 100, generator=g, dtype=torch.float64).cuda()
    before = dig.ozaki_matmul(A, B)
    torch.cuda.synchronize()

    prev = dig.bigemm_set_pair_mode(dig.PAIR_ALWAYS if pair_mode else dig.PAIR_AUTO)
    try:
        t0 = time.time()
        assert dig.bigemm_selftest_ozaki_order_timeout() == 0
        st = dig.bigemm_device_status(reset=True)      # synchronises
        elapsed = time.time() - t0
    finally:
        dig.bigemm_set_pair_mode(prev)
    assert st == ERR_TIMEOUT, st
    assert 1.5 < elapsed < 8.0, elapsed                # one limit for the grid
    assert dig.bigemm_device_status(reset=False) == 0

    after = dig.ozaki_matmul(A, B)
    torch.cuda.synchronize()
    assert torch.equal(after.view(torch.int64), before.view(torch.int64))
    assert dig.bigemm_device_status(reset=False) == 0
