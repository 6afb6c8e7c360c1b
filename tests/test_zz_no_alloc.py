"""bigemm_run_splitk_static: the split-K product for callers that cannot
allocate device memory.

Some callers may not allocate per call, and cannot hand the library a
workspace either: for example a serving loop that forbids allocation after
start-up (cudaMalloc can synchronise the whole device), or a plugin inside a
host framework that owns all device memory through its own allocator and does
not expose it over a C interface.  For them the library keeps a fixed 16 MiB
array of split-K scratch in its device image.

This file is collected last, so that a run stopping at its first failure has
run every other test before it.  The call shares one array across calls, so
the check below covers two calls in a row, with the second one finding the
first one's partial sums still in the array; the tests that use the array
hold the `builtin_scratch` fixture, which keeps them from overlapping.  Each
result must equal the ordinary entry point's (bigemm_run with a caller
workspace) within the parity tolerance, and in fact bit for bit, since the
same kernels run.
"""
import numpy as np
import pytest
import torch

import deterministic_invariant_gemm_gb300 as dig
import workloads
from gemm_check import check_tolerance, oracle_rows, round_up, to_f64

pytestmark = pytest.mark.gpu


def _device_pair(M, N, K, seed):
    A, B = workloads.pair(M, N, K, seed, a_std=1.0, b_std=0.02)
    lda, ldb = round_up(K, 8), round_up(N, 8)
    Ad = torch.zeros((M, lda), dtype=torch.bfloat16, device="cuda")
    Bd = torch.zeros((K, ldb), dtype=torch.bfloat16, device="cuda")
    Ad[:, :K] = A.cuda()
    Bd[:, :N] = B.cuda()
    return A, B, Ad, Bd, lda, ldb


@pytest.mark.parametrize("order", ["static_first", "workspace_first"])
def test_static_scratch_matches_workspace_entry_point(builtin_scratch, order):
    # Two calls in a row with different shapes and splits; the second finds
    # the first call's partials in the shared array.
    # splits above 8 always take the workspace path (partial + reduction), so
    # the array is really used
    cases = [(16, 4096, 8192, 16, 21), (64, 1000, 3000, 12, 22)]
    for M, N, K, S, seed in cases:
        assert 0 < dig.bigemm_workspace_bytes(M, N, K, S) <= dig.STATIC_SCRATCH_BYTES
        A, B, Ad, Bd, lda, ldb = _device_pair(M, N, K, seed)
        ldc = round_up(N, 4)
        c_static = torch.full((M, ldc), float("nan"), device="cuda")
        c_ws = torch.full((M, ldc), float("nan"), device="cuda")
        need = dig.bigemm_workspace_bytes(M, N, K, S)
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")

        def run_static():
            dig.bigemm_run_splitk_static(Ad, Bd, c_static, M, N, K, lda, ldb, ldc, S)
            assert dig.bigemm_last_launch_count() == 2

        def run_workspace():
            dig.bigemm_run(Ad, Bd, c_ws, M, N, K, lda, ldb, ldc, S, ws, need)

        if order == "static_first":
            run_static()
            run_workspace()
        else:
            run_workspace()
            run_static()
        torch.cuda.synchronize()
        Cref, D = oracle_rows(A, B, M, N, K)
        got = to_f64(c_static[:, :N])
        check_tolerance(got, to_f64(c_ws[:, :N]), D, False, "static vs workspace M=%d" % M)
        check_tolerance(got, Cref, D, False, "static vs oracle M=%d" % M)
        assert torch.equal(c_static[:, :N].contiguous().view(torch.int32),
                           c_ws[:, :N].contiguous().view(torch.int32))
        assert torch.isnan(c_static[:, N:]).all()
    assert dig.bigemm_device_status(reset=True) == 0


def test_static_scratch_rejects_products_past_its_size(builtin_scratch):
    M, N, K, S = 512, 4096, 4096, 8             # needs 64 MiB of split-K scratch
    assert not dig.bigemm_split_is_folded(M, N, K, S)   # 64 tiles: the workspace path
    assert dig.bigemm_workspace_bytes(M, N, K, S) > dig.STATIC_SCRATCH_BYTES
    a = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    b = torch.zeros((K, N), dtype=torch.bfloat16, device="cuda")
    c = torch.full((M, N), float("nan"), device="cuda")
    st = dig.bigemm_run_splitk_static(a, b, c, M, N, K, K, N, N, S, check=False)
    assert st == 7 and "STATIC_LIMIT" in dig.bigemm_status_string(st)
    assert dig.bigemm_last_launch_count() == 0
    torch.cuda.synchronize()
    assert torch.isnan(c).all()
    # without a split it needs no scratch at all
    dig.bigemm_run_splitk_static(a, b, c, M, N, K, K, N, N, 1)
    torch.cuda.synchronize()
    assert torch.equal(c, torch.zeros_like(c))
    assert np.isfinite(c.cpu().numpy()).all()
