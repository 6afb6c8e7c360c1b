"""GPU: folded split-K.  A split product whose whole tiles already fill the
GPU (bigemm_split_is_folded) has each CTA compute its tile's S segment
partials one after another and add them in the order 0..S-1, instead of
writing them to the workspace for the reduction kernel.  Both ways form every
sum the same way, so the bits must agree: with the explicit two-kernel path
at the same M (bigemm_run_partial + bigemm_splitk_reduce), and with rows
computed in small batches, which never fold.  (Tencent AI-infra article
"腾讯エンジニア：大規模モデルの出力を確定させるための AI インフラ手法": "Split-K"
fixes the segment order; "Batch Invariance の由来" forbids a split that
depends on the batch -- here S stays a function of K while the way it is
executed changes with M.)"""
import pytest
import torch

import deterministic_invariant_gemm_gb300 as dig
import oracle
import workloads
from gemm_check import (bits_equal, canary_intact, check_tolerance, device_matrix, expected_launches,
                        round_up, run_gemm, to_f64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device(cuda_device):
    dig.load()
    yield
    assert dig.bigemm_device_status(reset=True) == 0


def two_kernel_path(A, B, M, N, K, S, bf16_out):
    """The same product through the workspace: partial kernel, then reduction
    (A, B on the CPU; rows padded to the 16-byte multiples the ABI wants)."""
    lda, ldb = round_up(K, 8), round_up(N, 8)
    Ad, Bd = device_matrix(A, lda), device_matrix(B, ldb)
    s_eff = dig.bigemm_effective_split_k(K, S)
    need = dig.bigemm_partial_workspace_bytes(M, N, K, S)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    dig.bigemm_run_partial(Ad, Bd, M, N, K, lda, ldb, S, ws, need)
    ldc = round_up(N, 8)
    C = torch.empty((M, ldc), dtype=torch.bfloat16 if bf16_out else torch.float32, device="cuda")
    dig.bigemm_splitk_reduce(ws, s_eff, M, N, C, ldc, bf16_out)
    assert dig.bigemm_last_launch_count() == 1
    return C[:, :N]


@pytest.mark.parametrize("M,N,K,S", [
    (1024, 4096, 4096, 8),       # a prefill-sized batch at the decode shapes' K and split
    (1000, 4100, 4000, 8),       # ragged M, N and K: 8 x 17 tiles, 63 K blocks
    (2048, 2048, 8192, 16),      # exactly FOLD_MIN_TILES tiles
    (256, 32768, 2048, 3),       # two tile rows, 128 tile columns; 3 segments of 11, 11, 10 blocks
    (4096, 4096, 4096, 0),       # the K-only default split (8)
])
@pytest.mark.parametrize("bf16_out", [False, True])
def test_fold_equals_the_two_kernel_path(M, N, K, S, bf16_out):
    assert dig.bigemm_split_is_folded(M, N, K, S)
    assert dig.bigemm_workspace_bytes(M, N, K, S) == 0
    A, B = workloads.pair(M, N, K, M + N + K)
    C, buf = run_gemm(A, B, M, N, K, S, bf16_out)
    assert dig.bigemm_last_launch_count() == 1
    assert canary_intact(buf, M, N)
    ref = two_kernel_path(A, B, M, N, K, S, bf16_out)
    torch.cuda.synchronize()
    assert bits_equal(C, ref)
    rows = [0, 1, M // 2, M - 1]
    Cref, D = oracle.gemm_rows(A, B, M, N, K, rows=rows)
    check_tolerance(to_f64(C[torch.tensor(rows, device="cuda")]), Cref, D, bf16_out,
                    "folded M=%d N=%d K=%d S=%d" % (M, N, K, S))


def test_folded_rows_match_small_batches():
    """Rows of a folded 1024-row product equal the same rows computed at
    M = 1, 7 and 64 (workspace path), bit for bit."""
    M, N, K, S = 1024, 4096, 4096, 8
    A, B = workloads.pair(M, N, K, 91, a_std=1.0, b_std=0.02)
    A, B = A.cuda(), B.cuda()
    full = dig.matmul(A, B, split_k=S)
    assert dig.bigemm_last_launch_count() == 1
    for m in (1, 7, 64):
        assert not dig.bigemm_split_is_folded(m, N, K, S)
        for off in (0, 129, M - m):
            part = dig.matmul(A[off:off + m].contiguous(), B, split_k=S)
            assert dig.bigemm_last_launch_count() == expected_launches(m, N, K, S)
            assert bits_equal(part, full[off:off + m]), (m, off)


def test_fold_bit_stable_over_10_runs():
    A, B = workloads.pair(2048, 4096, 4096, 5)
    A, B = A.cuda(), B.cuda()
    first = dig.matmul(A, B, split_k=8)
    for _ in range(9):
        assert bits_equal(dig.matmul(A, B, split_k=8), first)


@pytest.mark.parametrize("bf16_out", [False, True])
def test_folded_linear_with_bias(bf16_out):
    """The linear layer: bias added after the folded sum, as the reduction
    kernel adds it after the workspace sum."""
    M, N, K, S = 1024, 6144, 4096, 8
    A = workloads.normal_bf16((M, K), 61)
    W = workloads.normal_bf16((N, K), 62, 0.02)
    b = workloads.normal_bf16((N,), 63)
    Ad, Wd, bd = A.cuda(), W.cuda(), b.cuda()
    dt = torch.bfloat16 if bf16_out else torch.float32
    assert dig.bigemm_split_is_folded(M, N, K, S)
    full = dig.linear(Ad, Wd, bd, out_dtype=dt, split_k=S)
    for lo, hi in ((0, 16), (500, 564), (1023, 1024)):
        part = dig.linear(Ad[lo:hi].contiguous(), Wd, bd, out_dtype=dt, split_k=S)
        assert bits_equal(part, full[lo:hi]), (lo, hi)
    rows = [0, 511, 1023]
    Cref, D = oracle.linear_rows(A, W, b, M, N, K, rows=rows)
    check_tolerance(to_f64(full[torch.tensor(rows, device="cuda")]), Cref, D, bf16_out,
                    "folded linear")


def test_folded_fp8_linear_with_scale_and_bias():
    M, N, K, S = 1024, 4096, 8192, 8
    g = workloads.generator(71)
    A = torch.randn(M, K, generator=g).to(torch.float8_e4m3fn)
    W = (torch.randn(N, K, generator=g) * 0.05).to(torch.float8_e4m3fn)
    b = workloads.normal_bf16((N,), 72)
    Ad, Wd, bd = A.cuda(), W.cuda(), b.cuda()
    assert dig.bigemm_fp8_effective_split_k(K, S) == 8
    assert dig.bigemm_fp8_workspace_bytes(M, N, K, S) == 0
    full = dig.linear_fp8(Ad, Wd, 0.75, bd, split_k=S)
    for lo, hi in ((0, 1), (300, 340), (1000, 1024)):
        part = dig.linear_fp8(Ad[lo:hi].contiguous(), Wd, 0.75, bd, split_k=S)
        assert bits_equal(part, full[lo:hi]), (lo, hi)
    rows = [0, 700, 1023]
    Cref, D = oracle.linear8_rows(A, W, oracle.FMT_E4M3, oracle.FMT_E4M3, M, N, K, 0.75, b, rows=rows)
    check_tolerance(to_f64(full[torch.tensor(rows, device="cuda")]), Cref, D, False, "folded fp8")


def test_static_entry_point_folds_without_scratch():
    """A 1024 x 4096 split product would need 128 MiB of split-K scratch; folded
    it needs none, so the built-in-array entry point accepts it."""
    M, N, K, S = 1024, 4096, 4096, 8
    assert dig.bigemm_workspace_bytes(M, N, K, S) == 0
    A, B = workloads.pair(M, N, K, 81)
    A, B = A.cuda(), B.cuda()
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    dig.bigemm_run_splitk_static(A, B, C, M, N, K, K, N, N, S)
    ref = dig.matmul(A, B, split_k=S)
    torch.cuda.synchronize()
    assert bits_equal(C, ref)
