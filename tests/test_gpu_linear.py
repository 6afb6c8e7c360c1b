"""GPU parity and invariance of the batch-invariant linear layer
(bigemm_linear: C = A W^T + bias, W [N, K] in the layout linear layers keep),
against the binary64 oracle (oracle.linear_rows).  Shapes include the pages'
worked example of a fused QKV projection, N = 6144, K = 4096 (Tencent
AI-infra article, "演算子チューニング")."""
import numpy as np
import pytest
import torch

import deterministic_invariant_gemm_gb300 as dig
import oracle
import workloads
from gemm_check import (bits_equal, canary_intact, check_tolerance, device_matrix, output_buffer,
                        round_up, to_f64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device(cuda_device):
    dig.load()
    yield
    assert dig.bigemm_device_status(reset=True) == 0


def run_linear(A, W, b, M, N, K, split_k=1, bf16_out=False, extra_rows=3):
    lda, ldw = round_up(max(K, 1), 8), round_up(max(K, 1), 8)
    ldc = round_up(max(N, 1), 8 if bf16_out else 4)
    Ad = device_matrix(A, lda)
    Wd = device_matrix(W, ldw)
    bd = None if b is None else b.cuda()
    Cbuf = output_buffer(M, N, ldc, bf16_out, extra_rows)
    need = dig.bigemm_workspace_bytes(M, N, K, split_k)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda") if need else None
    dig.bigemm_linear(Ad, Wd, bd, Cbuf, M, N, K, lda, ldw, ldc, split_k, bf16_out, ws, need)
    torch.cuda.synchronize()
    return Cbuf[:M, :N], Cbuf


def case(M, N, K, seed, bias=True):
    A = workloads.normal_bf16((M, K), seed)
    W = workloads.normal_bf16((N, K), seed + 1, 0.02)
    b = workloads.normal_bf16((N,), seed + 2) if bias else None
    return A, W, b


@pytest.mark.parametrize("M,N,K,splits", [
    (64, 256, 512, (1, 4)),
    (300, 600, 1000, (1, 3)),
    (7, 13, 24, (1,)),
    (16, 4096, 4096, (8,)),
    (32, 6144, 4096, (1, 8)),        # fused QKV of the pages' Llama-3-8B example
])
@pytest.mark.parametrize("bf16_out", [False, True])
@pytest.mark.parametrize("bias", [True, False])
def test_linear_parity(M, N, K, splits, bf16_out, bias):
    A, W, b = case(M, N, K, 10 * M + N + K, bias)
    Cref, D = oracle.linear_rows(A, W, b, M, N, K)
    for s in splits:
        C, buf = run_linear(A, W, b, M, N, K, s, bf16_out)
        check_tolerance(to_f64(C), Cref, D, bf16_out, "linear M=%d N=%d K=%d S=%d" % (M, N, K, s))
        assert canary_intact(buf, M, N)


def test_linear_rows_invariant_across_batches():
    N, K = 4096, 4096
    A, W, b = case(200, N, K, 5)
    Wd, bd = W.cuda(), b.cuda()
    for S in (1, 8):
        full = dig.linear(A.cuda(), Wd, bd, split_k=S)
        for lo, hi in ((0, 1), (5, 12), (63, 64), (100, 164), (127, 129), (199, 200)):
            part = dig.linear(A[lo:hi].contiguous().cuda(), Wd, bd, split_k=S)
            assert bits_equal(part, full[lo:hi]), (S, lo, hi)
        again = dig.linear(A.cuda(), Wd, bd, split_k=S)
        assert bits_equal(again, full)
    torch.cuda.synchronize()


def test_linear_empty_k_gives_the_bias():
    M, N = 5, 40
    A = torch.zeros(M, 0, dtype=torch.bfloat16)
    W = torch.zeros(N, 0, dtype=torch.bfloat16)
    b = workloads.normal_bf16((N,), 9)
    for bf16_out in (False, True):
        C, buf = run_linear(A, W, b, M, N, 0, 1, bf16_out)
        want = b.float().expand(M, N)
        assert torch.equal(C.float().cpu(), want)
        assert canary_intact(buf, M, N)


def test_linear_matches_matmul_on_the_transposed_weight():
    """Both entry points compute A W^T within tolerance; whether the bits also
    agree (the weight is read K-major here, N-major there) is reported."""
    M, N, K = 64, 1024, 2048
    A, W, _ = case(M, N, K, 77, bias=False)
    Cref, D = oracle.linear_rows(A, W, None, M, N, K)
    Ad, Wd = A.cuda(), W.cuda()
    lin = dig.linear(Ad, Wd)
    mm = dig.matmul(Ad, Wd.t().contiguous())
    torch.cuda.synchronize()
    check_tolerance(to_f64(lin), Cref, D, False, "linear")
    check_tolerance(to_f64(mm), Cref, D, False, "matmul on W^T")
    same = bits_equal(lin, mm)
    print("\n[linear vs matmul(W^T)] bitwise equal: %s" % same)
