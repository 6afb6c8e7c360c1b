"""GPU: the largest shapes -- a batch of more than 2^20 rows, and a K of more
than 2^20 -- where row offsets, tile counts and K-block counts leave the range
small tests reach.  Sampled rows are held to the binary64 oracle, and a row
computed alone must match its copy inside the big batch bit for bit (Tencent
AI-infra article, "Batch Invariance の由来")."""
import pytest
import torch

import deterministic_invariant_gemm_gb300 as dig
import oracle
import workloads
from gemm_check import bits_equal, check_tolerance, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device(cuda_device):
    dig.load()
    yield
    assert dig.bigemm_device_status(reset=True) == 0


def test_more_than_a_million_rows():
    M, N, K = (1 << 20) + 37, 512, 128          # 8193 tile rows, 2 GiB of FP32 output
    g = workloads.generator(4242)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = torch.randn(K, N, generator=g).to(torch.bfloat16)
    Ad, Bd = A.cuda(), B.cuda()
    C = dig.matmul(Ad, Bd)
    torch.cuda.synchronize()
    rows = [0, 127, 128, 1 << 19, (1 << 20) - 1, 1 << 20, M - 1]
    Cref, D = oracle.gemm_rows(A, B, M, N, K, rows=rows)
    check_tolerance(to_f64(C[torch.tensor(rows, device="cuda")]), Cref, D, False, "M > 2^20")
    for r in (0, 1 << 20, M - 1):
        one = dig.matmul(Ad[r:r + 1].contiguous(), Bd)
        assert bits_equal(one, C[r:r + 1]), r
    del C
    torch.cuda.empty_cache()


@pytest.mark.parametrize("split_k", [0, 1])
def test_k_beyond_a_million(split_k):
    M, N, K = 16, 256, (1 << 20) + 40            # 16385 K blocks, the last one ragged
    A, B = workloads.pair(M, N, K, 4343)
    Ad, Bd = A.cuda(), B.cuda()
    C = dig.matmul(Ad, Bd, split_k=split_k)
    torch.cuda.synchronize()
    Cref, D = oracle.gemm_rows(A, B, M, N, K)
    check_tolerance(to_f64(C), Cref, D, False, "K > 2^20, split_k=%d" % split_k)
    one = dig.matmul(Ad[7:8].contiguous(), Bd, split_k=split_k)
    assert bits_equal(one, C[7:8])
