"""GPU parity: the CUDA path, called through the C ABI, against the binary64
CPU oracle on the same seeded inputs.

Sizes: small and ragged shapes that span several 128 x 256 tiles and several
64-wide K blocks with ragged tails (whole outputs compared), the five
workload shapes at full size (whole outputs where the oracle takes seconds,
sampled rows otherwise), exact-arithmetic regimes compared bitwise, and edge
cases (K = 0, M = 0, K < 64, single row/column, padded leading dimensions
with NaN canaries in the padding and around the output).
"""
import numpy as np
import pytest
import torch

import deterministic_invariant_gemm_gb300 as dig
import oracle
import workloads
from gemm_check import (bits_equal, canary_intact, check_tolerance, device_matrix, expected_launches,
                        oracle_rows, round_up, run_gemm, sample_rows, to_f64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device(cuda_device):
    dig.load()
    yield
    assert dig.bigemm_device_status(reset=True) == 0, "a kernel reported a wait timeout"


# ------------------------------------------------------------ small / ragged --

SHAPES = [
    # M, N, K, splits
    (64, 256, 512, (1, 2, 4, 8)),          # the small workload
    (300, 600, 1000, (1, 3, 16)),          # 3 x 3 tiles, ragged everywhere
    (129, 257, 65, (1, 2)),                # one row / column / k past a tile
    (1, 1, 1, (1,)),
    (7, 13, 24, (1,)),                     # K shorter than one block
    (5, 40, 640, (7,)),                    # split 7 -> 5 non-empty segments
    (256, 512, 4096, (1, 8, 64)),          # one block per segment at 64
    (1000, 300, 333, (1, 5)),
]


@pytest.mark.parametrize("M,N,K,splits", SHAPES)
@pytest.mark.parametrize("bf16_out", [False, True])
def test_parity_small_and_ragged(M, N, K, splits, bf16_out):
    A, B = workloads.pair(M, N, K, 31 + M + N + K)
    Cref, D = oracle_rows(A, B, M, N, K)
    for s in splits:
        C, buf = run_gemm(A, B, M, N, K, split_k=s, bf16_out=bf16_out)
        check_tolerance(to_f64(C), Cref, D, bf16_out, "M=%d N=%d K=%d S=%d bf16=%d" % (M, N, K, s, bf16_out))
        assert canary_intact(buf, M, N), "wrote outside C"


@pytest.mark.parametrize("M,N,K", [(96, 300, 4096), (130, 256, 2048), (1, 512, 4096)])
@pytest.mark.parametrize("split", [1, 4, 0])
def test_integer_inputs_bit_exact(M, N, K, split):
    """Entries in [-8, 8]: every partial sum is an integer below 2^24, exact in
    FP32 in any order, so the GPU must equal the oracle bit for bit."""
    A, B = workloads.pair(M, N, K, 900 + K, dist="int")
    Cref, _ = oracle_rows(A, B, M, N, K)
    C, _ = run_gemm(A, B, M, N, K, split_k=split)
    assert np.array_equal(to_f64(C), Cref)


def test_bf16_slices_are_exact_in_fp32():
    """cuTile/Ozaki article (techplay.jp, "最適化後の結果"): BF16 slices sharing
    one power-of-two scale, K = 128: 16 + 7 <= 24 bits, so the tensor-core FP32
    accumulation is exact and must equal the oracle bit for bit."""
    M, N, K = 256, 512, 128
    A = workloads.scaled_slices_bf16((M, K), 61, -9)
    B = workloads.scaled_slices_bf16((K, N), 62, 4)
    Cref, _ = oracle_rows(A, B, M, N, K)
    assert np.array_equal(Cref.astype(np.float32).astype(np.float64), Cref)
    C, _ = run_gemm(A, B, M, N, K)
    assert np.array_equal(to_f64(C), Cref)


def test_padded_leading_dimensions():
    M, N, K = 200, 300, 700
    A, B = workloads.pair(M, N, K, 71)
    Cref, D = oracle_rows(A, B, M, N, K)
    for s in (1, 4):
        C, buf = run_gemm(A, B, M, N, K, split_k=s, lda=768, ldb=320, ldc=340)
        check_tolerance(to_f64(C), Cref, D, False, "padded S=%d" % s)
        assert canary_intact(buf, M, N)
        C2, buf2 = run_gemm(A, B, M, N, K, split_k=s, lda=704, ldb=304, ldc=312, bf16_out=True)
        check_tolerance(to_f64(C2), Cref, D, True, "padded bf16 S=%d" % s)
        assert canary_intact(buf2, M, N)


def test_empty_products():
    # K == 0: C is all +0.0 (both output types), the rest untouched
    for bf16 in (False, True):
        A = torch.zeros(5, 0, dtype=torch.bfloat16)
        B = torch.zeros(0, 9, dtype=torch.bfloat16)
        C, buf = run_gemm(A, B, 5, 9, 0, bf16_out=bf16, lda=8, ldb=16)
        assert torch.equal(C.float().cpu(), torch.zeros(5, 9)) and not torch.signbit(C.float()).any()
        assert canary_intact(buf, 5, 9)
    # M == 0 or N == 0: nothing happens at all
    buf = torch.full((4, 8), float("nan"), device="cuda")
    a = torch.zeros(8, 8, dtype=torch.bfloat16, device="cuda")
    dig.bigemm_run(a, a, buf, 0, 8, 8, 8, 8, 8, 1)
    dig.bigemm_run(a, a, buf, 8, 0, 8, 8, 8, 8, 1)
    torch.cuda.synchronize()
    assert torch.isnan(buf).all()
    assert dig.bigemm_last_launch_count() == 0


def test_matmul_wrapper_and_launch_count(cuda_device):
    M, N, K = 100, 320, 2048
    A, B = workloads.pair(M, N, K, 5)
    Cref, D = oracle_rows(A, B, M, N, K)
    Ad, Bd = A.cuda(), B.cuda()
    C = dig.matmul(Ad, Bd, split_k=4)
    assert dig.bigemm_last_launch_count() == expected_launches(M, N, K, 4)
    C1 = dig.matmul(Ad, Bd, split_k=1)
    assert dig.bigemm_last_launch_count() == 1
    torch.cuda.synchronize()
    check_tolerance(to_f64(C), Cref, D, False, "matmul S=4")
    check_tolerance(to_f64(C1), Cref, D, False, "matmul S=1")
    # a B whose row stride is not a multiple of 8 elements is refused up front
    Bbad = workloads.normal_bf16((K, 300), 6).cuda()
    with pytest.raises(ValueError):
        dig.matmul(Ad, Bbad)


# -------------------------------------------------- the reduction, bitwise --

@pytest.mark.parametrize("S", [1, 2, 3, 8, 9, 13, 32])
@pytest.mark.parametrize("bf16_out", [False, True])
def test_splitk_reduce_bit_exact(S, bf16_out):
    """The reduction kernel alone on a synthetic workspace whose partials span
    many binades (so the addition order shows in the bits): it must equal the
    oracle's serial binary32 sum w0 + w1 + ... bit for bit, then one RNE
    rounding to bf16."""
    M, N = 37, 1001
    ld = dig.bigemm_workspace_ld(N)
    g = torch.Generator().manual_seed(100 + S)
    mant = torch.randn(S, M, ld, generator=g, dtype=torch.float32)
    expo = torch.randint(-20, 21, (S, M, ld), generator=g).to(torch.float32)
    W = mant * torch.pow(2.0, expo)
    W[0, 0, :8] = -0.0                       # a lone negative zero survives S == 1
    want = oracle.splitk_reduce_f32(W.numpy())[:, :N]
    ldc = 1008
    Cbuf = torch.full((M + 2, ldc), float("nan"), device="cuda") if not bf16_out else \
        torch.full((M + 2, ldc), 0, dtype=torch.int16, device="cuda").fill_(0x7FC5).view(torch.bfloat16)
    dig.bigemm_splitk_reduce(W.cuda(), S, M, N, Cbuf, ldc, bf16_out)
    torch.cuda.synchronize()
    got = Cbuf[:M, :N].cpu()
    if bf16_out:
        want_bits = oracle.encode_rne(oracle.FMT_BF16, want.astype(np.float64))
        assert np.array_equal(got.view(torch.int16).numpy().view(np.uint16), want_bits)
    else:
        assert np.array_equal(got.numpy().view(np.uint32), want.view(np.uint32))
    assert canary_intact(Cbuf, M, N)


@pytest.mark.parametrize("bf16_out", [False, True])
def test_splitk_reduce_more_groups_than_threads(bf16_out):
    """More four-column groups (80 x 8196) than the reduction launches threads
    for (16 blocks of 128 per SM), so threads take several groups each: still
    the serial binary32 sum of the oracle, bit for bit, and nothing written
    outside C."""
    S, M, N = 3, 80, 32780
    ld = dig.bigemm_workspace_ld(N)
    g = torch.Generator().manual_seed(4242)
    W = torch.randn(S, M, ld, generator=g, dtype=torch.float32) * \
        torch.pow(2.0, torch.randint(-12, 13, (S, M, ld), generator=g).to(torch.float32))
    want = oracle.splitk_reduce_f32(W.numpy())[:, :N]
    ldc = N + 4
    if bf16_out:
        Cbuf = torch.full((M + 2, ldc), 0, dtype=torch.int16, device="cuda").fill_(0x7FC5).view(torch.bfloat16)
    else:
        Cbuf = torch.full((M + 2, ldc), float("nan"), device="cuda")
    dig.bigemm_splitk_reduce(W.cuda(), S, M, N, Cbuf, ldc, bf16_out)
    torch.cuda.synchronize()
    got = Cbuf[:M, :N].cpu()
    if bf16_out:
        want_bits = oracle.encode_rne(oracle.FMT_BF16, want.astype(np.float64))
        assert np.array_equal(got.view(torch.int16).numpy().view(np.uint16), want_bits)
    else:
        assert np.array_equal(got.numpy().view(np.uint32), want.view(np.uint32))
    assert canary_intact(Cbuf, M, N)


def test_partial_kernel_slices_sum_to_result():
    """bigemm_run_partial + bigemm_splitk_reduce == bigemm_run, bitwise."""
    M, N, K, S = 70, 520, 3000, 6
    A, B = workloads.pair(M, N, K, 12)
    lda, ldb = round_up(K, 8), round_up(N, 8)
    Ad, Bd = device_matrix(A, lda), device_matrix(B, ldb)
    nb = dig.bigemm_partial_workspace_bytes(M, N, K, S)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    dig.bigemm_run_partial(Ad, Bd, M, N, K, lda, ldb, S, ws, nb)
    Se = dig.bigemm_effective_split_k(K, S)
    C1 = torch.empty(M, N, device="cuda")
    dig.bigemm_splitk_reduce(ws, Se, M, N, C1, N, 0)
    C2, _ = run_gemm(A, B, M, N, K, split_k=S)
    torch.cuda.synchronize()
    assert bits_equal(C1, C2.contiguous())
    # every slice is itself a partial product over its K segment
    ld = dig.bigemm_workspace_ld(N)
    slices = ws.view(torch.float32)[: Se * M * ld].view(Se, M, ld)[:, :, :N].cpu().double().numpy()
    kb = -(-K // 64)                 # K blocks
    L = -(-kb // S) * 64             # K columns per segment
    for s in range(Se):
        k0, k1 = s * L, min((s + 1) * L, K)
        Cs, Ds = oracle_rows(A[:, k0:k1].contiguous(), B[k0:k1].contiguous(), M, N, k1 - k0)
        check_tolerance(slices[s], Cs, Ds, False, "slice %d" % s)


# ------------------------------------------------------ the five workloads --

def test_workload_small():
    w = workloads.WORKLOADS["small"]
    M, N, K = w["M"], w["N"], w["K"]
    A, B = workloads.pair(M, N, K, workloads.BASE_SEED + w["index"])
    Cref, D = oracle_rows(A, B, M, N, K)
    for s in (1, 0):
        C, _ = run_gemm(A, B, M, N, K, split_k=s)
        check_tolerance(to_f64(C), Cref, D, False, "small S=%d" % s)


def test_workload_decode():
    w = workloads.WORKLOADS["decode"]
    N, K = w["N"], w["K"]
    Mmax = max(w["Ms"])
    A, B = workloads.pair(Mmax, N, K, workloads.BASE_SEED + w["index"], a_std=w["a_std"],
                          b_std=w["b_std"])
    Cref, D = oracle_rows(A, B, Mmax, N, K)
    S = dig.bigemm_default_split_k(K)
    assert S == 8
    for M in w["Ms"]:
        C, _ = run_gemm(A[:M].contiguous(), B, M, N, K, split_k=0)
        check_tolerance(to_f64(C), Cref[:M], D[:M], False, "decode M=%d" % M)


@pytest.mark.parametrize("size", [2048, 4096, 8192])
def test_workload_square(size):
    w = workloads.WORKLOADS["square"]
    M = N = K = size
    A, B = workloads.pair(M, N, K, workloads.BASE_SEED + w["index"] + size, dist="uniform")
    rows = None if size <= 2048 else sample_rows(M, {4096: 128, 8192: 48}[size], seed=size)
    Cref, D = oracle_rows(A, B, M, N, K, rows=rows)
    C, _ = run_gemm(A, B, M, N, K, split_k=1)
    got = to_f64(C) if rows is None else to_f64(C[torch.tensor(rows, device="cuda")])
    check_tolerance(got, Cref, D, False, "square %d" % size)


def test_workload_large_bf16_out():
    w = workloads.WORKLOADS["large"]
    M, N, K = w["M"], w["N"], w["K"]
    A, B = workloads.pair(M, N, K, workloads.BASE_SEED + w["index"])
    rows = sample_rows(M, 16, seed=3)
    Cref, D = oracle_rows(A, B, M, N, K, rows=rows)
    idx = torch.tensor(rows, device="cuda")
    C, _ = run_gemm(A, B, M, N, K, split_k=1, bf16_out=True, extra_rows=1)
    check_tolerance(to_f64(C[idx]), Cref, D, True, "large bf16")
    del C
    torch.cuda.empty_cache()
    C32, _ = run_gemm(A, B, M, N, K, split_k=1, extra_rows=1)
    check_tolerance(to_f64(C32[idx]), Cref, D, False, "large fp32")


@pytest.fixture(scope="module")
def longk_case():
    w = workloads.WORKLOADS["longk"]
    M, N, K = w["M"], w["N"], w["K"]
    A, B = workloads.pair(M, N, K, workloads.BASE_SEED + w["index"])
    Cref, D = oracle_rows(A, B, M, N, K)
    return A, B, Cref, D


@pytest.mark.parametrize("S", [1, 8, 16, 32])
def test_workload_longk(longk_case, S):
    A, B, Cref, D = longk_case
    M, K = A.shape
    N = B.shape[1]
    C, _ = run_gemm(A, B, M, N, K, split_k=S)
    check_tolerance(to_f64(C), Cref, D, False, "longk S=%d" % S)


@pytest.mark.parametrize("S", [8, 32])
def test_workload_longk_atomic_contrast_within_tolerance(longk_case, S):
    """The atomic contrast is still a correct sum (only its bits wander)."""
    A, B, Cref, D = longk_case
    M, K = A.shape
    N = B.shape[1]
    C, _ = run_gemm(A, B, M, N, K, split_k=S, atomic=True)
    check_tolerance(to_f64(C), Cref, D, False, "longk atomic S=%d" % S)
