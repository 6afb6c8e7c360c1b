"""GPU parity and invariance of the 8-bit float linear layer
(bigemm_linear_fp8: C = scale * (A W^T) + bias, A and W in E4M3 or E5M2)
against the binary64 oracle (oracle.linear8_rows).  The pages benchmark FP8
matrix products (cuTile article, "TileGymで行列積ベンチマーク", float8_e5m2);
here they get the same deterministic, batch-invariant treatment as BF16."""
import numpy as np
import pytest
import torch

import deterministic_invariant_gemm_gb300 as dig
import oracle
import workloads
from gemm_check import bits_equal, canary_intact, check_tolerance, output_buffer, round_up, to_f64

pytestmark = pytest.mark.gpu

TD = {oracle.FMT_E4M3: torch.float8_e4m3fn, oracle.FMT_E5M2: torch.float8_e5m2}
LIB = {oracle.FMT_E4M3: dig.FP8_E4M3, oracle.FMT_E5M2: dig.FP8_E5M2}


@pytest.fixture(scope="module", autouse=True)
def _device(cuda_device):
    dig.load()
    yield
    assert dig.bigemm_device_status(reset=True) == 0


def fp8_inputs(M, N, K, seed, fa, fb, a_std=1.0, w_std=0.05):
    g = workloads.generator(seed)
    A = (torch.randn(M, K, generator=g) * a_std).to(TD[fa])
    W = (torch.randn(N, K, generator=g) * w_std).to(TD[fb])
    return A, W


def padded_device(t, ld):
    rows, cols = t.shape
    buf = torch.zeros((rows, ld), dtype=torch.uint8, device="cuda")
    buf[:, :cols] = t.view(torch.uint8).cuda()
    return buf.view(t.dtype)


def run_fp8(A, W, fa, fb, scale, b, M, N, K, split_k=1, bf16_out=False):
    lda = ldw = round_up(max(K, 1), 16)
    ldc = round_up(max(N, 1), 8 if bf16_out else 4)
    Ad, Wd = padded_device(A, lda), padded_device(W, ldw)
    bd = None if b is None else b.cuda()
    Cbuf = output_buffer(M, N, ldc, bf16_out)
    need = dig.bigemm_fp8_workspace_bytes(M, N, K, split_k)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda") if need else None
    dig.bigemm_linear_fp8(Ad, Wd, LIB[fa], LIB[fb], scale, bd, Cbuf, M, N, K, lda, ldw, ldc, split_k,
                          bf16_out, ws, need)
    torch.cuda.synchronize()
    return Cbuf[:M, :N], Cbuf


@pytest.mark.parametrize("M,N,K,splits", [
    (64, 256, 512, (1, 2)),
    (300, 600, 1000, (1, 3)),        # ragged everywhere; K not a multiple of 128
    (16, 4096, 4096, (1, 8)),        # decode-shaped
    (7, 40, 96, (1,)),               # K shorter than one 128-element block
])
@pytest.mark.parametrize("fa,fb", [(oracle.FMT_E4M3, oracle.FMT_E4M3),
                                   (oracle.FMT_E5M2, oracle.FMT_E4M3),
                                   (oracle.FMT_E4M3, oracle.FMT_E5M2)])
def test_fp8_linear_parity(M, N, K, splits, fa, fb):
    A, W = fp8_inputs(M, N, K, 3 * M + N + K, fa, fb)
    b = workloads.normal_bf16((N,), 5)
    for scale, bias, bf16_out in ((1.0, None, False), (0.8125, b, False), (2.0, b, True)):
        Cref, D = oracle.linear8_rows(A, W, fa, fb, M, N, K, scale, bias)
        for s in splits:
            C, buf = run_fp8(A, W, fa, fb, scale, bias, M, N, K, s, bf16_out)
            check_tolerance(to_f64(C), Cref, D, bf16_out,
                            "fp8 M=%d N=%d K=%d S=%d scale=%g" % (M, N, K, s, scale))
            assert canary_intact(buf, M, N)


def test_fp8_small_integers_bit_exact():
    """|values| <= 8 are exact in both formats; every partial sum is an
    integer below 2^24, so the GPU result must equal the oracle exactly."""
    M, N, K = 96, 320, 2048
    g = workloads.generator(17)
    ai = torch.randint(-8, 9, (M, K), generator=g).float()
    wi = torch.randint(-8, 9, (N, K), generator=g).float()
    for fa, fb in ((oracle.FMT_E4M3, oracle.FMT_E4M3), (oracle.FMT_E5M2, oracle.FMT_E4M3)):
        A, W = ai.to(TD[fa]), wi.to(TD[fb])
        Cref, _ = oracle.linear8_rows(A, W, fa, fb, M, N, K)
        assert np.array_equal(Cref, (ai.double() @ wi.double().T).numpy())
        for s in (1, 4):
            C, _ = run_fp8(A, W, fa, fb, 1.0, None, M, N, K, s)
            assert np.array_equal(to_f64(C), Cref)


def test_fp8_rows_invariant_across_batches():
    N, K = 2048, 4096
    fa = fb = oracle.FMT_E4M3
    A, W = fp8_inputs(192, N, K, 23, fa, fb)
    b = workloads.normal_bf16((N,), 24).cuda()
    Ad, Wd = A.cuda(), W.cuda()
    for S in (1, 8):
        full = dig.linear_fp8(Ad, Wd, 0.5, b, split_k=S)
        Cref, D = oracle.linear8_rows(A, W, fa, fb, 192, N, K, 0.5, b.cpu(), rows=[0, 100, 191])
        check_tolerance(to_f64(full[[0, 100, 191]]), Cref, D, False, "fp8 invariance reference")
        for lo, hi in ((0, 1), (3, 19), (100, 164), (127, 129), (191, 192)):
            part = dig.linear_fp8(Ad[lo:hi].contiguous(), Wd, 0.5, b, split_k=S)
            assert bits_equal(part, full[lo:hi]), (S, lo, hi)
        assert bits_equal(dig.linear_fp8(Ad, Wd, 0.5, b, split_k=S), full)


def test_fp8_square_2048_sampled():
    M = N = K = 2048
    fa, fb = oracle.FMT_E4M3, oracle.FMT_E4M3
    A, W = fp8_inputs(M, N, K, 31, fa, fb, 1.0, 1.0)
    rows = [0, 127, 128, 1023, 2047]
    Cref, D = oracle.linear8_rows(A, W, fa, fb, M, N, K, rows=rows)
    C, _ = run_fp8(A, W, fa, fb, 1.0, None, M, N, K)
    check_tolerance(to_f64(C[torch.tensor(rows, device="cuda")]), Cref, D, False, "fp8 2048")


def test_fp8_argument_checks():
    a = torch.zeros(8, 16, dtype=torch.uint8, device="cuda")
    c = torch.zeros(8, 8, device="cuda")
    # unknown format
    assert dig.bigemm_linear_fp8(a, a, 2, 0, 1.0, None, c, 8, 8, 16, 16, 16, 8, 1, 0,
                                 check=False) == 1
    # fp8 rows must be 16-byte multiples
    assert dig.bigemm_linear_fp8(a, a, 0, 0, 1.0, None, c, 8, 8, 8, 8, 16, 8, 1, 0,
                                 check=False) == 2
    assert dig.bigemm_fp8_effective_split_k(4096, 8) == 8
    assert dig.bigemm_fp8_effective_split_k(4096, 33) == 0      # 32 blocks of 128


@pytest.mark.parametrize("M,N,K,S", [
    (64, 256, 512, 1),
    (300, 600, 992, 3),          # ragged rows, columns and K (not a multiple of 128)
    (7, 45, 96, 1),              # N not a multiple of 4: the transpose's byte edge
    (1024, 8192, 4096, 4),       # folded split on CTA pairs
])
@pytest.mark.parametrize("fa,fb", [(oracle.FMT_E4M3, oracle.FMT_E4M3), (oracle.FMT_E5M2, oracle.FMT_E4M3)])
def test_fp8_with_b_k_by_n_equals_the_weight_layout(M, N, K, S, fa, fb):
    """bigemm_run_fp8 takes B [K, N] (copied transposed into the workspace):
    the bits of bigemm_linear_fp8 with W = B^T, rows computed alone give the
    same bits, and sampled rows meet the oracle's tolerance."""
    A, W = fp8_inputs(M, N, K, 61 + M + N, fa, fb)
    B = W.t().contiguous()                                    # [K, N]
    b = workloads.normal_bf16((N,), 62).cuda()
    Ad, Bd, Wd = A.cuda(), B.cuda(), W.cuda()
    if N % 16:
        # the [K, N] rows need a 16-byte multiple: pad the leading dimension
        ldb = round_up(N, 16)
        Bp = torch.zeros((K, ldb), dtype=torch.uint8, device="cuda")
        Bp[:, :N] = Bd.view(torch.uint8)
        Bd = Bp.view(B.dtype)[:, :N]
    ldc = round_up(N, 4)                                   # fp32 rows: 16-byte multiples
    out = lambda m: torch.empty((m, ldc), dtype=torch.float32, device="cuda")[:, :N]
    got = dig.matmul_fp8(Ad, Bd, 0.5, b, split_k=S, out=out(M))
    assert dig.bigemm_last_launch_count() >= 2             # the transpose, then the product
    want = dig.linear_fp8(Ad, Wd, 0.5, b, split_k=S, out=out(M))
    torch.cuda.synchronize()
    assert bits_equal(got, want)
    for r in (0, M - 1):
        one = dig.matmul_fp8(Ad[r:r + 1].contiguous(), Bd, 0.5, b, split_k=S, out=out(1))
        assert bits_equal(one, got[r:r + 1]), r
    rows = sorted({0, M // 2, M - 1})
    Cref, D = oracle.linear8_rows(A, W, fa, fb, M, N, K, 0.5, b.cpu(), rows=rows)
    check_tolerance(to_f64(got[torch.tensor(rows, device="cuda")]), Cref, D, False, "fp8 B [K, N]")


def test_fp8_b_k_by_n_workspace_and_argument_checks():
    M, N, K = 40, 48, 256
    up = lambda x: (x + 255) // 256 * 256
    assert dig.bigemm_fp8_kn_workspace_bytes(M, N, K, 1) == up(N * K)
    assert dig.bigemm_fp8_kn_workspace_bytes(M, N, 300, 1) == up(N * 304)
    assert dig.bigemm_fp8_kn_workspace_bytes(M, N, K, 2) == up(N * K) + dig.bigemm_fp8_workspace_bytes(M, N, K, 2)
    a = torch.zeros((M, K), dtype=torch.uint8, device="cuda")
    bmat = torch.zeros((K, N), dtype=torch.uint8, device="cuda")
    c = torch.empty((M, N), dtype=torch.float32, device="cuda")
    # no workspace (WORKSPACE), a bad format and ldb < N (ARG), ldb not a
    # multiple of 16 (ALIGN); nothing is launched
    assert dig.bigemm_run_fp8(a, bmat, 0, 0, 1.0, None, c, M, N, K, K, N, N, 1, 0, None, 0,
                              check=False) == 3
    assert dig.bigemm_run_fp8(a, bmat, 2, 0, 1.0, None, c, M, N, K, K, N, N, 1, 0, None, 0,
                              check=False) == 1
    assert dig.bigemm_run_fp8(a, bmat, 0, 0, 1.0, None, c, M, N, K, K, N - 8, N, 1, 0, None, 0,
                              check=False) == 1
    assert dig.bigemm_run_fp8(a, bmat, 0, 0, 1.0, None, c, M, N, K, K, N + 8, N, 1, 0, None, 0,
                              check=False) == 2
    assert dig.bigemm_last_launch_count() == 0
