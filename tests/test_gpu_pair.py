"""GPU: the 2-SM kernel (bigemm_pair_kernel).  A thread-block cluster of two
CTAs computes a 256 x 256 output tile with tcgen05.mma.cta_group::2: each CTA
loads its 128 rows of A and its 128 columns of B, and holds its 128 rows of
the FP32 sum.  The instruction shape changes (M = 256 across two SMs), the
reduction order of an element must not: every comparison here is bit for
bit -- against the 1-SM kernel on the same product (pair mode NEVER), against
the same rows computed in a batch of one (the few-row kernel), and against
the oracle's tolerance.  (Tencent AI-infra article "腾讯エンジニア：大規模モデル
の出力を確定させるための AI インフラ手法", "Tiling" and "Batch Invariance の由来".)"""
import pytest
import torch

import deterministic_invariant_gemm_gb300 as dig
import oracle
import workloads
from gemm_check import bits_equal, canary_intact, check_tolerance, run_gemm, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device(cuda_device):
    dig.load()
    yield
    assert dig.bigemm_device_status(reset=True) == 0


@pytest.fixture(autouse=True)
def _auto_mode():
    """Every test leaves the process in the default mode."""
    yield
    dig.bigemm_set_pair_mode(dig.PAIR_AUTO)


def cdiv(a, b):
    return -(-a // b)


def product(A, B, mode, bf16_out=False, wt=False, bias=None):
    dig.bigemm_set_pair_mode(mode)
    dt = torch.bfloat16 if bf16_out else torch.float32
    if wt:
        C = dig.linear(A, B, bias, out_dtype=dt, split_k=1)
    else:
        C = dig.matmul(A, B, out_dtype=dt, split_k=1)
    torch.cuda.synchronize()
    return C


def test_rule():
    """Eligible: bf16 products of at least 256 rows with 256-wide tiles,
    unsplit or folded.  AUTO takes those whose 256 x 256 tiles fill two waves
    of pairs."""
    cap = dig.bigemm_pair_capacity()
    assert cap >= 1
    dig.bigemm_set_pair_mode(dig.PAIR_AUTO)
    n_two_waves = 256 * cdiv(2 * cap, 16)          # 16 tile rows of 256
    assert dig.bigemm_uses_pair(4096, n_two_waves, 1024, 1) == 1
    assert dig.bigemm_uses_pair(4096, n_two_waves - 256, 1024, 1) == (1 if 16 * (cdiv(2 * cap, 16) - 1) >= 2 * cap else 0)
    assert dig.bigemm_uses_pair(8192, 8192, 8192, 1) == 1
    assert dig.bigemm_uses_pair(2048, 2048, 2048, 1) == 0      # 64 tiles: one wave
    assert dig.bigemm_uses_pair(8192, 8192, 8192, 2) == 1      # a folded split
    assert dig.bigemm_uses_pair(8192, 8192, 8192, 0) == 1      # the default split, 16, folds
    assert dig.bigemm_uses_pair(256, 2048, 4096, 8) == 0       # split, not folded (16 tiles)
    assert dig.bigemm_uses_pair(8192, 8192, 8192, 1, fp8=True) == 1
    assert dig.bigemm_uses_pair(2048, 2048, 2048, 1, fp8=True) == 0
    assert dig.bigemm_uses_pair(255, 65536, 1024, 1) == 0       # fewer than 256 rows
    dig.bigemm_set_pair_mode(dig.PAIR_ALWAYS)
    assert dig.bigemm_uses_pair(256, 256, 128, 1) == 1
    assert dig.bigemm_uses_pair(255, 256, 128, 1) == 0
    assert dig.bigemm_uses_pair(256, 256, 65536, 1) == 0        # narrow tiles (long K, one tile)
    assert dig.bigemm_uses_pair(4096, 4096, 4096, 0) == 1       # the default split 8 folds
    assert dig.bigemm_uses_pair(256, 4096, 4096, 8) == 0        # split, 64 tiles: not folded
    dig.bigemm_set_pair_mode(dig.PAIR_NEVER)
    assert dig.bigemm_uses_pair(8192, 8192, 8192, 1) == 0
    with pytest.raises(ValueError):
        dig.bigemm_set_pair_mode(3)
    assert dig.bigemm_set_pair_mode(dig.PAIR_AUTO) == dig.PAIR_NEVER


@pytest.mark.parametrize("M,N,K", [
    (256, 256, 128),             # one pair tile, two K blocks
    (256, 256, 1024),
    (257, 264, 64),              # 511 rows of the second pair tile past M; a 8-column third tile
    (300, 520, 776),             # ragged M (CTA 1 of the second tile row has no rows), N and K
    (512, 768, 1000),            # K ends in a partial block
    (1024, 1024, 1024),
    (768, 1280, 1984),
    (4096, 4096, 4096),          # the default rule's choice, 3.4 waves of pairs
])
@pytest.mark.parametrize("bf16_out", [False, True])
def test_equals_the_1sm_kernel_bit_for_bit(M, N, K, bf16_out):
    A = workloads.normal_bf16((M, K), 3 * M + K).cuda()
    B = workloads.normal_bf16((K, N), 5 * N + K, 0.05).cuda()
    pair = product(A, B, dig.PAIR_ALWAYS, bf16_out)
    assert dig.bigemm_last_launch_count() == 1
    single = product(A, B, dig.PAIR_NEVER, bf16_out)
    assert bits_equal(pair, single)


@pytest.mark.parametrize("M,N,K,S", [
    (4096, 4096, 4096, 8),       # the default split of K = 4096, folded; AUTO takes pairs
    (1024, 8192, 2048, 4),       # 256 tiles of 128 x 256: folds; 4 x 32 pair tiles
    (300, 32768, 1000, 3),       # ragged rows and K (16 blocks in segments of 6, 6, 4)
    (512, 33024, 8192, 16),      # 16 segments; a ragged last tile column (N = 129 x 256)
])
@pytest.mark.parametrize("bf16_out", [False, True])
def test_folded_split_equals_the_1sm_fold_and_the_workspace_path(M, N, K, S, bf16_out):
    """A folded split on pairs: each CTA's epilogue adds the segment partials
    in the order 0..S-1 -- the bits of the 1-SM fold and of the two-kernel
    path (partial kernel + reduction kernel, run explicitly)."""
    assert dig.bigemm_split_is_folded(M, N, K, S)
    A = workloads.normal_bf16((M, K), M + S).cuda()
    B = workloads.normal_bf16((K, N), N + S, 0.05).cuda()
    dt = torch.bfloat16 if bf16_out else torch.float32
    dig.bigemm_set_pair_mode(dig.PAIR_ALWAYS)
    assert dig.bigemm_uses_pair(M, N, K, S) == 1
    pair = dig.matmul(A, B, out_dtype=dt, split_k=S)
    assert dig.bigemm_last_launch_count() == 1
    dig.bigemm_set_pair_mode(dig.PAIR_NEVER)
    single = dig.matmul(A, B, out_dtype=dt, split_k=S)
    torch.cuda.synchronize()
    assert bits_equal(pair, single)
    s_eff = dig.bigemm_effective_split_k(K, S)
    need = dig.bigemm_partial_workspace_bytes(M, N, K, S)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    dig.bigemm_run_partial(A, B, M, N, K, K, N, S, ws, need)
    C = torch.empty((M, N), dtype=dt, device="cuda")
    dig.bigemm_splitk_reduce(ws, s_eff, M, N, C, N, bf16_out)
    torch.cuda.synchronize()
    assert bits_equal(pair, C)


@pytest.mark.parametrize("M,N,K,S", [
    (256, 512, 1024, 1),         # one K block of 128 elements per 128 bytes
    (300, 600, 992, 1),          # ragged rows, columns and K (not a multiple of 128)
    (1024, 8192, 4096, 4),       # folded split
])
@pytest.mark.parametrize("fa,fb", [(dig.FP8_E4M3, dig.FP8_E4M3), (dig.FP8_E5M2, dig.FP8_E4M3)])
@pytest.mark.parametrize("bf16_out", [False, True])
def test_fp8_linear_equals_the_1sm_kernel(M, N, K, S, fa, fb, bf16_out):
    """8-bit float operands on pairs (kind::f8f6f4, K = 32 per instruction)
    with the output scale and a bias: the 1-SM kernel's bits."""
    tda = torch.float8_e4m3fn if fa == dig.FP8_E4M3 else torch.float8_e5m2
    tdb = torch.float8_e4m3fn if fb == dig.FP8_E4M3 else torch.float8_e5m2
    g = workloads.generator(M + N + K)
    A = torch.randn(M, K, generator=g).to(tda).cuda()
    W = (torch.randn(N, K, generator=g) * 0.05).to(tdb).cuda()
    b = workloads.normal_bf16((N,), 4).cuda()
    dt = torch.bfloat16 if bf16_out else torch.float32
    dig.bigemm_set_pair_mode(dig.PAIR_ALWAYS)
    assert dig.bigemm_uses_pair(M, N, K, S, fp8=True) == 1
    pair = dig.linear_fp8(A, W, 0.5, b, out_dtype=dt, split_k=S)
    dig.bigemm_set_pair_mode(dig.PAIR_NEVER)
    single = dig.linear_fp8(A, W, 0.5, b, out_dtype=dt, split_k=S)
    torch.cuda.synchronize()
    assert bits_equal(pair, single)
    for r in (0, 255, M - 1):
        one = dig.linear_fp8(A[r:r + 1].contiguous(), W, 0.5, b, out_dtype=dt, split_k=S)
        assert bits_equal(one, pair[r:r + 1]), r


@pytest.mark.parametrize("bf16_out", [False, True])
def test_folded_linear_with_bias_equals_the_1sm_fold(bf16_out):
    """A folded split of the weight layout with a bias on pairs (the bias added
    once after the 0..S-1 sum): the 1-SM fold's bits and the rows alone."""
    M, N, K, S = 512, 33024, 2048, 4
    A = workloads.normal_bf16((M, K), 201).cuda()
    W = workloads.normal_bf16((N, K), 202, 0.02).cuda()
    b = workloads.normal_bf16((N,), 203).cuda()
    dt = torch.bfloat16 if bf16_out else torch.float32
    assert dig.bigemm_split_is_folded(M, N, K, S)
    dig.bigemm_set_pair_mode(dig.PAIR_ALWAYS)
    assert dig.bigemm_uses_pair(M, N, K, S) == 1
    pair = dig.linear(A, W, b, out_dtype=dt, split_k=S)
    dig.bigemm_set_pair_mode(dig.PAIR_NEVER)
    single = dig.linear(A, W, b, out_dtype=dt, split_k=S)
    torch.cuda.synchronize()
    assert bits_equal(pair, single)
    for r in (0, 255, 256, M - 1):
        one = dig.linear(A[r:r + 1].contiguous(), W, b, out_dtype=dt, split_k=S)
        assert bits_equal(one, pair[r:r + 1]), r


@pytest.mark.parametrize("M,N,K", [(256, 512, 1024), (520, 6144, 4096), (768, 1280, 1984)])
@pytest.mark.parametrize("bf16_out", [False, True])
def test_linear_with_bias_equals_the_1sm_kernel(M, N, K, bf16_out):
    """The weight layout W [N, K] (boxes of 128 weight rows per CTA) with a
    bias, including the pages' fused QKV width N = 6144."""
    A = workloads.normal_bf16((M, K), M + 1).cuda()
    W = workloads.normal_bf16((N, K), N + 2, 0.02).cuda()
    b = workloads.normal_bf16((N,), 3).cuda()
    pair = product(A, W, dig.PAIR_ALWAYS, bf16_out, wt=True, bias=b)
    single = product(A, W, dig.PAIR_NEVER, bf16_out, wt=True, bias=b)
    assert bits_equal(pair, single)
    rows = [0, 127, 128, 255, M - 1]
    Cref, D = oracle.linear_rows(A.cpu(), W.cpu(), b.cpu(), M, N, K, rows=rows)
    check_tolerance(to_f64(pair[torch.tensor(rows, device="cuda")]), Cref, D, bf16_out, "pair linear")


@pytest.mark.parametrize("bf16_out", [False, True])
def test_rows_equal_one_row_products(bf16_out):
    """Rows on both CTAs of a pair tile and on both sides of tile boundaries
    equal the same rows computed alone (the few-row kernel, one CTA)."""
    M, N, K = 1024, 768, 2048
    A = workloads.normal_bf16((M, K), 71).cuda()
    B = workloads.normal_bf16((K, N), 72, 0.05).cuda()
    full = product(A, B, dig.PAIR_ALWAYS, bf16_out)
    dt = torch.bfloat16 if bf16_out else torch.float32
    for r in (0, 1, 127, 128, 200, 255, 256, 383, 384, 511, 512, 1023):
        one = dig.matmul(A[r:r + 1].contiguous(), B, out_dtype=dt, split_k=1)
        assert bits_equal(one, full[r:r + 1]), r


def test_rule_edge_and_row_windows():
    """Under the default rule: products on both sides of the two-wave edge
    (one pair tile column fewer) and windows of rows at 255 / 256 rows give the
    bits of the largest product."""
    cap = dig.bigemm_pair_capacity()
    rows = 256 * cdiv(2 * cap, 8)                  # 8 tile columns of 256 reach two waves
    N, K = 8 * 256, 512
    A = workloads.normal_bf16((rows, K), 81).cuda()
    B = workloads.normal_bf16((K, N), 82, 0.05).cuda()
    dig.bigemm_set_pair_mode(dig.PAIR_AUTO)
    assert dig.bigemm_uses_pair(rows, N, K, 1) == 1
    assert dig.bigemm_uses_pair(rows, N - 256, K, 1) == 0 or 7 * cdiv(rows, 256) >= 2 * cap
    full = dig.matmul(A, B, split_k=1)
    narrow = dig.matmul(A, B[:, :N - 256].contiguous(), split_k=1)
    assert bits_equal(narrow, full[:, :N - 256])
    for lo, hi in ((0, 255), (0, 256), (1, 257), (rows - 300, rows)):
        part = dig.matmul(A[lo:hi].contiguous(), B, split_k=1)
        assert bits_equal(part, full[lo:hi]), (lo, hi)


def test_writes_only_c_and_meets_the_oracle():
    """Padded leading dimensions: nothing outside C is written; sampled rows
    within the oracle's tolerance."""
    M, N, K = 300, 520, 776
    A, B = workloads.pair(M, N, K, 91, a_std=1.0, b_std=0.05)
    dig.bigemm_set_pair_mode(dig.PAIR_ALWAYS)
    for bf16_out in (False, True):
        C, buf = run_gemm(A, B, M, N, K, 1, bf16_out, lda=K + 8, ldb=N + 16, ldc=N + 8 * 4)
        assert canary_intact(buf, M, N)
        rows = [0, 128, 255, 256, 299]
        Cref, D = oracle.gemm_rows(A, B, M, N, K, rows=rows)
        check_tolerance(to_f64(C[torch.tensor(rows, device="cuda")]), Cref, D, bf16_out, "pair")


def test_integer_inputs_equal_the_oracle_bitwise():
    M, N, K = 512, 512, 1024
    g = workloads.generator(93)
    A = torch.randint(-8, 9, (M, K), generator=g).to(torch.bfloat16)
    B = torch.randint(-8, 9, (K, N), generator=g).to(torch.bfloat16)
    dig.bigemm_set_pair_mode(dig.PAIR_ALWAYS)
    C, _ = run_gemm(A, B, M, N, K, 1)
    Cref, _ = oracle.gemm_rows(A, B, M, N, K)
    assert (to_f64(C) == Cref).all()


def test_two_streams_and_a_graph_replay():
    """Two 2-SM products enqueued on two streams at once, and a CUDA graph of
    a chain of them (programmatic launches), give the serial results' bits."""
    dig.bigemm_set_pair_mode(dig.PAIR_ALWAYS)
    shapes = [(1024, 2048, 1024, 95), (768, 1536, 2048, 96)]
    data = [(workloads.normal_bf16((M, K), s).cuda(), workloads.normal_bf16((K, N), s + 1, 0.05).cuda())
            for M, N, K, s in shapes]
    serial = [dig.matmul(a, b, split_k=1) for a, b in data]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in data]
    for _ in range(3):
        outs = []
        torch.cuda.current_stream().synchronize()
        for (a, b), st in zip(data, streams):
            with torch.cuda.stream(st):
                outs.append(dig.matmul(a, b, split_k=1, stream=st))
        torch.cuda.synchronize()
        for got, want in zip(outs, serial):
            assert bits_equal(got, want)
    a, b = data[0]
    M, K = a.shape
    N = b.shape[1]
    outs = [torch.empty((M, N), device="cuda") for _ in range(3)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for c in outs:
            dig.bigemm_run(a, b, c, M, N, K, K, N, N, 1, None, 0, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(2):
        for c in outs:
            c.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for c in outs:
            assert bits_equal(c, serial[0])
    assert dig.bigemm_device_status(reset=True) == 0


def test_bit_stable_over_10_runs():
    A = workloads.normal_bf16((4096, 4096), 97).cuda()
    B = workloads.normal_bf16((4096, 4096), 98, 0.02).cuda()
    dig.bigemm_set_pair_mode(dig.PAIR_AUTO)
    assert dig.bigemm_uses_pair(4096, 4096, 4096, 1) == 1
    first = dig.matmul(A, B, split_k=1)
    for _ in range(9):
        assert bits_equal(dig.matmul(A, B, split_k=1), first)
