"""GPU: clustered split-K.  A split product (S = 2..8) whose tiles' clusters
of S CTAs all fit on the GPU at once runs as one kernel: CTA s of a cluster
computes K segment s of the tile into its shared memory, and the cluster adds
the partials through distributed shared memory in the order 0..S-1 with the
reduction kernel's FP32 additions.  The bits must equal the workspace path's
(partial kernel + splitk_reduce_kernel, run here explicitly), at every M, and
meet the oracle's tolerance.  (Tencent AI-infra article "腾讯エンジニア：
大規模モデルの出力を確定させるための AI インフラ手法": "Split-K" -- a fixed
segment order and no atomics; "Batch Invariance の由来" -- the split depends on
K only.)"""
import pytest
import torch

import deterministic_invariant_gemm_gb300 as dig
import oracle
import workloads
from gemm_check import (bits_equal, canary_intact, check_tolerance, device_matrix, output_buffer,
                        round_up, run_gemm, to_f64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device(cuda_device):
    dig.load()
    yield
    assert dig.bigemm_device_status(reset=True) == 0


def two_kernel_path(A, B, M, N, K, S, bf16_out):
    """The product through the workspace: partial kernel, then reduction."""
    lda, ldb = round_up(K, 8), round_up(N, 8)
    Ad, Bd = device_matrix(A, lda), device_matrix(B, ldb)
    s_eff = dig.bigemm_effective_split_k(K, S)
    need = dig.bigemm_partial_workspace_bytes(M, N, K, S)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    dig.bigemm_run_partial(Ad, Bd, M, N, K, lda, ldb, S, ws, need)
    ldc = round_up(N, 8)
    C = torch.empty((M, ldc), dtype=torch.bfloat16 if bf16_out else torch.float32, device="cuda")
    dig.bigemm_splitk_reduce(ws, s_eff, M, N, C, ldc, bf16_out)
    return C[:, :N]


def tiles(M, N):
    return -(-M // 128) * -(-N // 256)


def test_path_rule(capsys):
    """A split product (S = 2..8) that is not folded and runs wide tiles
    clusters exactly when its tiles are no more than the device's cluster
    capacity for S; the capacity is the device's (printed)."""
    caps = {S: dig.bigemm_cluster_capacity(S) for S in range(2, 9)}
    with capsys.disabled():
        print("\n[cluster path] capacity for S = 2..8: %s" % [caps[S] for S in range(2, 9)])
    assert all(c >= 1 for c in caps.values())
    for M in (1, 16, 32, 33, 64, 128, 200, 640):
        for N in (256, 1024, 2048, 3840, 4096, 6144):
            for K, S in ((4096, 8), (4096, 4), (3000, 3), (640, 2), (8192, 16), (4096, 1)):
                s = dig.bigemm_effective_split_k(K, S)
                if s == 1:
                    want = dig.PATH_UNSPLIT
                elif M <= dig.SKINNY_MAX_ROWS and s <= dig.SKINNY_MAX_SPLIT:
                    want = dig.PATH_SKINNY
                elif dig.bigemm_split_is_folded(M, N, K, S):
                    want = dig.PATH_FOLDED
                elif dig.bigemm_tile_n(M, N, K, S) != 256:
                    want = dig.PATH_WORKSPACE
                elif s <= 8 and tiles(M, N) <= caps[s]:
                    want = dig.PATH_CLUSTER
                else:
                    want = dig.PATH_WORKSPACE
                assert dig.bigemm_split_path(M, N, K, S) == want, (M, N, K, S)


@pytest.mark.parametrize("M,N,K,S", [
    (40, 2048, 4096, 8),         # rows against a 2048-wide weight: 8 clusters of 8
    (33, 2048, 4096, 8),
    (64, 3840, 4096, 8),         # 15 tiles
    (128, 2048, 4096, 8),
    (48, 4096, 4096, 4),         # 16 clusters of 4
    (64, 4096, 4096, 6),         # 11 blocks per segment, the last 9
    (200, 1024, 4096, 8),        # two tile rows, the second ragged
    (37, 1000, 3000, 3),         # ragged N (4 tiles, the last 232 wide), S = 3 segments of 16, 16, 15
    (35, 300, 1000, 5),          # N not a multiple of 4: the last columns stored one by one
    (64, 2048, 640, 2),          # two segments of 5 blocks
    (33, 512, 8192, 7),          # 128 blocks in 7 segments of 19 (the last 14)
])
@pytest.mark.parametrize("bf16_out", [False, True])
def test_cluster_equals_the_two_kernel_path(M, N, K, S, bf16_out):
    path = dig.bigemm_split_path(M, N, K, S)
    if path != dig.PATH_CLUSTER:
        pytest.skip("this device fits too few clusters of %d for %d tiles" % (S, -(-M // 128) * -(-N // 256)))
    A, B = workloads.pair(M, N, K, 3 * M + N + K + S)
    C, buf = run_gemm(A, B, M, N, K, S, bf16_out)
    assert dig.bigemm_last_launch_count() == 1
    assert canary_intact(buf, M, N)
    ref = two_kernel_path(A, B, M, N, K, S, bf16_out)
    torch.cuda.synchronize()
    assert bits_equal(C, ref)
    rows = sorted({0, M // 2, M - 1})
    Cref, D = oracle.gemm_rows(A, B, M, N, K, rows=rows)
    check_tolerance(to_f64(C[torch.tensor(rows, device="cuda")]), Cref, D, bf16_out,
                    "cluster M=%d N=%d K=%d S=%d" % (M, N, K, S))


def test_cluster_rows_equal_workspace_rows_of_a_larger_batch():
    """Rows computed at M = 1, 4, 16 (few-row kernel) and 33, 48 (cluster path)
    equal the same rows inside a 640-row batch, which has too many tiles to
    cluster and is not folded (workspace path)."""
    N, K, S = 2048, 4096, 8
    M = 640
    assert dig.bigemm_split_path(M, N, K, S) == dig.PATH_WORKSPACE
    A, B = workloads.pair(M, N, K, 7, a_std=1.0, b_std=0.02)
    A, B = A.cuda(), B.cuda()
    full = dig.matmul(A, B, split_k=S)
    assert dig.bigemm_last_launch_count() == 2
    for m in (1, 4, 16, 33, 48):
        for off in (0, 300, M - m):
            part = dig.matmul(A[off:off + m].contiguous(), B, split_k=S)
            assert dig.bigemm_last_launch_count() == 1
            assert bits_equal(part, full[off:off + m]), (m, off)


def test_cluster_bit_stable_over_10_runs():
    A, B = workloads.pair(40, 2048, 4096, 8)
    A, B = A.cuda(), B.cuda()
    assert dig.bigemm_split_path(40, 2048, 4096, 8) == dig.PATH_CLUSTER
    first = dig.matmul(A, B, split_k=8)
    for _ in range(9):
        assert bits_equal(dig.matmul(A, B, split_k=8), first)


@pytest.mark.parametrize("bf16_out", [False, True])
def test_clustered_linear_with_bias(bf16_out):
    """The fused QKV shape of the pages (N = 6144, K = 4096): rows at M = 1 and
    16 against the same rows in a 640-row batch (workspace path), and the
    oracle on samples.  Its 24 tile columns need 24 clusters of 8 CTAs, more
    than the GPU has SMs, so a small batch clusters only where the device
    fits them; the bits agree whichever path runs.  The bias is added after
    the cluster's sum, as after the reduction kernel's."""
    M, N, K, S = 640, 6144, 4096, 8
    A = workloads.normal_bf16((M, K), 41)
    W = workloads.normal_bf16((N, K), 42, 0.02)
    b = workloads.normal_bf16((N,), 43)
    Ad, Wd, bd = A.cuda(), W.cuda(), b.cuda()
    dt = torch.bfloat16 if bf16_out else torch.float32
    assert dig.bigemm_split_path(M, N, K, S) == dig.PATH_WORKSPACE
    full = dig.linear(Ad, Wd, bd, out_dtype=dt, split_k=S)
    for lo, hi in ((0, 1), (100, 116), (639, 640)):
        part = dig.linear(Ad[lo:hi].contiguous(), Wd, bd, out_dtype=dt, split_k=S)
        assert bits_equal(part, full[lo:hi]), (lo, hi)
    rows = [0, 115, 639]
    Cref, D = oracle.linear_rows(A, W, b, M, N, K, rows=rows)
    check_tolerance(to_f64(full[torch.tensor(rows, device="cuda")]), Cref, D, bf16_out,
                    "clustered linear")


def test_clustered_fp8_linear_with_scale_and_bias():
    M, N, K, S = 640, 2048, 8192, 8
    g = workloads.generator(51)
    A = torch.randn(M, K, generator=g).to(torch.float8_e4m3fn)
    W = (torch.randn(N, K, generator=g) * 0.05).to(torch.float8_e4m3fn)
    b = workloads.normal_bf16((N,), 52)
    Ad, Wd, bd = A.cuda(), W.cuda(), b.cuda()
    assert dig.bigemm_split_path(M, N, K, S, fp8=True) == dig.PATH_WORKSPACE
    full = dig.linear_fp8(Ad, Wd, 1.25, bd, split_k=S)
    for lo, hi in ((0, 1), (200, 264), (630, 640)):
        assert dig.bigemm_split_path(hi - lo, N, K, S, fp8=True) == dig.PATH_CLUSTER
        part = dig.linear_fp8(Ad[lo:hi].contiguous(), Wd, 1.25, bd, split_k=S)
        assert bits_equal(part, full[lo:hi]), (lo, hi)
    rows = [0, 263, 639]
    Cref, D = oracle.linear8_rows(A, W, oracle.FMT_E4M3, oracle.FMT_E4M3, M, N, K, 1.25, b, rows=rows)
    check_tolerance(to_f64(full[torch.tensor(rows, device="cuda")]), Cref, D, False, "clustered fp8")


def test_cluster_path_leaves_the_workspace_alone():
    """The workspace is required by the shape rule but the cluster path does
    not touch it."""
    M, N, K, S = 40, 2048, 4096, 8
    assert dig.bigemm_split_path(M, N, K, S) == dig.PATH_CLUSTER
    A, B = workloads.pair(M, N, K, 9)
    A, B = A.cuda(), B.cuda()
    need = dig.bigemm_workspace_bytes(M, N, K, S)
    ws = torch.full((need,), 0x5A, dtype=torch.uint8, device="cuda")
    C = output_buffer(M, N, N, False)
    dig.bigemm_run(A, B, C, M, N, K, K, N, N, S, ws, need)
    torch.cuda.synchronize()
    assert bool((ws == 0x5A).all())
    assert canary_intact(C, M, N)
