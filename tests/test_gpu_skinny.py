"""GPU: the few-row kernel.  A bf16 product of at most 32 rows with at most
8 K segments runs as one launch: the S CTAs of each 128 x 256 output tile
form a thread-block cluster, CTA s computes K segment s with the wide
kernel's instructions (M = 128, N = 256, K = 16, the same operand roles),
and the cluster adds the partials through distributed shared memory in the
order 0..S-1 with the reduction kernel's FP32 additions.  Its bits must
equal the workspace path's (partial kernel + splitk_reduce_kernel, run here
explicitly) and the rows of larger batches, which run the other paths; and
it must meet the oracle's tolerance.  (Tencent AI-infra article "腾讯エンジ
ニア：大規模モデルの出力を確定させるための AI インフラ手法": "Split-K" -- a fixed
segment order, no atomics; "Batch Invariance の由来" -- the split depends on
K only, and the tile sizes M and N do not enter the reduction order.)"""
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


def test_path_rule():
    """Few rows and at most 8 segments: the few-row kernel, with no workspace
    and one launch; one more row, or one more segment, or 8-bit operands: the
    other paths."""
    for M in (1, 2, 16, 17, 31, 32):
        for K, S in ((4096, 8), (4096, 2), (3000, 3), (4096, 0), (640, 1)):
            s = dig.bigemm_effective_split_k(K, S)
            want = dig.PATH_SKINNY if s > 1 else dig.PATH_UNSPLIT
            assert dig.bigemm_split_path(M, 4096, K, S) == want, (M, K, S)
            assert dig.bigemm_workspace_bytes(M, 4096, K, S) == 0
            assert dig.bigemm_tile_n(M, 4096, K, S) == 256
            assert dig.bigemm_split_path(M, 4096, K, S, fp8=True) != dig.PATH_SKINNY
    assert dig.bigemm_split_path(33, 4096, 4096, 8) != dig.PATH_SKINNY
    assert dig.bigemm_split_path(16, 4096, 8192, 16) != dig.PATH_SKINNY
    assert dig.bigemm_split_path(16, 4096, 8192, 0) != dig.PATH_SKINNY    # default split 16
    assert dig.bigemm_workspace_bytes(33, 4096, 4096, 8) > 0
    assert dig.bigemm_workspace_bytes(16, 4096, 8192, 16) > 0


@pytest.mark.parametrize("M,N,K,S", [
    (1, 4096, 4096, 8),          # the decode workload's rows: 16 clusters of 8
    (4, 4096, 4096, 8),
    (16, 4096, 4096, 8),
    (17, 4096, 4096, 8),         # 32-row A stages
    (32, 4096, 4096, 8),         # the most rows the kernel takes
    (1, 256, 512, 1),            # unsplit: clusters of one CTA
    (7, 520, 4104, 5),           # ragged N (the third tile 8 wide) and K (65 blocks in 5 segments of 13)
    (13, 1000, 1000, 3),         # 16 blocks in segments of 6, 6, 4
    (5, 301, 3000, 7),           # N not a multiple of 4: the last columns stored one by one
    (32, 260, 8192, 8),          # a 4-column second tile
    (3, 64, 640, 2),             # N below one tile
    (9, 2048, 65536, 8),         # long segments (128 blocks)
])
@pytest.mark.parametrize("bf16_out", [False, True])
def test_equals_the_two_kernel_path_and_the_oracle(M, N, K, S, bf16_out):
    assert dig.bigemm_split_path(M, N, K, S) in (dig.PATH_SKINNY, dig.PATH_UNSPLIT)
    A, B = workloads.pair(M, N, K, 11 * M + N + K + S, a_std=1.0, b_std=0.02)
    C, buf = run_gemm(A, B, M, N, K, S, bf16_out)
    assert dig.bigemm_last_launch_count() == 1
    assert canary_intact(buf, M, N)
    ref = two_kernel_path(A, B, M, N, K, S, bf16_out)
    torch.cuda.synchronize()
    assert bits_equal(C, ref)
    Cref, D = oracle.gemm_rows(A, B, M, N, K)
    check_tolerance(to_f64(C), Cref, D, bf16_out, "few-row M=%d N=%d K=%d S=%d" % (M, N, K, S))


@pytest.mark.parametrize("bf16_out", [False, True])
def test_rows_equal_the_rows_of_larger_batches(bf16_out):
    """Every batch size from 1 to 33 (the last one past the kernel) against the
    same rows of a 300-row batch (three tile rows: the cluster or the
    workspace path), at offsets that cross the larger batch's tile
    boundaries."""
    N, K, S = 1024, 4096, 8
    Mbig = 300
    A, B = workloads.pair(Mbig, N, K, 23, a_std=1.0, b_std=0.02)
    Ad, Bd = A.cuda(), B.cuda()
    dt = torch.bfloat16 if bf16_out else torch.float32
    full = dig.matmul(Ad, Bd, out_dtype=dt, split_k=S)
    assert dig.bigemm_split_path(Mbig, N, K, S) in (dig.PATH_CLUSTER, dig.PATH_WORKSPACE)
    for m in list(range(1, 34)):
        for off in (0, 127 - m // 2, Mbig - m):
            part = dig.matmul(Ad[off:off + m].contiguous(), Bd, out_dtype=dt, split_k=S)
            assert bits_equal(part, full[off:off + m]), (m, off)


@pytest.mark.parametrize("bf16_out", [False, True])
def test_linear_with_bias_equals_larger_batches(bf16_out):
    """The weight layout W [N, K] (the pages' fused QKV width, N = 6144) with a
    bias added after the cluster's sum: rows at M = 1, 8, 32 against a
    200-row batch, and the oracle."""
    M, N, K, S = 200, 6144, 4096, 8
    A = workloads.normal_bf16((M, K), 31)
    W = workloads.normal_bf16((N, K), 32, 0.02)
    b = workloads.normal_bf16((N,), 33)
    Ad, Wd, bd = A.cuda(), W.cuda(), b.cuda()
    dt = torch.bfloat16 if bf16_out else torch.float32
    full = dig.linear(Ad, Wd, bd, out_dtype=dt, split_k=S)
    for lo, hi in ((0, 1), (100, 108), (168, 200)):
        assert dig.bigemm_split_path(hi - lo, N, K, S) == dig.PATH_SKINNY
        part = dig.linear(Ad[lo:hi].contiguous(), Wd, bd, out_dtype=dt, split_k=S)
        assert dig.bigemm_last_launch_count() == 1
        assert bits_equal(part, full[lo:hi]), (lo, hi)
    rows = [0, 107, 199]
    Cref, D = oracle.linear_rows(A, W, b, M, N, K, rows=rows)
    check_tolerance(to_f64(full[torch.tensor(rows, device="cuda")]), Cref, D, bf16_out, "few-row linear")


def test_bit_stable_over_10_runs():
    A, B = workloads.pair(16, 4096, 4096, 41, a_std=1.0, b_std=0.02)
    A, B = A.cuda(), B.cuda()
    first = dig.matmul(A, B, split_k=8)
    for _ in range(9):
        assert bits_equal(dig.matmul(A, B, split_k=8), first)


def test_integer_inputs_equal_the_oracle_bitwise():
    """Small integers, every partial sum an integer below 2^24: FP32 is exact
    in any order, so the result equals the binary64 oracle exactly."""
    M, N, K, S = 5, 520, 4096, 8
    g = workloads.generator(43)
    A = torch.randint(-8, 9, (M, K), generator=g).to(torch.bfloat16)
    B = torch.randint(-8, 9, (K, N), generator=g).to(torch.bfloat16)
    C, _ = run_gemm(A, B, M, N, K, S)
    Cref, _ = oracle.gemm_rows(A, B, M, N, K)
    assert (to_f64(C) == Cref).all()


def test_graph_replay_of_a_chain_equals_eager_calls():
    """A chain of products captured in a CUDA graph (the next product's CTAs
    start early and warm L2 with their weights under programmatic launch)
    gives the bits of the same products called one by one."""
    N = K = 4096
    Bs = [workloads.normal_bf16((K, N), 50 + j, 0.02).cuda() for j in range(4)]
    As = [workloads.normal_bf16((m, K), 60 + m).cuda() for m in (1, 4, 16, 32)]
    eager = [dig.matmul(a, b, split_k=8) for a, b in zip(As, Bs)]
    outs = [torch.empty_like(e) for e in eager]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for a, b, c in zip(As, Bs, outs):
            dig.bigemm_run(a, b, c, a.shape[0], N, K, K, N, N, 8, None, 0)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        for c in outs:
            c.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for c, e in zip(outs, eager):
            assert bits_equal(c, e)


def test_runs_without_a_workspace_and_writes_only_c():
    M, N, K, S = 16, 2048, 4096, 8
    A, B = workloads.pair(M, N, K, 47)
    A, B = A.cuda(), B.cuda()
    assert dig.bigemm_workspace_bytes(M, N, K, S) == 0
    C = output_buffer(M, N, N, False)
    dig.bigemm_run(A, B, C, M, N, K, K, N, N, S, None, 0)
    assert dig.bigemm_last_launch_count() == 1
    torch.cuda.synchronize()
    assert canary_intact(C, M, N)
    assert bits_equal(C[:M, :N], dig.matmul(A, B, split_k=S))
