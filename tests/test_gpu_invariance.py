"""GPU invariance: the bits of a row of C depend only on that row of A, on B,
on K and on split_k -- not on M, on the other rows of the batch, on where the
row sits, or on the run (Tencent AI-infra article "腾讯エンジニア：大規模モデルの
出力を確定させるための AI インフラ手法": "背景" defines run-to-run determinism and
batch invariance; "Batch Invariance の由来" and "Split-K" say which tiling
choices may and may not change the reduction order).

All comparisons are bitwise (int32 / int16 views).  The atomic-add split-K
contrast is measured here too; its run-to-run spread is reported, not
asserted, since the order of atomic additions is up to the hardware.
"""
import numpy as np
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


def assert_correct(C, A, B, bf16_out=False, rows=None):
    """Bitwise agreement alone would also accept a consistently wrong result:
    the reference output of each invariance check is held to the oracle too
    (on a row sample for large products)."""
    M, K = A.shape
    N = B.shape[1]
    Cref, D = oracle.gemm_rows(A.cpu(), B.cpu(), M, N, K, rows=rows)
    got = C if rows is None else C[torch.tensor(rows, device=C.device)]
    check_tolerance(to_f64(got), Cref, D, bf16_out, "invariance reference")


def gemm(A, B, split_k=1, bf16_out=False, atomic=False, ws=None):
    return dig.matmul(A, B, out_dtype=torch.bfloat16 if bf16_out else torch.float32,
                      split_k=split_k, atomic=atomic, workspace=ws)


@pytest.mark.parametrize("split_k", [1, 4])
@pytest.mark.parametrize("bf16_out", [False, True])
def test_small_rows_invariant_at_m_1_7_64(split_k, bf16_out):
    """Every row of the 64 x 256 x 512 product, recomputed alone (M = 1), inside
    every 7-row window that contains it, and inside the full 64-row batch,
    is byte-identical."""
    w = workloads.WORKLOADS["small"]
    M, N, K = w["M"], w["N"], w["K"]
    A, B = workloads.pair(M, N, K, workloads.BASE_SEED + w["index"])
    A, B = A.cuda(), B.cuda()
    full = gemm(A, B, split_k, bf16_out)
    assert_correct(full, A, B, bf16_out)
    for i in range(M):
        one = gemm(A[i:i + 1].contiguous(), B, split_k, bf16_out)
        assert bits_equal(one, full[i:i + 1]), "row %d differs at M=1" % i
    for s in range(0, M - 6):
        win = gemm(A[s:s + 7].contiguous(), B, split_k, bf16_out)
        assert bits_equal(win, full[s:s + 7]), "window %d..%d differs at M=7" % (s, s + 6)
    torch.cuda.synchronize()


def test_decode_rows_invariant_across_batch_sizes():
    """Decode shapes (N = K = 4096, split_k from K only): rows computed at
    M = 1, 4, 16, 64, and at offsets inside the batch, agree bit for bit."""
    w = workloads.WORKLOADS["decode"]
    N, K = w["N"], w["K"]
    A, B = workloads.pair(64, N, K, workloads.BASE_SEED + w["index"], a_std=w["a_std"],
                          b_std=w["b_std"])
    A, B = A.cuda(), B.cuda()
    ref = gemm(A, B, split_k=0)
    assert_correct(ref, A, B)
    for M in w["Ms"]:
        for off in (0, 64 - M, (64 - M) // 2):
            out = gemm(A[off:off + M].contiguous(), B, split_k=0)
            assert bits_equal(out, ref[off:off + M]), "M=%d offset %d" % (M, off)
    # a big batch (many M tiles) containing the decode rows at a tile boundary
    big = torch.cat([workloads.normal_bf16((127, K), 5).cuda(), A,
                     workloads.normal_bf16((300, K), 6).cuda()])
    out = gemm(big, B, split_k=0)
    assert bits_equal(out[127:191], ref)


def test_row_position_inside_tiles():
    """One row placed at every position of a 128-row tile (and across tile
    boundaries of a 3-tile batch) gives the same bits."""
    N, K = 512, 1536
    row, B = workloads.pair(1, N, K, 44)
    filler = workloads.normal_bf16((383, K), 45)
    row, B, filler = row.cuda(), B.cuda(), filler.cuda()
    ref = gemm(row, B)
    assert_correct(ref, row, B)
    for pos in (0, 1, 31, 32, 63, 64, 95, 96, 127, 128, 255, 256, 383):
        batch = torch.cat([filler[:pos], row, filler[pos:]])
        out = gemm(batch, B)
        assert bits_equal(out[pos:pos + 1], ref), "position %d" % pos


@pytest.mark.parametrize("size,bf16_out", [(2048, False), (16384, True)])
def test_mixed_batch_permuted_and_padded(size, bf16_out):
    """Rows permuted by a seeded permutation and padded with r random extra
    rows (so the batch is no multiple of 128): C'[pi^-1(i)] == C[i] bytewise."""
    M = N = K = size
    A, B = workloads.pair(M, N, K, workloads.BASE_SEED + 3)
    A, B = A.cuda(), B.cuda()
    C = gemm(A, B, 1, bf16_out)
    assert_correct(C, A, B, bf16_out, rows=[0, 1, size // 2, size - 1])
    g = torch.Generator().manual_seed(size)
    perm = torch.randperm(M, generator=g).cuda()
    r = int(torch.randint(1, 128, (1,), generator=g))
    extra = workloads.normal_bf16((r, K), 99).cuda()
    Ap = torch.cat([A[perm], extra])                     # row t of Ap is row perm[t] of A
    Cp = gemm(Ap, B, 1, bf16_out)
    torch.cuda.synchronize()
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(M, device="cuda")
    assert bits_equal(Cp[:M][inv], C)


@pytest.mark.parametrize("S", [8, 16, 32])
def test_longk_workspace_path_bit_stable_over_10_runs(S):
    w = workloads.WORKLOADS["longk"]
    M, N, K = w["M"], w["N"], w["K"]
    A, B = workloads.pair(M, N, K, workloads.BASE_SEED + w["index"])
    A, B = A.cuda(), B.cuda()
    first = gemm(A, B, S)
    assert_correct(first, A, B)
    for _ in range(9):
        assert bits_equal(gemm(A, B, S), first)


def test_square_bit_stable_over_10_runs():
    A, B = workloads.pair(4096, 4096, 4096, 77, dist="uniform")
    A, B = A.cuda(), B.cuda()
    first = gemm(A, B, 1)
    for _ in range(9):
        assert bits_equal(gemm(A, B, 1), first)


def test_split_changes_bits_only_through_split_k():
    """Different split_k values are allowed to differ (a different but fixed
    reduction tree); the same split_k never does."""
    A, B = workloads.pair(32, 512, 8192, 17)
    A, B = A.cuda(), B.cuda()
    outs = {S: gemm(A, B, S) for S in (1, 2, 4, 8, 16)}
    for S, o in outs.items():
        assert_correct(o, A, B)
        assert bits_equal(gemm(A, B, S), o)
    assert any(not bits_equal(outs[1], outs[S]) for S in (2, 4, 8, 16))


def test_atomic_contrast_spread(capsys):
    """The atomic-add split-K variant over 10 runs: counted and printed.  The
    workspace path on the same inputs is asserted stable alongside it."""
    w = workloads.WORKLOADS["longk"]
    M, N, K = w["M"], w["N"], w["K"]
    A, B = workloads.pair(M, N, K, workloads.BASE_SEED + w["index"])
    A, B = A.cuda(), B.cuda()
    report = []
    for S in w["splits"]:
        runs = [gemm(A, B, S, atomic=True).view(torch.int32).cpu().numpy() for _ in range(10)]
        distinct = len({r.tobytes() for r in runs})
        differing = int((np.stack(runs) != runs[0]).any(axis=0).sum())
        report.append("S=%d: %d distinct results in 10 runs, %d of %d elements vary"
                      % (S, distinct, differing, M * N))
        det = [gemm(A, B, S) for _ in range(3)]
        assert bits_equal(det[0], det[1]) and bits_equal(det[0], det[2])
    with capsys.disabled():
        print("\n[atomic split-K contrast] " + "; ".join(report))


# ------------------------------- short and long batches in the partial kernel --

@pytest.mark.parametrize("N,K,S", [(256, 512, 2), (296, 1000, 3), (520, 3000, 6), (4096, 4096, 8)])
def test_partials_same_bits_for_short_and_long_batches(N, K, S):
    """The split-K partial kernel loads only the batch's rows of A for short
    batches (a 32- or 64-row A box, the rest of each stage zero) and 128-row
    boxes otherwise.  Every workspace slice row of a short batch must equal
    the same row inside a 200-row batch bit for bit (and the long batch's
    slices are held to the oracle through the full product)."""
    Mbig = 200
    A, B = workloads.pair(Mbig, N, K, 700 + N + S)
    Ad, Bd = A.cuda(), B.cuda()
    ld = dig.bigemm_workspace_ld(N)
    Se = dig.bigemm_effective_split_k(K, S)

    def slices(a):
        M = a.shape[0]
        nb = dig.bigemm_partial_workspace_bytes(M, N, K, S)
        ws = torch.full((nb // 4,), float("nan"), device="cuda")
        dig.bigemm_run_partial(a, Bd, M, N, K, K, N, S, ws, nb)
        return ws, ws[: Se * M * ld].view(Se, M, ld)[:, :, :N]

    ws_full, full = slices(Ad)
    C = torch.empty(Mbig, N, device="cuda")
    dig.bigemm_splitk_reduce(ws_full, Se, Mbig, N, C, N, 0)
    assert_correct(C, Ad, Bd, rows=[0, 63, 64, 199])
    for M in (1, 15, 16, 17, 33, 48, 64):
        for off in (0, 64, Mbig - M):
            _, part = slices(Ad[off:off + M].contiguous())
            assert bits_equal(part.contiguous(), full[:, off:off + M].contiguous()), (M, off)
    torch.cuda.synchronize()


def test_linear_short_batches_match_long_batches_both_dtypes():
    """Linear layers N = K = 4096, split_k = 8 (16 tiles: the workspace path,
    or for bf16 at M <= 32 the few-row kernel): bf16 and E4M3 rows computed at
    M <= 64 (short A boxes) equal the same rows inside a 200-row batch (full A
    boxes)."""
    N = K = 4096
    Mbig = 200
    x = workloads.normal_bf16((Mbig, K), 81).cuda()
    w = workloads.normal_bf16((N, K), 82, 0.02).cuda()
    b = workloads.normal_bf16((N,), 83).cuda()
    full = dig.linear(x, w, b, split_k=8)
    x8, w8 = x.to(torch.float8_e4m3fn), (w * 16).to(torch.float8_e4m3fn)
    full8 = dig.linear_fp8(x8, w8, 0.25, b, split_k=8)
    for fp8 in (False, True):
        assert dig.bigemm_split_path(Mbig, N, K, 8, fp8) == dig.PATH_WORKSPACE
    for M, off in ((1, 0), (16, 100), (32, 9), (33, 50), (40, 7), (64, 136)):
        assert dig.bigemm_split_path(M, N, K, 8, True) == dig.PATH_WORKSPACE
        assert dig.bigemm_split_path(M, N, K, 8, False) == (
            dig.PATH_SKINNY if M <= dig.SKINNY_MAX_ROWS else dig.PATH_WORKSPACE)
        part = dig.linear(x[off:off + M].contiguous(), w, b, split_k=8)
        assert bits_equal(part, full[off:off + M]), ("bf16", M, off)
        part8 = dig.linear_fp8(x8[off:off + M].contiguous(), w8, 0.25, b, split_k=8)
        assert bits_equal(part8, full8[off:off + M]), ("e4m3", M, off)
    torch.cuda.synchronize()
