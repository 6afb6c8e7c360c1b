"""GPU: narrow output tiles.  A bf16 product whose 256-column work units
(tiles x K segments) would occupy fewer than half of the SMs while each unit
streams at least 32 K blocks runs with 128- or 64-column tiles
(bigemm_tile_n), so that more SMs stream its operands -- the small-tile,
long-K case the Tencent AI-infra article's "Split-K" section describes
("腾讯エンジニア：大規模モデルの出力を確定させるための AI インフラ手法").  The width
sets only the N extent of each 128-row tensor-core instruction; which K
blocks an element sums, and in what order, does not change ("Batch
Invariance の由来": the tile sizes M and N do not enter the reduction order).
So rows must be bit-identical whether their batch runs 64-, 128- or
256-wide, and every width must meet the oracle's tolerance."""
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


def cdiv(a, b):
    return -(-a // b)


def half_the_sms():
    return torch.cuda.get_device_properties(0).multi_processor_count // 2


def expected_width(M, N, K, S):
    """The documented rule, restated: 256 unless the 256-wide units (tiles x
    segments) fall below half the SMs and a segment has >= 32 K blocks; then
    the widest of 128, 64 whose units reach half the SMs, else 64."""
    s_req = S if S else dig.bigemm_default_split_k(K)
    s = dig.bigemm_effective_split_k(K, S)
    L = cdiv(cdiv(K, 64), s_req)
    if M == 0 or N == 0 or K == 0 or L < 32 or dig.bigemm_split_is_folded(M, N, K, S):
        return 256
    if M <= dig.SKINNY_MAX_ROWS and s <= dig.SKINNY_MAX_SPLIT:
        return 256      # the few-row kernel, always 256 wide
    
    mt, half = cdiv(M, 128), half_the_sms()
    for w in (256, 128):
        if mt * cdiv(N, w) * s >= half:
            return w
    return 64


def test_width_rule_and_paths():
    seen = set()
    for M in (1, 16, 33, 48, 128, 200, 640, 1280, 4096):
        for N in (64, 256, 300, 512, 1024, 2048, 4096):
            for K, S in ((65536, 8), (65536, 16), (65536, 32), (16384, 8), (4096, 1), (2048, 1),
                         (4096, 8), (1984, 1), (8192, 0)):
                w = dig.bigemm_tile_n(M, N, K, S)
                assert w == expected_width(M, N, K, S), (M, N, K, S, w)
                seen.add(w)
                if w != 256 and dig.bigemm_effective_split_k(K, S) > 1:
                    # narrow split products sum through the workspace
                    assert dig.bigemm_split_path(M, N, K, S) == dig.PATH_WORKSPACE
    assert seen == {64, 128, 256}
    # the few-row kernel takes the small batches of split counts up to 8
    assert dig.bigemm_tile_n(1, 256, 65536, 8) == 256
    assert dig.bigemm_split_path(1, 256, 65536, 8) == dig.PATH_SKINNY
    assert dig.bigemm_tile_n(33, 256, 65536, 8) == 64
    # the decode shape of the pages' linear layers stays wide
    for M in (1, 4, 16, 64):
        assert dig.bigemm_tile_n(M, 4096, 4096, 8) == 256
    # 8-bit products are always wide
    assert dig.bigemm_tile_n(1, 256, 65536, 8, fp8=True) == 256


def batch_sizes(N, K, S):
    """Batch sizes at which a product of (N, K, S) runs 64-, 128- and 256-wide
    on this device: one tile row, then just enough tile rows for the wider
    units to reach half the SMs."""
    s = dig.bigemm_effective_split_k(K, S)
    half = half_the_sms()
    m128 = 128 * cdiv(half, cdiv(N, 128) * s)
    m256 = 128 * cdiv(half, cdiv(N, 256) * s)
    # one tile row, but more rows than the few-row kernel takes
    return {64: dig.SKINNY_MAX_ROWS + 1, 128: m128, 256: m256}


@pytest.mark.parametrize("N,K,S", [
    (256, 16384, 8),     # segments of 32 blocks
    (256, 65536, 8),     # the long-K workload's split at 8
    (512, 4096, 1),      # unsplit, direct epilogue
    (320, 3000, 1),      # ragged N (the 64-wide tiles' last is full, the 128-wide half) and K
])
@pytest.mark.parametrize("bf16_out", [False, True])
def test_rows_equal_across_widths(N, K, S, bf16_out):
    sizes = batch_sizes(N, K, S)
    Mbig = sizes[256]
    for w, m in sizes.items():
        assert dig.bigemm_tile_n(m, N, K, S) == w, (w, m)
    A, B = workloads.pair(Mbig, N, K, 17 * N + K + S)
    Ad, Bd = A.cuda(), B.cuda()
    dt = torch.bfloat16 if bf16_out else torch.float32
    full = dig.matmul(Ad, Bd, out_dtype=dt, split_k=S)            # 256 wide
    mid = dig.matmul(Ad[:sizes[128]].contiguous(), Bd, out_dtype=dt, split_k=S)   # 128 wide
    assert bits_equal(mid, full[:sizes[128]])
    for lo, hi in ((0, 1), (77, 78), (Mbig - 1, Mbig), (130, 194), (Mbig - 100, Mbig), (40, 73)):
        part = dig.matmul(Ad[lo:hi].contiguous(), Bd, out_dtype=dt, split_k=S)
        if hi - lo > dig.SKINNY_MAX_ROWS:
            assert dig.bigemm_tile_n(hi - lo, N, K, S) == 64
        else:
            assert dig.bigemm_split_path(hi - lo, N, K, S) in (dig.PATH_SKINNY, dig.PATH_UNSPLIT)
        assert bits_equal(part, full[lo:hi]), (lo, hi)
    rows = [0, 77, Mbig - 1]
    Cref, D = oracle.gemm_rows(A, B, Mbig, N, K, rows=rows)
    check_tolerance(to_f64(full[torch.tensor(rows, device="cuda")]), Cref, D, bf16_out,
                    "widths N=%d K=%d S=%d" % (N, K, S))


@pytest.mark.parametrize("bf16_out", [False, True])
def test_linear_rows_equal_across_widths(bf16_out):
    """The weight layout W [N, K] (K-major boxes of tile-width rows) with a
    bias, added after the split sum."""
    N, K, S = 256, 8192, 4
    sizes = batch_sizes(N, K, S)
    Mbig = sizes[256]
    A = workloads.normal_bf16((Mbig, K), 61)
    W = workloads.normal_bf16((N, K), 62, 0.02)
    b = workloads.normal_bf16((N,), 63)
    Ad, Wd, bd = A.cuda(), W.cuda(), b.cuda()
    dt = torch.bfloat16 if bf16_out else torch.float32
    full = dig.linear(Ad, Wd, bd, out_dtype=dt, split_k=S)
    mid = dig.linear(Ad[:sizes[128]].contiguous(), Wd, bd, out_dtype=dt, split_k=S)
    assert bits_equal(mid, full[:sizes[128]])
    for lo, hi in ((0, 1), (500, 532), (Mbig - 1, Mbig)):
        part = dig.linear(Ad[lo:hi].contiguous(), Wd, bd, out_dtype=dt, split_k=S)
        assert bits_equal(part, full[lo:hi]), (lo, hi)
    rows = [0, 531, Mbig - 1]
    Cref, D = oracle.linear_rows(A, W, b, Mbig, N, K, rows=rows)
    check_tolerance(to_f64(full[torch.tensor(rows, device="cuda")]), Cref, D, bf16_out,
                    "narrow linear")


@pytest.mark.parametrize("M,N,K,S", [
    (37, 300, 4096, 1),      # 64 wide: five tiles, the last 44 columns
    (37, 301, 4096, 1),      # N not a multiple of 4: the last columns stored one by one
    (200, 200, 4096, 2),     # two tile rows (the second ragged), two segments of 32 blocks
    (35, 130, 2112, 1),      # 33 K blocks
    (1200, 1000, 2048, 1),   # 128 wide: ten tile rows of eight tiles
])
@pytest.mark.parametrize("bf16_out", [False, True])
def test_narrow_edges_against_the_oracle(M, N, K, S, bf16_out):
    assert dig.bigemm_tile_n(M, N, K, S) in (64, 128)
    A, B = workloads.pair(M, N, K, 5 * M + N + K)
    C, buf = run_gemm(A, B, M, N, K, S, bf16_out)
    assert canary_intact(buf, M, N)
    Cref, D = oracle.gemm_rows(A, B, M, N, K)
    check_tolerance(to_f64(C), Cref, D, bf16_out, "narrow M=%d N=%d K=%d S=%d" % (M, N, K, S))


def test_narrow_partial_kernel_writes_the_slices_the_reduction_sums():
    """bigemm_run_partial (narrow) then bigemm_splitk_reduce gives bigemm_run's
    bits, and every slice element is written."""
    M, N, K, S = 16, 252, 65536, 16
    assert dig.bigemm_tile_n(M, N, K, S) == 64
    A, B = workloads.pair(M, N, K, 71)
    lda, ldb = round_up(K, 8), round_up(N, 8)
    Ad, Bd = device_matrix(A, lda), device_matrix(B, ldb)
    need = dig.bigemm_partial_workspace_bytes(M, N, K, S)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")   # NaN until written
    dig.bigemm_run_partial(Ad, Bd, M, N, K, lda, ldb, S, ws, need)
    C = output_buffer(M, N, N, False)
    dig.bigemm_splitk_reduce(ws, S, M, N, C, N, False)
    ref, _ = run_gemm(A, B, M, N, K, S)
    torch.cuda.synchronize()
    assert bits_equal(C[:M, :N], ref)
    slices = ws.view(torch.float32).view(S, M, dig.bigemm_workspace_ld(N))
    assert bool(torch.isfinite(slices[:, :, :N]).all())


def test_narrow_atomic_contrast_within_tolerance():
    M, N, K, S = 64, 256, 16384, 8
    assert dig.bigemm_tile_n(M, N, K, S) == 64
    A, B = workloads.pair(M, N, K, 81)
    C, buf = run_gemm(A, B, M, N, K, S, atomic=True)
    assert canary_intact(buf, M, N)
    Cref, D = oracle.gemm_rows(A, B, M, N, K)
    check_tolerance(to_f64(C), Cref, D, False, "narrow atomic")


def test_integer_exact_narrow_equals_the_oracle_bitwise():
    """Small integers, every partial sum below 2^24: FP32 is exact in any
    order, so the narrow path equals the binary64 oracle exactly."""
    M, N, K, S = 34, 192, 4096, 2
    assert dig.bigemm_tile_n(M, N, K, S) == 64
    g = workloads.generator(91)
    A = torch.randint(-8, 9, (M, K), generator=g).to(torch.bfloat16)
    B = torch.randint(-8, 9, (K, N), generator=g).to(torch.bfloat16)
    C, _ = run_gemm(A, B, M, N, K, S)
    Cref, _ = oracle.gemm_rows(A, B, M, N, K)
    assert (to_f64(C) == Cref).all()
