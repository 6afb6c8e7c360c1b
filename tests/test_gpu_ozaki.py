"""GPU: the Ozaki scheme's binary64 product on the bfloat16 tensor cores
(bigemm_ozaki_split, bigemm_ozaki_dgemm) against the binary64 oracle
(oracle.ozaki_split, oracle.ozaki_gemm) -- cuTile article, "倍精度行列積
エミュレーション".  The split is the Veltkamp split of eqs. (1)-(5); the
slice-pair products are exact in FP32 (eq. (11)); the binary64 sum of eq. (10)
runs in the same pair order on both sides, so the GPU's C must equal the
oracle's exactly, not just within a tolerance."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import deterministic_invariant_gemm_gb300 as dig
import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device(cuda_device):
    dig.load()
    yield
    assert dig.bigemm_device_status(reset=True) == 0


def wide(shape, seed, spread=20):
    """Normal values scaled over 2^-spread .. 2^spread, a few exact zeros."""
    g = workloads.generator(seed)
    x = torch.randn(shape, generator=g, dtype=torch.float64)
    e = torch.randint(-spread, spread + 1, shape, generator=g).double()
    x = x * torch.exp2(e)
    x.view(-1)[:: 97] = 0.0
    return x


def gpu_split(X, axis, rho, slices, out_rows=None):
    rows, cols = X.shape
    out_ld = cols + (-cols) % 8
    out_rows = rows if out_rows is None else out_rows
    plane_rows = rows if axis == 0 else out_rows
    out = torch.full((slices, plane_rows, out_ld), -1.0, dtype=torch.bfloat16, device="cuda")
    exps = torch.empty(rows if axis == 0 else cols, dtype=torch.int32, device="cuda")
    Xd = X.cuda()
    dig.bigemm_ozaki_split(Xd, rows, cols, cols, axis, rho, slices, out, out_ld, out_rows, exps)
    torch.cuda.synchronize()
    return out, exps


@pytest.mark.parametrize("axis", [0, 1])
@pytest.mark.parametrize("rows,cols,K", [
    (37, 300, 256),      # rho 45: 6 slices of width 9 (the split kernels' fixed shapes)
    (70, 64, 512),       # rho 46: 7 x 8
    (300, 37, 4096),     # rho 47: 8 x 7
    (64, 70, 8192),      # rho 48: 9 x 6
    (40, 33, 65536),     # rho 49: 11 x 5
    (5, 8, 1 << 20),     # rho 51: 18 slices, the general kernels
])
def test_split_matches_the_oracle_bit_for_bit(axis, rows, cols, K):
    X = wide((rows, cols), rows * cols + axis)
    X[0, 0] = -0.0
    X[1, :] = 0.0                               # an all-zero row
    X[2, 3] = 2.0 ** -1060                      # a subnormal
    X[3, 1] = 2.0 ** 30                         # a power-of-two maximum
    rho = dig.bigemm_ozaki_rho(K)
    assert rho == oracle.ozaki_rho(K)
    slices = dig.bigemm_ozaki_default_slices(K)
    S, c1, _ = oracle.ozaki_split(X, axis, rho, slices)
    out_rows = rows + 5 if axis == 1 else None
    got, exps = gpu_split(X, axis, rho, slices, out_rows)
    assert np.array_equal(exps.cpu().numpy(), c1)
    want = oracle.encode_rne(oracle.FMT_BF16, S)            # exact: every slice is a bf16 value
    assert np.array_equal(oracle.decode(oracle.FMT_BF16, want), S)
    have = got[:, :rows, :cols].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    # +0.0 and -0.0 slices are both zero terms: compare values, then bits of the nonzeros
    assert np.array_equal(oracle.decode(oracle.FMT_BF16, have), S)
    if axis == 1:
        assert (got[:, rows:, :cols].float() == 0).all()    # the padding rows are zeros


@pytest.mark.parametrize("axis", [0, 1])
def test_split_rounding_ties_match_the_oracle(axis):
    """Small integers, halves and quarters put many residuals exactly halfway
    between two multiples of a slice's unit, where the split rounds to the
    even neighbour: the GPU's slices must still equal the oracle's bit for
    bit, on a row long enough to take the register-cached and the re-read
    parts of the row kernel (9000 > 4096 columns) and an odd column count."""
    g = workloads.generator(515)
    rows, cols = (6, 9001) if axis == 0 else (9001, 6)
    X = torch.randint(-1000, 1001, (rows, cols), generator=g).double()
    X = X * torch.tensor([1.0, 0.5, 0.25, 8.0])[torch.randint(0, 4, (rows, cols), generator=g)]
    X[0, 0] = 1024.0 if axis == 0 else X[0, 0]
    for K in (4096, 1 << 16):
        rho = dig.bigemm_ozaki_rho(K)
        slices = dig.bigemm_ozaki_default_slices(K)
        S, c1, _ = oracle.ozaki_split(X, axis, rho, slices)
        got, exps = gpu_split(X, axis, rho, slices, rows + 3 if axis == 1 else None)
        assert np.array_equal(exps.cpu().numpy(), c1)
        have = got[:, :rows, :cols].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(oracle.decode(oracle.FMT_BF16, have), S), K


def run_dgemm(A, B, slices=0, d=0, ldc_pad=0):
    M, K = A.shape
    N = B.shape[1]
    ldc = N + (N & 1) + ldc_pad
    C = torch.full((M + 2, ldc), float("nan"), dtype=torch.float64, device="cuda")
    need = dig.bigemm_ozaki_workspace_bytes(M, N, K, slices)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    dig.bigemm_ozaki_dgemm(A.cuda(), B.cuda(), C, M, N, K, K, N, ldc, slices, d, ws, need)
    torch.cuda.synchronize()
    assert torch.isnan(C[:M, N:]).all() and torch.isnan(C[M:]).all()   # nothing written outside C
    return C[:M, :N].cpu().numpy()


@pytest.mark.parametrize("M,N,K,slices,d", [
    (64, 256, 512, 0, 0),
    (100, 70, 300, 0, 0),        # ragged: one partial tile, N not a multiple of 32
    (257, 300, 1000, 0, 0),      # three tile rows, two tile columns
    (130, 512, 4096, 0, 0),      # rho = 47: six-bit slices
    (64, 256, 512, 4, 3),        # Fast Mode: 6 pairs of 16
    (64, 256, 512, 7, 1),        # the leading pair alone
    (33, 96, 70, 3, 5),          # d beyond 2 (slices - 1): every pair
])
def test_dgemm_equals_the_oracle_exactly(M, N, K, slices, d):
    A = wide((M, K), M + K, 12)
    B = wide((K, N), N + K, 12)
    C = run_dgemm(A, B, slices, d)
    rho = oracle.ozaki_rho(K)
    s = slices or oracle.ozaki_default_slices(rho)
    Cref, inexact = oracle.ozaki_gemm(A, B, rho=rho, slices=s, d=d or s)
    assert inexact == 0
    assert np.array_equal(C, Cref)


def banded(shape, seed, axis):
    """Vectors (rows for axis 0, columns for axis 1) of different magnitude
    profiles -- flat (every entry near the maximum), normal, one dominant
    entry, wide exponents, now and then all zero -- so that Fast Mode's
    automatic d differs from element to element."""
    g = workloads.generator(seed)
    n, k = (shape[0], shape[1]) if axis == 0 else (shape[1], shape[0])
    x = torch.randn((n, k), generator=g, dtype=torch.float64)
    for v in range(n):
        kind = v % 5
        if kind == 0:                                       # flat: |x| in [0.75, 1]
            x[v] = torch.sign(x[v]) * (0.75 + 0.25 * torch.rand(k, generator=g, dtype=torch.float64))
        elif kind == 2:                                     # one entry dominates
            x[v] *= 2.0 ** -30
            x[v, v % k] = 2.0 ** 10
        elif kind == 3:                                     # wide exponents
            x[v] *= torch.exp2(torch.randint(-20, 21, (k,), generator=g).double())
        elif kind == 4 and v % 10 == 4:
            x[v] = 0.0
    return x if axis == 0 else x.t().contiguous()


@pytest.mark.parametrize("M,N,K,slices", [
    (100, 70, 300, 12),          # ragged, one partial tile; more slices than the default 7
    (257, 300, 1000, 11),        # three tile rows, two tile columns
    (130, 512, 4096, 0),         # the default slices (8 at rho = 47)
    (5, 40, 70000, 0),           # long K (14 slices)
])
def test_fast_mode_automatic_d_equals_the_oracle_exactly(M, N, K, slices):
    """d = -1 (Fast Mode's automatic d, "Fast Mode（GEMMの削減）"): each
    element takes the pairs p + q < d_ij that the oracle takes, so C equals the
    oracle's bit for bit; the inputs make d_ij vary, and some pairs are skipped."""
    A = banded((M, K), 3 * M + K, 0)
    B = banded((K, N), 5 * N + K, 1)
    rho = oracle.ozaki_rho(K)
    s = slices or oracle.ozaki_default_slices(rho)
    D, _, _ = oracle.ozaki_fast_d(A, B, rho=rho, slices=s)
    assert D.min() < D.max() == s              # d varies; the zero vectors take every pair
    C = run_dgemm(A, B, slices, -1, ldc_pad=6)
    Cref, inexact = oracle.ozaki_gemm(A, B, rho=rho, slices=s, d=-1)
    assert inexact == 0
    assert np.array_equal(C.view(np.int64), Cref.view(np.int64))


def test_fast_mode_rows_are_batch_invariant():
    """d_ij depends on row i of A and column j of B only (their masses), so
    Fast Mode's rows are the same at M = 1, in a window and in the full batch."""
    M, N, K = 300, 384, 777
    A = banded((M, K), 15, 0)
    B = banded((K, N), 16, 1)
    full = run_dgemm(A, B, 10, -1)
    for lo, hi in ((0, 1), (1, 2), (2, 3), (128, 129), (299, 300), (37, 170)):
        part = run_dgemm(A[lo:hi].clone(), B, 10, -1)
        assert np.array_equal(part.view(np.int64), full[lo:hi].view(np.int64)), (lo, hi)


def test_fast_mode_meets_the_pages_bound_on_normal_data():
    """On normal data with K = 4096 the automatic d skips pairs the default
    keeps (d < slices for most elements), C equals the oracle's, and the error
    against exact rational products stays within the page's 2 sqrt(k) u |A||B|."""
    M, N, K = 64, 96, 4096
    g = workloads.generator(81)
    A = torch.randn(M, K, generator=g, dtype=torch.float64)
    B = torch.randn(K, N, generator=g, dtype=torch.float64)
    C = run_dgemm(A, B, 0, -1)
    D, _, _ = oracle.ozaki_fast_d(A, B)
    s = oracle.ozaki_default_slices(oracle.ozaki_rho(K))
    assert (D < s).mean() > 0.5
    Cref, _ = oracle.ozaki_gemm(A, B, d=-1)
    assert np.array_equal(C.view(np.int64), Cref.view(np.int64))
    a, b = A.numpy(), B.numpy()
    scale = np.abs(a) @ np.abs(b)
    for i, j in ((0, 0), (10, 40), (63, 95), (7, 70)):
        exact = sum((Fraction(a[i, k]) * Fraction(b[k, j]) for k in range(K)), Fraction(0))
        err = abs(float(Fraction(C[i, j]) - exact))
        assert err <= 2 * np.sqrt(K) * 2.0 ** -53 * scale[i, j], (i, j, err / scale[i, j])


@pytest.mark.parametrize("M,N,K,slices,d", [
    (257, 300, 1000, 0, 0),      # two pair tile rows, the second with one row
    (300, 384, 777, 0, 0),       # CTA 1 of the second tile row has no rows
    (512, 768, 1024, 4, 3),      # Fast Mode, fixed d
    (256, 512, 4096, 0, -1),     # Fast Mode, automatic d
])
def test_pair_kernel_equals_the_1sm_kernel_and_the_oracle(M, N, K, slices, d):
    """The slice-pair products on CTA pairs (256 x 256 tiles, each CTA adding
    its 128 rows under its own 128 x 256 tile's count): the bits of the 1-SM
    kernel and of the oracle."""
    A = wide((M, K), 2 * M + K, 10)
    B = wide((K, N), 2 * N + K, 10)
    prev = dig.bigemm_set_pair_mode(dig.PAIR_ALWAYS)
    try:
        pair = run_dgemm(A, B, slices, d)
        dig.bigemm_set_pair_mode(dig.PAIR_NEVER)
        single = run_dgemm(A, B, slices, d)
    finally:
        dig.bigemm_set_pair_mode(prev)
    assert np.array_equal(pair.view(np.int64), single.view(np.int64))
    rho = oracle.ozaki_rho(K)
    s = slices or oracle.ozaki_default_slices(rho)
    Cref, _ = oracle.ozaki_gemm(A, B, rho=rho, slices=s, d=d if d < 0 else (d or s))
    assert np.array_equal(pair.view(np.int64), Cref.view(np.int64))


@pytest.mark.parametrize("pair_mode", ["never", "always"])
def test_staged_epilogue_rows_far_apart_equal_the_oracle(pair_mode):
    """C rows at least 8192 elements apart take the epilogue that reads and
    writes C through shared memory: a padded ldc puts a small, ragged product
    on it (single CTAs and CTA pairs); the bits are the oracle's."""
    M, N, K = 300, 320, 500
    A = wide((M, K), 97, 12)
    B = wide((K, N), 98, 12)
    prev = dig.bigemm_set_pair_mode(dig.PAIR_NEVER if pair_mode == "never" else dig.PAIR_ALWAYS)
    try:
        C = run_dgemm(A, B, 0, 0, ldc_pad=8192 - N)
        Cf = run_dgemm(A, B, 0, -1, ldc_pad=8192 - N)
    finally:
        dig.bigemm_set_pair_mode(prev)
    Cref, _ = oracle.ozaki_gemm(A, B)
    assert np.array_equal(C.view(np.int64), Cref.view(np.int64))
    Cref_f, _ = oracle.ozaki_gemm(A, B, d=-1)
    assert np.array_equal(Cf.view(np.int64), Cref_f.view(np.int64))


def test_dgemm_accuracy_against_exact_products():
    """1024^3 normal inputs: rows computed by the oracle match exactly, and
    the error against exact rational products on a sample is binary64's."""
    M = N = K = 1024
    g = workloads.generator(77)
    A = torch.randn(M, K, generator=g, dtype=torch.float64)
    B = torch.randn(K, N, generator=g, dtype=torch.float64)
    C = run_dgemm(A, B)
    rows = [0, 511, 1023]
    Cref, _ = oracle.ozaki_gemm(A[rows], B)                 # rows split alone: the same slices
    assert np.array_equal(C[rows], Cref)
    a, b = A.numpy(), B.numpy()
    scale = np.abs(a) @ np.abs(b)
    for i, j in ((0, 0), (511, 700), (1023, 1023), (17, 999)):
        exact = sum((Fraction(a[i, k]) * Fraction(b[k, j]) for k in range(K)), Fraction(0))
        err = abs(float(Fraction(C[i, j]) - exact))
        assert err <= 8 * 2.0 ** -53 * scale[i, j], (i, j, err / scale[i, j])
    # and against numpy's own binary64 product, elementwise on the whole matrix
    assert np.max(np.abs(C - a @ b) / scale) < 1e-14


def test_dgemm_rows_are_batch_invariant():
    """Each row of A is split by its own maximum, so row i of C is the same at
    M = 1, inside a window and inside the full batch, bit for bit."""
    M, N, K = 300, 384, 777
    A = wide((M, K), 5, 8)
    B = wide((K, N), 6, 8)
    full = run_dgemm(A, B)
    for lo, hi in ((0, 1), (128, 129), (299, 300), (37, 170)):
        part = run_dgemm(A[lo:hi].clone(), B)
        assert np.array_equal(part.view(np.int64), full[lo:hi].view(np.int64)), (lo, hi)


def test_dgemm_bit_stable_over_10_runs():
    A = wide((256, 512), 8, 4)
    B = wide((512, 256), 9, 4)
    first = run_dgemm(A, B)
    for _ in range(9):
        assert np.array_equal(run_dgemm(A, B).view(np.int64), first.view(np.int64))


def test_dgemm_small_integers_exact():
    g = workloads.generator(3)
    A = torch.randint(-1000, 1001, (96, 200), generator=g).double()
    B = torch.randint(-1000, 1001, (200, 130), generator=g).double()
    C = run_dgemm(A, B)
    assert np.array_equal(C, (A.long() @ B.long()).double().numpy())


def test_dgemm_wrapper_and_edge_cases():
    A = torch.randn(40, 50, dtype=torch.float64, device="cuda")
    B = torch.randn(50, 33, dtype=torch.float64, device="cuda")
    C = dig.ozaki_matmul(A, B)
    assert dig.bigemm_last_launch_count() == 4
    torch.cuda.synchronize()
    assert torch.allclose(C, A @ B, rtol=0, atol=1e-13)
    # K = 0: the empty sum
    Z = dig.ozaki_matmul(torch.zeros(4, 0, dtype=torch.float64, device="cuda"),
                         torch.zeros(0, 6, dtype=torch.float64, device="cuda"))
    assert torch.equal(Z.cpu(), torch.zeros(4, 6, dtype=torch.float64))
    # argument checks: odd ldc, missing workspace, bad slice count
    c = torch.empty(40, 33, dtype=torch.float64, device="cuda")
    assert dig.bigemm_ozaki_dgemm(A, B, c, 40, 33, 50, 50, 33, 33, 0, 0, None, 0, check=False) == 2
    c2 = torch.empty(40, 34, dtype=torch.float64, device="cuda")
    assert dig.bigemm_ozaki_dgemm(A, B, c2, 40, 33, 50, 50, 33, 34, 0, 0, None, 0, check=False) == 3
    assert dig.bigemm_ozaki_dgemm(A, B, c2, 40, 33, 50, 50, 33, 34, 33, 0, None, 0, check=False) == 1


def test_concurrent_products_on_two_streams_and_a_graph_replay():
    """The slice-pair kernel's CTAs wait on one another (a tile's pairs run on
    different CTAs, in pair order), so it is a cooperative launch: two products
    enqueued on two streams at once, each with a CTA on every SM, must both
    finish (no bounded wait may run out) with the serial results' bits, and so
    must a CUDA graph replay of one."""
    shapes = [(512, 768, 1024, 21), (640, 512, 2048, 22)]
    data = []
    for M, N, K, seed in shapes:
        A = wide((M, K), seed, 8).cuda()
        B = wide((K, N), seed + 1, 8).cuda()
        data.append((A, B))
    serial = [dig.ozaki_matmul(A, B) for A, B in data]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in data]
    outs = []
    for _ in range(3):
        outs = []
        torch.cuda.current_stream().synchronize()
        for (A, B), st in zip(data, streams):
            with torch.cuda.stream(st):
                outs.append(dig.ozaki_matmul(A, B, stream=st))
        torch.cuda.synchronize()
        assert dig.bigemm_device_status(reset=True) == 0
        for got, want in zip(outs, serial):
            assert torch.equal(got.view(torch.int64), want.view(torch.int64))
    A, B = data[0]
    M, K = A.shape
    N = B.shape[1]
    C = torch.empty((M, N), dtype=torch.float64, device="cuda")
    ws = torch.empty(dig.bigemm_ozaki_workspace_bytes(M, N, K, 0), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        dig.ozaki_matmul(A, B, out=C, workspace=ws, stream=s)
    for _ in range(2):
        C.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(C.view(torch.int64), serial[0].view(torch.int64))
    assert dig.bigemm_device_status(reset=True) == 0


def test_dgemm_4096_rows_equal_the_oracle_and_one_row_products():
    """A 4096^3 product (36 slice pairs dealt over every SM, 18432 items):
    sampled rows equal the oracle's exactly and the same rows of one-row
    products, bit for bit; also with Fast Mode's fixed and automatic d."""
    M = N = K = 4096
    g = workloads.generator(79)
    A = torch.randn(M, K, generator=g, dtype=torch.float64)
    B = torch.randn(K, N, generator=g, dtype=torch.float64)
    rows = [0, 3071, 3072, 4095]
    for d in (0, 6, -1):
        C = run_dgemm(A, B, 0, d)
        s = oracle.ozaki_default_slices(oracle.ozaki_rho(K))
        Cref, _ = oracle.ozaki_gemm(A[rows], B, d=d or s)
        assert np.array_equal(C[rows], Cref), d
        for r in rows[1:3]:
            one = run_dgemm(A[r:r + 1].clone(), B, 0, d)
            assert np.array_equal(one.view(np.int64), C[r:r + 1].view(np.int64)), (d, r)
