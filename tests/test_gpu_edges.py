"""GPU: every switch between the library's execution paths, at both sides of
its edge.  The path a product takes depends on its shape (and, between the
cluster and workspace paths, on the device's cluster capacity); the bits must
not.  At each edge the same rows are computed on both sides and alone (M = 1,
the few-row kernel), and compared bit for bit; the columns two products with
different N share must also agree.  (Tencent AI-infra article "腾讯エンジニア：
大規模モデルの出力を確定させるための AI インフラ手法", "Batch Invariance の由来":
a row's reduction order may depend on K and the split only.)"""
import pytest
import torch

import deterministic_invariant_gemm_gb300 as dig
import workloads
from gemm_check import bits_equal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device(cuda_device):
    dig.load()
    yield
    assert dig.bigemm_device_status(reset=True) == 0


def cdiv(a, b):
    return -(-a // b)


def rows_alone(A, B, rows, S):
    """Each row computed in a batch of one (the few-row kernel)."""
    return torch.cat([dig.matmul(A[r:r + 1].contiguous(), B, split_k=S) for r in rows])


def check_edge(A, B, M_lo, M_hi, N_lo, N_hi, S, want_lo, want_hi):
    """Products (M_lo, N_lo) and (M_hi, N_hi) on paths want_lo / want_hi:
    their common rows and columns agree bitwise, and sampled rows equal the
    same rows computed alone."""
    K = A.shape[1]
    assert dig.bigemm_split_path(M_lo, N_lo, K, S) == want_lo, (M_lo, N_lo, K, S)
    assert dig.bigemm_split_path(M_hi, N_hi, K, S) == want_hi, (M_hi, N_hi, K, S)
    lo = dig.matmul(A[:M_lo].contiguous(), B[:, :N_lo].contiguous(), split_k=S)
    hi = dig.matmul(A[:M_hi].contiguous(), B[:, :N_hi].contiguous(), split_k=S)
    m, n = min(M_lo, M_hi), min(N_lo, N_hi)
    assert bits_equal(lo[:m, :n], hi[:m, :n])
    rows = sorted({0, m // 2, m - 1})
    alone = rows_alone(A, B[:, :n].contiguous(), rows, S)
    assert bits_equal(alone, hi[rows, :n])


def test_fold_edge_rows_96_97():
    """Folding starts at 97 rows (with at least 128 tiles): 96 rows take the
    workspace path, 97 fold."""
    K, S = 1024, 2
    N = 128 * 256
    A, B = workloads.pair(97, N, K, 501, a_std=1.0, b_std=0.1)
    A, B = A.cuda(), B.cuda()
    check_edge(A, B, 96, 97, N, N, S, dig.PATH_WORKSPACE, dig.PATH_FOLDED)


def test_fold_edge_tiles_127_128():
    """Folding needs 128 tiles of 128 x 256: 100 rows against 127 tile
    columns take the workspace path, against 128 (eight columns more) they
    fold."""
    K, S = 1024, 2
    A, B = workloads.pair(100, 128 * 256, K, 502, a_std=1.0, b_std=0.1)
    A, B = A.cuda(), B.cuda()
    # (one tile more with eight more columns: B's rows stay 16-byte multiples)
    check_edge(A, B, 100, 100, 127 * 256, 127 * 256 + 8, S, dig.PATH_WORKSPACE, dig.PATH_FOLDED)


def test_cluster_capacity_edge():
    """A split product clusters while its tiles fit the device's cluster
    capacity for its split; one tile more and it takes the workspace path."""
    K, S = 4096, 8
    cap = dig.bigemm_cluster_capacity(S)
    assert cap >= 1
    M = 40                                   # past the few-row kernel, one tile row
    N_fit, N_over = cap * 256, cap * 256 + 8
    A, B = workloads.pair(M, N_over, K, 503, a_std=1.0, b_std=0.02)
    A, B = A.cuda(), B.cuda()
    check_edge(A, B, M, M, N_fit, N_over, S, dig.PATH_CLUSTER, dig.PATH_WORKSPACE)


def test_few_row_edge_32_33():
    """The few-row kernel takes up to 32 rows; 33 rows go to the cluster path
    (one tile row of 8 tiles fits every GB300's cluster capacity)."""
    K, S, N = 4096, 8, 2048
    A, B = workloads.pair(33, N, K, 504, a_std=1.0, b_std=0.02)
    A, B = A.cuda(), B.cuda()
    check_edge(A, B, 32, 33, N, N, S, dig.PATH_SKINNY, dig.PATH_CLUSTER)


def width_edges(N, K, S):
    """Batch sizes on either side of each switch of bigemm_tile_n's rule on
    this device: the rule takes the widest of 256 and 128 whose units
    (tile rows x tile columns x segments) reach half the SMs, else 64."""
    half = torch.cuda.get_device_properties(0).multi_processor_count // 2
    s = dig.bigemm_effective_split_k(K, S)
    m128 = cdiv(half, cdiv(N, 128) * s)      # tile rows where 128-wide units reach half
    m256 = cdiv(half, cdiv(N, 256) * s)
    return [(128 * (m128 - 1), 64), (128 * (m128 - 1) + 1, 128),
            (128 * (m256 - 1), 128), (128 * (m256 - 1) + 1, 256)]


def test_tile_width_edges():
    """Rows on both sides of each width switch (64 | 128 | 256 columns) equal
    the same rows of the widest product and the rows computed alone."""
    N, K, S = 256, 65536, 8
    edges = width_edges(N, K, S)
    Mbig = max(m for m, _ in edges)
    A, B = workloads.pair(Mbig, N, K, 505, a_std=1.0, b_std=0.02)
    A, B = A.cuda(), B.cuda()
    full = dig.matmul(A, B, split_k=S)
    for m, w in edges:
        assert dig.bigemm_tile_n(m, N, K, S) == w, (m, w)
        part = dig.matmul(A[:m].contiguous(), B, split_k=S)
        assert bits_equal(part, full[:m]), (m, w)
    rows = [0, edges[0][0] - 1, Mbig - 1]
    assert bits_equal(rows_alone(A, B, rows, S), full[rows])
