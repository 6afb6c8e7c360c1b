"""GPU: a seeded sweep across the path rule.  For each shape (N, K, split_k,
layout of the second operand, output dtype, bias) the first M rows of one A
are multiplied for a ladder of batch sizes M that crosses every switch of the
rule -- the few-row kernel (M <= 32, split <= 8), the cluster and workspace
sums, the fold (M >= 97 with at least 128 tiles), the narrow tiles of small
long-K products and the CTA pairs (pair tiles filling two waves) -- and every
row must carry the same bits in every product, whatever path computed it.
Rows of the largest product are checked against the binary64 oracle.
(Tencent AI-infra article "腾讯エンジニア：大規模モデルの出力を確定させるための
AI インフラ手法", "Batch Invariance の由来": the reduction order of an element
depends on K and the tile configuration only, never on M.)"""
import random

import pytest
import torch

import deterministic_invariant_gemm_gb300 as dig
import oracle
import workloads
from gemm_check import bits_equal, check_tolerance, to_f64

pytestmark = pytest.mark.gpu

LADDER = (1, 5, 16, 32, 33, 64, 96, 97, 128, 200, 256, 257, 512, 1024, 2048, 4096)


@pytest.fixture(scope="module", autouse=True)
def _device(cuda_device):
    dig.load()
    dig.bigemm_set_pair_mode(dig.PAIR_AUTO)
    yield
    assert dig.bigemm_device_status(reset=True) == 0


def fixed_shapes():
    """Shapes chosen so that each switch is crossed on the ladder (the pair
    shape's N gives 256 x 256 tiles for two waves of pairs at M = 4096)."""
    cap = dig.bigemm_pair_capacity()
    n_pair = 256 * -(-2 * cap // 16) - 40
    return [
        # (N, K, split_k, wt, bf16_out, bias, M max)
        (4096, 4096, 8, False, False, False, 1024),    # decode shape: few-row, workspace, fold at 128 tiles
        (3840, 4096, 8, True, True, True, 512),        # clusters of 8 below the fold
        (4096, 2048, 4, False, True, False, 1024),     # folds at M = 1024 (128 tiles); clusters, workspace, few-row below
        (n_pair, 1000, 1, False, False, False, 4096),  # CTA pairs at the top of the ladder
        (n_pair, 2048, 0, True, False, True, 4096),    # default split (4): folds, pairs at 4096
        (512, 16384, 4, False, False, False, 4096),    # narrow tiles below, wide at 4096
        (264, 8192, 16, True, True, False, 1024),      # split 16: never the few-row kernel
    ]


def seeded_shapes(n=16, seed=20261202):
    r = random.Random(seed)
    out = []
    for _ in range(n):
        N = max(8, 256 * r.randint(1, 24) + r.choice((0, -8, -40, 24)))
        K = r.choice((64, 520, 1000, 2048, 4096, 8192))
        S = r.choice((0, 1, 2, 4, 8, 16))
        S = min(S, -(-K // 64)) if S else 0       # at most one segment per K block of 64
        wt = r.random() < 0.5
        out.append((N, K, S, wt, r.random() < 0.5, wt and r.random() < 0.5, r.choice((1024, 2048, 4096))))
    return out


def product(A, B, b, M, wt, bf16_out, S):
    dt = torch.bfloat16 if bf16_out else torch.float32
    a = A[:M].contiguous()
    if wt:
        return dig.linear(a, B, b, out_dtype=dt, split_k=S)
    return dig.matmul(a, B, out_dtype=dt, split_k=S)


def run_shape(N, K, S, wt, bf16_out, bias, m_max, seen):
    A = workloads.normal_bf16((m_max, K), N + 7 * K + S).cuda()
    B = workloads.normal_bf16((N, K) if wt else (K, N), 3 * N + K, 0.05).cuda()
    b = workloads.normal_bf16((N,), N + 1).cuda() if bias else None
    full = product(A, B, b, m_max, wt, bf16_out, S)
    torch.cuda.synchronize()
    for M in LADDER:
        if M > m_max:
            break
        seen.add(("path", dig.bigemm_split_path(M, N, K, S)))
        seen.add(("pair", dig.bigemm_uses_pair(M, N, K, S)))
        seen.add(("narrow", dig.bigemm_tile_n(M, N, K, S) < 256))
        C = full if M == m_max else product(A, B, b, M, wt, bf16_out, S)
        torch.cuda.synchronize()
        assert bits_equal(C, full[:M]), (N, K, S, wt, bf16_out, bias, M)
    rows = [0, m_max // 2, m_max - 1]
    if wt:
        Cref, D = oracle.linear_rows(A.cpu(), B.cpu(), b.cpu() if bias else None, m_max, N, K, rows=rows)
    else:
        Cref, D = oracle.gemm_rows(A.cpu(), B.cpu(), m_max, N, K, rows=rows)
    check_tolerance(to_f64(full[torch.tensor(rows, device="cuda")]), Cref, D, bf16_out, "sweep")


def test_every_path_switch_keeps_row_bits():
    seen = set()
    for shape in fixed_shapes():
        run_shape(*shape, seen)
    # the fixed shapes cross every switch of the rule on their ladders
    for key in (("path", dig.PATH_SKINNY), ("path", dig.PATH_CLUSTER), ("path", dig.PATH_WORKSPACE),
                ("path", dig.PATH_FOLDED), ("path", dig.PATH_UNSPLIT), ("pair", 1), ("pair", 0),
                ("narrow", True), ("narrow", False)):
        assert key in seen, key


@pytest.mark.parametrize("shape", seeded_shapes(), ids=lambda s: "N%d_K%d_S%d_%s_%s%s" % (
    s[0], s[1], s[2], "W" if s[3] else "B", "bf16" if s[4] else "f32", "_bias" if s[5] else ""))
def test_seeded_shapes_keep_row_bits(shape):
    run_shape(*shape, set())
