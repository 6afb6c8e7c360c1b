"""Pins for the CPU oracle (no GPU).

Each test ties an oracle function to something other than the oracle itself:
the pages' FP16 worked example, IEEE-754 field definitions checked
exhaustively against torch's own conversions, exact integer / rational
arithmetic, identity and permutation products, hand-computed binary32 sums and
the BF16 exact-accumulation claim of the cuTile/Ozaki article.  A plausible
slip in the oracle (a dropped term, a wrong sign, a transposed operand, an
index off by one, a wrong tie rule) fails at least one of them.
"""
import os
import random
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).numpy().view(np.uint16)


# --------------------------------------------------------------------------
# Codecs and the FP16 worked example
# --------------------------------------------------------------------------

def _golden_lines(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line


def test_fp16_worked_example_encodings():
    n = 0
    for line in _golden_lines("fp16_worked_example.txt"):
        parts = line.split()
        if parts[0] != "encoding":
            continue
        value, e_unb, e_bits, frac = float(parts[1]), int(parts[2]), parts[3], parts[4]
        bits = int(oracle.encode_rne(oracle.FMT_FP16, [value])[0])
        assert (bits >> 15) == 0
        biased = (bits >> 10) & 0x1F
        assert biased - 15 == e_unb, line
        if e_bits != "-":
            assert biased == int(e_bits, 2), line
        assert (bits & 0x3FF) == int(frac, 2), line
        assert oracle.decode(oracle.FMT_FP16, [bits])[0] == value
        n += 1
    assert n == 6


def test_fp16_worked_example_sum_and_ulp():
    seen = 0
    for line in _golden_lines("fp16_worked_example.txt"):
        parts = line.split()
        if parts[0] == "sum":
            a, b, want = map(float, parts[1:])
            assert oracle.fp16_add(a, b) == want
            seen += 1
        elif parts[0] == "ulp":
            x, want = map(float, parts[1:])
            assert oracle.ulp(oracle.FMT_FP16, x) == want
            seen += 1
    assert seen == 2
    # 2049 itself is not representable: it sits exactly halfway between its
    # neighbours, and ties go to the even fraction (2048: ...0000000000).
    assert oracle.decode(oracle.FMT_FP16, oracle.encode_rne(oracle.FMT_FP16, [2049.0]))[0] == 2048.0
    # 2051 is halfway between 2050 (fraction ...01, odd) and 2052 (...10, even).
    assert oracle.fp16_add(2048.0, 3.0) == 2052.0
    # slightly above the midpoint rounds up
    assert oracle.decode(oracle.FMT_FP16, oracle.encode_rne(oracle.FMT_FP16, [2049.0001]))[0] == 2050.0


def test_bf16_analogue_of_worked_example():
    # bfloat16 keeps 7 fraction bits: ULP(256) = 2^(8 - 7) = 2, and 256 + 1
    # (halfway between 256 and 258) rounds to the even neighbour 256.
    assert oracle.ulp(oracle.FMT_BF16, 256.0) == 2.0
    assert oracle.bf16_round([257.0])[0] == 256.0
    assert oracle.bf16_round([259.0])[0] == 260.0
    assert oracle.ulp(oracle.FMT_BF16, 1.0) == 2.0 ** -7


@pytest.mark.parametrize("fmt,tdtype", [(oracle.FMT_BF16, torch.bfloat16),
                                        (oracle.FMT_FP16, torch.float16)])
def test_decode_exhaustive_against_torch(fmt, tdtype):
    pats = np.arange(65536, dtype=np.uint16)
    ours = oracle.decode(fmt, pats)
    ref = torch.from_numpy(pats.view(np.int16).copy()).view(tdtype).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zeros decode with their sign
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


@pytest.mark.parametrize("fmt", [oracle.FMT_BF16, oracle.FMT_FP16])
def test_encode_decode_round_trip_exhaustive(fmt):
    pats = np.arange(65536, dtype=np.uint16)
    vals = oracle.decode(fmt, pats)
    finite = ~np.isnan(vals)
    back = oracle.encode_rne(fmt, vals[finite])
    assert np.array_equal(back, pats[finite])


@pytest.mark.parametrize("fmt,tdtype", [(oracle.FMT_BF16, torch.bfloat16),
                                        (oracle.FMT_FP16, torch.float16)])
def test_encode_matches_torch_rounding(fmt, tdtype):
    g = torch.Generator().manual_seed(7)
    # wide dynamic range, including subnormals and overflow for fp16
    mant = torch.rand(200000, generator=g, dtype=torch.float64) * 2 - 1
    expo = torch.randint(-40, 40, (200000,), generator=g).to(torch.float64)
    x32 = (mant * torch.pow(2.0, expo)).to(torch.float32)
    # exact midpoints between neighbouring bf16/fp16 values, both parities
    pats = torch.randint(0, 0x7B00, (20000,), generator=g, dtype=torch.int32).to(torch.int16)
    lo = pats.view(tdtype).to(torch.float64)
    hi = (pats + 1).view(tdtype).to(torch.float64)
    mid = ((lo + hi) / 2).to(torch.float32)
    x32 = torch.cat([x32, mid, -mid])
    ours = oracle.encode_rne(fmt, x32.to(torch.float64).numpy())
    ref = x32.to(tdtype).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


# --------------------------------------------------------------------------
# The product C = A B and the scale D = sum |a b|
# --------------------------------------------------------------------------

def _exact_product(A: torch.Tensor, B: torch.Tensor):
    """Exact C and D with Python integers scaled by a common power of two."""
    a = A.to(torch.float64).numpy()
    b = B.to(torch.float64).numpy()
    M, K = a.shape
    N = b.shape[1]
    C = [[Fraction(0)] * N for _ in range(M)]
    D = [[Fraction(0)] * N for _ in range(M)]
    for i in range(M):
        for j in range(N):
            s = Fraction(0)
            d = Fraction(0)
            for k in range(K):
                p = Fraction(float(a[i, k])) * Fraction(float(b[k, j]))
                s += p
                d += abs(p)
            C[i][j] = s
            D[i][j] = d
    return C, D


def test_identity_gives_B_exactly():
    K, N = 96, 40
    B = workloads.normal_bf16((K, N), 11)
    A = torch.eye(K, dtype=torch.bfloat16)
    C, D = oracle.gemm_rows(_bits(A), _bits(B), K, N, K)
    Bd = B.to(torch.float64).numpy()
    assert np.array_equal(C, Bd)
    assert np.array_equal(D, np.abs(Bd))


def test_permutations_move_rows_and_columns():
    K, N = 37, 29
    rng = np.random.default_rng(3)
    p = rng.permutation(K)
    q = rng.permutation(N)
    B = workloads.normal_bf16((K, N), 12)
    P = torch.zeros(K, K, dtype=torch.bfloat16)
    P[np.arange(K), p] = 1          # (P B)[i] = B[p[i]]
    C, _ = oracle.gemm_rows(_bits(P), _bits(B), K, N, K)
    Bd = B.to(torch.float64).numpy()
    assert np.array_equal(C, Bd[p])
    # right-multiplying by a permutation matrix permutes columns
    Q = torch.zeros(N, N, dtype=torch.bfloat16)
    Q[q, np.arange(N)] = 1          # (B Q)[:, j] = B[:, q[j]]
    C2, _ = oracle.gemm_rows(_bits(B), _bits(Q), K, N, N)
    assert np.array_equal(C2, Bd[:, q])


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (7, 13, 64), (33, 70, 515), (5, 300, 4096)])
def test_small_integers_exact(M, N, K):
    A, B = workloads.pair(M, N, K, 100 + K, dist="int")
    C, D = oracle.gemm_rows(_bits(A), _bits(B), M, N, K)
    ai = A.to(torch.int64).numpy()
    bi = B.to(torch.int64).numpy()
    assert np.array_equal(C, (ai @ bi).astype(np.float64))
    assert np.array_equal(D, (np.abs(ai) @ np.abs(bi)).astype(np.float64))


@pytest.mark.parametrize("seed", [1, 2, 3, 4])
def test_brute_force_rational_tiny(seed):
    rnd = random.Random(seed)
    M, N, K = rnd.randint(1, 5), rnd.randint(1, 5), rnd.randint(1, 6)
    A, B = workloads.pair(M, N, K, 500 + seed)
    C, D = oracle.gemm_rows(_bits(A), _bits(B), M, N, K)
    Ce, De = _exact_product(A, B)
    u = 2.0 ** -53
    for i in range(M):
        for j in range(N):
            # binary64 recursive summation: |C - exact| <= (K-1) u D (+ higher order)
            err = abs(Fraction(C[i, j]) - Ce[i][j])
            assert err <= Fraction(K * u) * De[i][j]
            assert Fraction(D[i, j]) - De[i][j] <= Fraction(K * u) * De[i][j]
            assert D[i, j] >= abs(C[i, j]) * (1 - K * u)


def test_exactly_representable_sums_are_exact():
    # power-of-two entries with nearby exponents: every partial sum fits 53 bits
    g = torch.Generator().manual_seed(5)
    M, N, K = 4, 6, 40
    ea = torch.randint(-4, 4, (M, K), generator=g).to(torch.float64)
    eb = torch.randint(-4, 4, (K, N), generator=g).to(torch.float64)
    sa = torch.randint(0, 2, (M, K), generator=g).to(torch.float64) * 2 - 1
    A = (sa * torch.pow(2.0, ea)).to(torch.bfloat16)
    B = torch.pow(2.0, eb).to(torch.bfloat16)
    C, _ = oracle.gemm_rows(_bits(A), _bits(B), M, N, K)
    Ce, _ = _exact_product(A, B)
    for i in range(M):
        for j in range(N):
            assert Fraction(C[i, j]) == Ce[i][j]


def test_sign_and_scale_relations():
    M, N, K = 9, 17, 130
    A, B = workloads.pair(M, N, K, 77)
    C, D = oracle.gemm_rows(_bits(A), _bits(B), M, N, K)
    Cn, Dn = oracle.gemm_rows(_bits(-A), _bits(B), M, N, K)
    assert np.array_equal(Cn, -C)
    assert np.array_equal(Dn, D)
    Ap, Bp = A.abs(), B.abs()
    Cp, Dp = oracle.gemm_rows(_bits(Ap), _bits(Bp), M, N, K)
    assert np.array_equal(Cp, Dp)
    assert np.array_equal(Dp, D)
    assert np.all(D >= np.abs(C))


def test_row_selection_and_leading_dimensions():
    M, N, K = 23, 31, 77
    A, B = workloads.pair(M, N, K, 88)
    C, D = oracle.gemm_rows(_bits(A), _bits(B), M, N, K)
    rows = [22, 0, 5, 5, 13]
    Cs, Ds = oracle.gemm_rows(_bits(A), _bits(B), M, N, K, rows=rows)
    assert np.array_equal(Cs, C[rows])
    assert np.array_equal(Ds, D[rows])
    # padded storage: the padding holds NaN, which must never be read
    Ap = workloads.padded(A, 88)
    Bp = workloads.padded(B, 40)
    Cpad, Dpad = oracle.gemm_rows(_bits(Ap.as_strided((M, 88), (88, 1))),
                                  _bits(Bp.as_strided((K, 40), (40, 1))),
                                  M, N, K, lda=88, ldb=40)
    assert np.array_equal(Cpad, C)
    assert np.array_equal(Dpad, D)


def test_bad_arguments_rejected():
    A = np.zeros((2, 2), np.uint16)
    with pytest.raises(ValueError):
        oracle.gemm_rows(A, A, 2, 2, 2, rows=[2])
    with pytest.raises(ValueError):
        oracle.gemm_rows(A, A, 2, 2, 2, lda=1)


def test_empty_shapes():
    C, D = oracle.gemm_rows(np.zeros(0, np.uint16), np.zeros(0, np.uint16), 0, 0, 0)
    assert C.shape == (0, 0)
    # K = 0: the empty sum is +0.0
    C, D = oracle.gemm_rows(np.zeros(3, np.uint16), np.zeros(4, np.uint16), 3, 4, 0)
    assert np.array_equal(C, np.zeros((3, 4))) and not np.signbit(C).any()


def test_bf16_slices_accumulate_exactly_in_fp32():
    """cuTile/Ozaki article (techplay.jp, "最適化後の結果"): 8-bit x 8-bit
    significand products fit in 16 bits, so 128 of them fit 16 + 7 = 23 <= 24
    bits and their binary32 sum is exact -- for slices that share one
    power-of-two scale.  With 11-bit (FP16) significands 22 + 7 = 29 > 24."""
    K = 128
    A = workloads.scaled_slices_bf16((8, K), 41, -6)
    B = workloads.scaled_slices_bf16((K, 8), 42, -3)
    C, _ = oracle.gemm_rows(_bits(A), _bits(B), 8, 8, K)
    assert np.array_equal(C.astype(np.float32).astype(np.float64), C)
    # the FP16 counterpart is not exact in binary32 in general
    g = torch.Generator().manual_seed(9)
    a = torch.randint(1025, 2048, (1, K), generator=g).to(torch.float64)
    b = torch.randint(1025, 2048, (K, 1), generator=g).to(torch.float64)
    exact = int((a @ b).item())
    assert exact > 2 ** 24 and float(np.float32(exact)) != exact


# --------------------------------------------------------------------------
# The split-K serial reduction
# --------------------------------------------------------------------------

def test_serial_f32_reduction_golden():
    n = 0
    for line in _golden_lines("f32_serial_sums.txt"):
        lhs, rhs = line.split("->")
        terms = [float(t) for t in lhs.split()]
        want = float(rhs)
        W = np.array(terms, dtype=np.float32).reshape(len(terms), 1)
        got = oracle.splitk_reduce_f32(W)[0]
        assert got == want and np.signbit(got) == np.signbit(want), line
        n += 1
    assert n == 7


def test_serial_f32_reduction_integers_and_shape():
    g = np.random.default_rng(4)
    W = g.integers(-1000, 1000, size=(8, 3, 5)).astype(np.float32)
    out = oracle.splitk_reduce_f32(W)
    assert out.shape == (3, 5)
    assert np.array_equal(out, W.astype(np.int64).sum(axis=0).astype(np.float32))
    assert np.array_equal(oracle.splitk_reduce_f32(W[:1]), W[0])


# --------------------------------------------------------------------------
# The linear layer C = A W^T + b
# --------------------------------------------------------------------------

def test_linear_zero_input_gives_the_bias():
    M, N, K = 5, 33, 70
    A = torch.zeros(M, K, dtype=torch.bfloat16)
    W = workloads.normal_bf16((N, K), 3)
    b = workloads.normal_bf16((N,), 4)
    C, D = oracle.linear_rows(A, W, b, M, N, K)
    bd = b.to(torch.float64).numpy()
    assert np.array_equal(C, np.broadcast_to(bd, (M, N)))
    assert np.array_equal(D, np.broadcast_to(np.abs(bd), (M, N)))


def test_linear_identity_weight_adds_bias_exactly():
    M, K = 9, 48
    A = workloads.normal_bf16((M, K), 5)
    W = torch.eye(K, dtype=torch.bfloat16)            # N = K
    b = workloads.normal_bf16((K,), 6)
    C, _ = oracle.linear_rows(A, W, b, M, K, K)
    # bf16 + bf16 is exact in binary64
    assert np.array_equal(C, A.to(torch.float64).numpy() + b.to(torch.float64).numpy()[None, :])
    C0, _ = oracle.linear_rows(A, W, None, M, K, K)
    assert np.array_equal(C0, A.to(torch.float64).numpy())


@pytest.mark.parametrize("seed", [11, 12, 13])
def test_linear_brute_force_rational(seed):
    rnd = random.Random(seed)
    M, N, K = rnd.randint(1, 4), rnd.randint(1, 5), rnd.randint(1, 6)
    A = workloads.normal_bf16((M, K), 600 + seed)
    W = workloads.normal_bf16((N, K), 700 + seed)
    b = workloads.normal_bf16((N,), 800 + seed)
    C, D = oracle.linear_rows(A, W, b, M, N, K)
    a = A.to(torch.float64).numpy()
    w = W.to(torch.float64).numpy()
    bb = b.to(torch.float64).numpy()
    u = Fraction(2.0 ** -53)
    for i in range(M):
        for j in range(N):
            terms = [Fraction(float(a[i, k])) * Fraction(float(w[j, k])) for k in range(K)]
            exact = sum(terms, Fraction(0)) + Fraction(float(bb[j]))
            scale = sum((abs(t) for t in terms), Fraction(0)) + abs(Fraction(float(bb[j])))
            assert abs(Fraction(C[i, j]) - exact) <= (K + 1) * u * scale
            assert abs(Fraction(D[i, j]) - scale) <= (K + 1) * u * scale


# --------------------------------------------------------------------------
# 8-bit floats and the 8-bit linear layer
# --------------------------------------------------------------------------

@pytest.mark.parametrize("fmt,tdtype", [(oracle.FMT_E4M3, torch.float8_e4m3fn),
                                        (oracle.FMT_E5M2, torch.float8_e5m2)])
def test_fp8_decode_exhaustive_against_torch(fmt, tdtype):
    pats = np.arange(256, dtype=np.uint8)
    ours = oracle.decode8(fmt, pats)
    ref = torch.from_numpy(pats.copy()).view(tdtype).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))
    if fmt == oracle.FMT_E4M3:
        assert np.nanmax(ours) == 448.0 and nan.sum() == 2          # no infinity
    else:
        assert np.isinf(ours).sum() == 2 and np.nanmax(ours[~np.isinf(ours)]) == 57344.0


def _fp8(t: torch.Tensor, fmt):
    return t.to(torch.float8_e4m3fn if fmt == oracle.FMT_E4M3 else torch.float8_e5m2)


@pytest.mark.parametrize("fa,fb", [(oracle.FMT_E4M3, oracle.FMT_E4M3),
                                   (oracle.FMT_E5M2, oracle.FMT_E4M3)])
def test_linear8_small_integers_exact(fa, fb):
    M, N, K = 6, 9, 300
    g = torch.Generator().manual_seed(1)
    ai = torch.randint(-8, 9, (M, K), generator=g)
    wi = torch.randint(-8, 9, (N, K), generator=g)
    A, W = _fp8(ai.float(), fa), _fp8(wi.float(), fb)      # |v| <= 8 is exact in both formats
    C, D = oracle.linear8_rows(A, W, fa, fb, M, N, K)
    assert np.array_equal(C, (ai.numpy() @ wi.numpy().T).astype(np.float64))
    assert np.array_equal(D, (np.abs(ai.numpy()) @ np.abs(wi.numpy()).T).astype(np.float64))


def test_linear8_scale_bias_and_rational_brute_force():
    M, N, K = 3, 4, 5
    g = torch.Generator().manual_seed(2)
    A = _fp8(torch.randn(M, K, generator=g) * 3, oracle.FMT_E4M3)
    W = _fp8(torch.randn(N, K, generator=g), oracle.FMT_E5M2)
    b = workloads.normal_bf16((N,), 3)
    scale = 0.375
    C, D = oracle.linear8_rows(A, W, oracle.FMT_E4M3, oracle.FMT_E5M2, M, N, K, scale, b)
    a = A.to(torch.float64).numpy()
    w = W.to(torch.float64).numpy()
    bb = b.to(torch.float64).numpy()
    u = Fraction(2.0 ** -53)
    for i in range(M):
        for j in range(N):
            terms = [Fraction(float(a[i, k])) * Fraction(float(w[j, k])) for k in range(K)]
            exact = Fraction(scale) * sum(terms, Fraction(0)) + Fraction(float(bb[j]))
            scl = Fraction(scale) * sum((abs(t) for t in terms), Fraction(0)) + abs(Fraction(float(bb[j])))
            assert abs(Fraction(C[i, j]) - exact) <= (K + 2) * u * scl
