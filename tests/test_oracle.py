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


# ------------------------------------------------------------ Ozaki scheme --
# cuTile article, "倍精度行列積エミュレーション": eqs. (1)-(5) split each vector
# into bfloat16 slices, eqs. (10)-(11) multiply slice pairs, Fast Mode skips the
# pairs with p + q >= d.

def test_ozaki_pair_counts_match_the_pages_table():
    path = os.path.join(os.path.dirname(__file__), "golden", "ozaki_fast_mode_pairs.txt")
    n = 0
    for line in open(path, encoding="utf-8"):
        if line.startswith("#") or not line.strip():
            continue
        s, d, want = (int(v) for v in line.split())
        assert oracle.ozaki_pairs(s, d) == want, (s, d)
        n += 1
    assert n == 6


def test_ozaki_rho_gives_the_widest_exact_slices():
    """beta = m1 - rho is the widest bfloat16 slice for which K products of two
    slices add up exactly in binary32 in any order: K * (2^beta)^2 <= 2^24,
    and either beta = 8 (all of bfloat16) or one more bit would break it."""
    for K in list(range(1, 70)) + [127, 128, 129, 255, 256, 257, 1000, 1024, 1025, 3000, 4096,
                                   4097, 8192, 16384, 65536, 1 << 20]:
        beta = 53 - oracle.ozaki_rho(K)
        assert 1 <= beta <= 8, K
        assert K * 4 ** beta <= 1 << 24, K
        assert beta == 8 or K * 4 ** (beta + 1) > 1 << 24, K


def _exact_sum(terms):
    return sum((Fraction(t) for t in terms), Fraction(0))


@pytest.mark.parametrize("axis", [0, 1])
def test_ozaki_split_reconstructs_exactly(axis):
    """Eq. (9) plus the residual: x = sum_p 2^(c^(p)) xbar^(p) + x^(s+1),
    exactly, for vectors with values across many binades, zeros included."""
    rng = np.random.default_rng(5 + axis)
    X = rng.standard_normal((12, 40)) * np.exp2(rng.integers(-30, 30, (12, 40)))
    X[3, :] = 0.0
    X[:, 7] = 0.0
    X[5, 9] = -0.0
    rho = oracle.ozaki_rho(40)
    beta = 53 - rho
    for slices in (1, 3, 9):
        S, c1, R = oracle.ozaki_split(X, axis, rho, slices)
        rows, cols = X.shape
        for i in range(rows):
            for j in range(cols):
                v = i if axis == 0 else j
                total = _exact_sum([Fraction(S[p, i, j]) * Fraction(2) ** (int(c1[v]) - p * (beta + 1))
                                    for p in range(slices)] + [R[i, j]])
                assert total == Fraction(X[i, j]), (slices, i, j)


def test_ozaki_slices_are_narrow_bfloat16_values():
    """Each slice value is an integer multiple of 2^(rho - 53) of magnitude at
    most 1: a bfloat16 value with at most beta = 53 - rho significant bits."""
    rng = np.random.default_rng(11)
    X = rng.standard_normal((20, 300)) * np.exp2(rng.integers(-8, 8, (20, 300)))
    for K in (300, 5000):
        rho = oracle.ozaki_rho(K)
        beta = 53 - rho
        S, c1, R = oracle.ozaki_split(X, 0, rho, 6)
        n = S * 2.0 ** (53 - rho)
        assert np.array_equal(n, np.round(n))
        assert np.abs(n).max() <= 2 ** beta
        assert np.abs(S).max() <= 1.0
        # exactly representable in bfloat16: the oracle's own codec round trip
        assert np.array_equal(oracle.decode(oracle.FMT_BF16, oracle.encode_rne(oracle.FMT_BF16, S)), S)


def test_ozaki_first_slice_is_x_rounded_to_its_grid():
    """Eq. (3) on the first slice is round-to-nearest-even of x to a multiple of
    2^(c^(1) + rho - 53), the unit of sigma's last place (the Veltkamp split):
    compared with numpy's half-to-even rounding."""
    rng = np.random.default_rng(2)
    X = rng.standard_normal((9, 64))
    X[0, :4] = [0.5, -0.75, 1.0, 0.0]
    # maxima that are exact powers of two: ceil(log2 m) = log2 m
    X[6] = rng.uniform(-1.0, 1.0, 64)
    X[6, 5] = 1.0
    X[7] = rng.uniform(-0.25, 0.25, 64) * 2.0 ** -30
    X[7, 9] = -(2.0 ** -30)
    X[8] = rng.uniform(-1.0, 1.0, 64) * 2.0 ** 40
    X[8, 0] = 2.0 ** 40
    rho = oracle.ozaki_rho(64)
    S, c1, R = oracle.ozaki_split(X, 0, rho, 1)
    assert list(c1[6:]) == [0, -30, 40]
    for i in range(9):
        u = 2.0 ** (int(c1[i]) + rho - 53)
        v = np.round(X[i] / u) * u
        assert np.array_equal(S[0, i] * 2.0 ** int(c1[i]), v)
        m = np.abs(X[i]).max()
        assert 2.0 ** (int(c1[i]) - 1) < m <= 2.0 ** int(c1[i])     # eq. (1)


def test_ozaki_zero_vectors_split_to_zero():
    X = np.zeros((3, 5))
    S, c1, R = oracle.ozaki_split(X, 1, 45, 4)
    assert not S.any() and not c1.any() and not R.any()


@pytest.mark.parametrize("M,N,K", [(9, 7, 31), (16, 40, 300)])
def test_ozaki_gemm_small_integers_exact(M, N, K):
    """Integer inputs up to 1000 in magnitude: every bit lands in a slice, every
    slice-pair sum and every binary64 partial sum is an exact integer, so C is
    the exact product."""
    rng = np.random.default_rng(M + K)
    A = rng.integers(-1000, 1001, (M, K)).astype(np.float64)
    B = rng.integers(-1000, 1001, (K, N)).astype(np.float64)
    C, inexact = oracle.ozaki_gemm(A, B)
    assert inexact == 0
    assert np.array_equal(C, (A.astype(np.int64) @ B.astype(np.int64)).astype(np.float64))


def test_ozaki_single_pair_is_the_product_of_leading_slices():
    """d = 1 keeps the pair (0, 0) alone: C = 2^(c_a + c_b) * (xbar_a^(1) . ybar_b^(1)),
    eq. (10) with one term, computed here from the oracle's slices with numpy."""
    rng = np.random.default_rng(4)
    A = rng.standard_normal((10, 64))
    B = rng.standard_normal((64, 12))
    rho = oracle.ozaki_rho(64)
    C, inexact = oracle.ozaki_gemm(A, B, rho=rho, slices=5, d=1)
    Sa, ca, _ = oracle.ozaki_split(A, 0, rho, 5)
    Sb, cb, _ = oracle.ozaki_split(B, 1, rho, 5)
    P = Sa[0] @ Sb[0]                       # integer multiples of one unit, < 2^24 of them: exact
    want = P * np.exp2(ca[:, None] + cb[None, :])
    assert inexact == 0 and np.array_equal(C, want)


def test_ozaki_gemm_accuracy_against_exact_products():
    """Random normal and wide-range inputs, against exact rational products.
    With the default slices and d the error is binary64's: at most 8 units of
    2^-53 of sum_k |a_ik b_kj| (the outer additions) plus what the slices
    leave out, K * 2^(c_a + c_b) * 2^-(s (beta + 1) - 3) -- each vector keeps
    s (beta + 1) - 1 >= 53 bits below its own maximum 2^c (eq. (1) scales by
    the vector's maximum, not the element's).  Fast Mode with a smaller d is
    never more accurate."""
    rng = np.random.default_rng(9)
    M, N, K = 8, 9, 200
    for A, B in (
        (rng.standard_normal((M, K)), rng.standard_normal((K, N))),
        (rng.standard_normal((M, K)) * np.exp2(rng.integers(-20, 20, (M, K))),
         rng.standard_normal((K, N)) * np.exp2(rng.integers(-20, 20, (K, N)))),
    ):
        exact = [[sum((Fraction(A[i, k]) * Fraction(B[k, j]) for k in range(K)), Fraction(0))
                  for j in range(N)] for i in range(M)]
        scale = np.abs(A) @ np.abs(B)
        errs = {}
        rho = oracle.ozaki_rho(K)
        beta = 53 - rho
        s = oracle.ozaki_default_slices(rho)
        _, ca, _ = oracle.ozaki_split(A, 0, rho, 1)
        _, cb, _ = oracle.ozaki_split(B, 1, rho, 1)
        left_out = K * np.exp2(ca[:, None] + cb[None, :] - (s * (beta + 1) - 3))
        bound = 8 * 2.0 ** -53 * scale + left_out
        for d in (s, s - 2, 3):
            C, inexact = oracle.ozaki_gemm(A, B, rho=rho, slices=s, d=d)
            assert inexact == 0
            err = np.array([[abs(float(Fraction(C[i, j]) - exact[i][j])) for j in range(N)]
                            for i in range(M)])
            if d == s:
                assert (err <= bound).all(), (err / bound).max()
            errs[d] = (err / scale).max()
        assert errs[s] <= errs[s - 2] <= errs[3], errs


def test_ozaki_inexact_count_flags_too_wide_slices():
    """With rho below the value K needs (full 8-bit slices at K = 4096), the
    slice-pair sums can exceed 2^24 units, and the oracle counts them; with
    rho(K) it counts none."""
    rng = np.random.default_rng(3)
    A = rng.uniform(0.5, 1.0, (4, 4096))
    B = rng.uniform(0.5, 1.0, (4096, 4))
    _, bad_wide = oracle.ozaki_gemm(A, B, rho=45, slices=7, d=7)
    _, bad_rho = oracle.ozaki_gemm(A, B)
    assert bad_wide > 0 and bad_rho == 0


# --- Fast Mode's automatic d (cuTile article, "Fast Mode（GEMMの削減）") ---

def _mass(x):
    """sum_k floor(|x_k| 2^(40 - c)), c = ceil(log2 max |x|), in exact rationals."""
    m = max(abs(Fraction(v)) for v in x)
    if m == 0:
        return 0
    c = 0
    while Fraction(2) ** c < m:
        c += 1
    while Fraction(2) ** (c - 1) >= m:
        c -= 1
    return sum(int(abs(Fraction(v)) * Fraction(2) ** (40 - c)) for v in x)


def _fast_d_brute(tx, ty, slices, beta, k):
    """The least d in 1 .. slices whose skipped pairs meet the bound:
    T_x T_y >= 2^(133 + ceil(log2 slices) + ceil(log2 k) - d (beta + 1)),
    compared as exact integers (Python), else slices."""
    ls = (slices - 1).bit_length()
    kap = (k - 1).bit_length()
    for d in range(1, slices + 1):
        e = 133 + ls + kap - d * (beta + 1)
        if (tx * ty) * (2 ** max(-e, 0)) >= 2 ** max(e, 0):
            return d
    return slices


def test_ozaki_fast_mode_masses_and_d_against_exact_integers():
    """The vectors' masses against exact rational floors (subnormals, zeros,
    powers of two and wide exponent ranges included), and every element's d
    against a brute-force search of the inequality in exact integers."""
    rng = np.random.default_rng(21)
    M, N, K = 6, 5, 300
    A = rng.standard_normal((M, K)) * np.exp2(rng.integers(-30, 30, (M, K)))
    B = rng.standard_normal((K, N))
    A[0, :] = 0.0                                  # a zero row: mass 0
    A[1, :] = 0.0
    A[1, 7] = 2.0 ** -1070                         # a subnormal alone
    A[2, 3] = 2.0 ** 40                            # a power-of-two maximum
    B[:, 0] = 1.0                                  # equal values
    B[5, 1] = 0.0
    rho = oracle.ozaki_rho(K)
    s = oracle.ozaki_default_slices(rho)
    D, Ta, Tb = oracle.ozaki_fast_d(A, B, rho=rho, slices=s)
    for i in range(M):
        assert int(Ta[i]) == _mass(A[i]), i
    for j in range(N):
        assert int(Tb[j]) == _mass(B[:, j]), j
    assert Ta[0] == 0 and Ta[1] == 2 ** 40         # one element at the maximum: 2^40
    assert int(Tb[0]) == K * 2 ** 40               # all equal to the maximum (a power of two)
    for i in range(M):
        for j in range(N):
            assert D[i, j] == _fast_d_brute(int(Ta[i]), int(Tb[j]), s, 53 - rho, K), (i, j)
    assert (D[0] == s).all()                       # nothing known about a zero row: every pair


def test_ozaki_fast_mode_meets_the_pages_bound_and_skips_pairs():
    """On normal data the automatic d skips pairs the default keeps (about a
    quarter at K = 4096), and every element stays within the page's bound
    2 sqrt(k) u |A||B| against exact rational products."""
    rng = np.random.default_rng(22)
    M, N, K = 6, 7, 4096
    A = rng.standard_normal((M, K))
    B = rng.standard_normal((K, N))
    rho = oracle.ozaki_rho(K)
    s = oracle.ozaki_default_slices(rho)
    D, _, _ = oracle.ozaki_fast_d(A, B, rho=rho, slices=s)
    assert D.max() <= s and D.min() >= 1
    assert (D < s).mean() > 0.5                    # most elements drop the last diagonal
    C, inexact = oracle.ozaki_gemm(A, B, rho=rho, slices=s, d=-1)
    assert inexact == 0
    scale = np.abs(A) @ np.abs(B)
    for i in range(M):
        for j in range(N):
            exact = sum((Fraction(A[i, k]) * Fraction(B[k, j]) for k in range(K)), Fraction(0))
            err = abs(float(Fraction(C[i, j]) - exact))
            assert err <= 2 * np.sqrt(K) * 2.0 ** -53 * scale[i, j], (i, j)


def test_ozaki_fast_mode_is_the_fixed_d_product_where_d_is_uniform():
    """Where every element's automatic d is the same d, the product is the
    fixed-d product, bit for bit; rows computed alone take the same d and give
    the same bits (d depends on the row and the column only)."""
    rng = np.random.default_rng(23)
    A = rng.standard_normal((5, 4096))
    B = rng.standard_normal((4096, 9))
    rho = oracle.ozaki_rho(4096)
    s = oracle.ozaki_default_slices(rho)
    D, _, _ = oracle.ozaki_fast_d(A, B, rho=rho, slices=s)
    C, _ = oracle.ozaki_gemm(A, B, rho=rho, slices=s, d=-1)
    for d in np.unique(D):
        Cd, _ = oracle.ozaki_gemm(A, B, rho=rho, slices=s, d=int(d))
        assert np.array_equal(C[D == d], Cd[D == d])
    for i in range(5):
        Di, _, _ = oracle.ozaki_fast_d(A[i:i + 1], B, rho=rho, slices=s)
        Ci, _ = oracle.ozaki_gemm(A[i:i + 1], B, rho=rho, slices=s, d=-1)
        assert np.array_equal(Di[0], D[i]) and np.array_equal(Ci[0], C[i])
