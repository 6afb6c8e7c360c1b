/*
 * oracle.c -- plain, slow, obviously correct CPU reference for the
 * deterministic batch-invariant BF16 GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library
 * and its Python binding) may include, link, load or call this file; only the
 * tests, the package's smoke() check and the benchmark's CPU-baseline leg do.
 * It shares no code, header, table or constant with the GPU path.
 *
 * What it computes, and the passage each function follows:
 *
 *   oracle_gemm_rows      C_ij = sum_{k=0}^{K-1} A_ik * B_kj, the plain
 *                         definition of the matrix product (Tencent AI-infra
 *                         article "腾讯エンジニア：大規模モデルの出力を確定させる
 *                         ための AI インフラ手法", section "Batch Invariance の由来",
 *                         and the i/j/k triple loop in "GEMM の最適化戦略"),
 *                         evaluated in binary64 with k ascending.  Every
 *                         bf16 x bf16 product is exact in binary64 (8 + 8 <= 53
 *                         significand bits), so only the additions round.
 *                         It also returns D_ij = sum_k |A_ik * B_kj|, the scale
 *                         the error criterion |C - C_ref| <= 1e-5 * D uses.
 *   oracle_decode         value of an IEEE-754 binary16 / bfloat16 bit pattern,
 *                         or of the 8-bit floats E5M2 / E4M3 (the FP8 formats
 *                         of the cuTile article's FP8 benchmark), written from
 *                         the field definitions (sign, biased exponent,
 *                         fraction; subnormals; inf/nan).
 *   oracle_linear8_rows   C_ij = sum_k A_ik W_jk for 8-bit float operands, W in
 *                         the weight layout [N][K], binary64, k ascending.
 *   oracle_encode_rne     round a binary64 value to the nearest binary16 /
 *                         bfloat16, ties to even (the rounding rule the same
 *                         article's "背景" section applies to 2048 + 1 in FP16).
 *   oracle_ulp            ULP(x) = 2^(E - M): E the unbiased exponent of x,
 *                         M the number of stored fraction bits ("背景").
 *   oracle_splitk_reduce_f32
 *                         the split-K workspace reduction of the same article's
 *                         "Split-K" section: out = w_0, then out = out + w_s for
 *                         s = 1 .. S-1, every addition rounded to binary32
 *                         (round to nearest even), in that serial order.
 *   oracle_ozaki_rho, oracle_ozaki_split, oracle_ozaki_pairs,
 *   oracle_ozaki_gemm     the Ozaki scheme of the cuTile article (section
 *                         "倍精度行列積エミュレーション"): a binary64 matrix product
 *                         from bfloat16 slices -- the Veltkamp split, eqs.
 *                         (1)-(5); slice-pair products, eqs. (10)-(11); the
 *                         binary64 outer accumulation; Fast Mode's skip of the
 *                         pairs with p + q >= d, a fixed d or its automatic
 *                         choice per output element (oracle_ozaki_fast_d).
 *
 * Build: a C99 compiler with -O2 -ffp-contract=off (no fused multiply-add, no
 * fast-math); OpenMP is optional and only splits the rows between threads --
 * each output element is still one thread's serial loop.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* IEEE-754 small formats.  A format is (exponent bits, fraction bits):       */
/*   binary16 (FP16): 5, 10     bfloat16 (BF16): 8, 7                         */
/* ------------------------------------------------------------------------ */

#define ORACLE_FMT_FP16 0
#define ORACLE_FMT_BF16 1
#define ORACLE_FMT_E5M2 2   /* 8-bit float, IEEE-style: 5 exponent, 2 fraction bits */
#define ORACLE_FMT_E4M3 3   /* 8-bit float, 4 exponent, 3 fraction bits, no infinity:
                               the all-ones exponent is an ordinary binade except
                               fraction 111, the only NaN (the "FN" variant) */

static void fmt_fields(int fmt, int *ebits, int *fbits) {
    if (fmt == ORACLE_FMT_FP16)      { *ebits = 5; *fbits = 10; }
    else if (fmt == ORACLE_FMT_E5M2) { *ebits = 5; *fbits = 2; }
    else if (fmt == ORACLE_FMT_E4M3) { *ebits = 4; *fbits = 3; }
    else                             { *ebits = 8; *fbits = 7; }
}

/* Decode one bit pattern of the given format to its exact binary64 value. */
double oracle_decode(int fmt, uint32_t bits) {
    int ebits, fbits;
    fmt_fields(fmt, &ebits, &fbits);
    const uint32_t nbits = 1u + (uint32_t)ebits + (uint32_t)fbits;
    bits &= (nbits == 32u) ? 0xFFFFFFFFu : ((1u << nbits) - 1u);
    const uint32_t sign = (bits >> (ebits + fbits)) & 1u;
    const uint32_t e = (bits >> fbits) & ((1u << ebits) - 1u);
    const uint32_t f = bits & ((1u << fbits) - 1u);
    const int bias = (1 << (ebits - 1)) - 1;
    const uint32_t emax_field = (1u << ebits) - 1u;
    double mag;
    if (fmt == ORACLE_FMT_E4M3 && e == emax_field) {
        /* no infinity: 1.f * 2^(15 - 7), except the single NaN pattern */
        mag = (f == 7u) ? NAN : ldexp((double)((1u << fbits) | f), (int)e - bias - fbits);
    } else if (e == emax_field) {
        mag = (f == 0) ? INFINITY : NAN;
    } else if (e == 0) {
        /* subnormal: 0.f * 2^(1 - bias) */
        mag = ldexp((double)f, 1 - bias - fbits);
    } else {
        /* normal: 1.f * 2^(e - bias) */
        mag = ldexp((double)((1u << fbits) | f), (int)e - bias - fbits);
    }
    return sign ? -mag : mag;
}

/* Round a binary64 value to the nearest representable value of the format,
 * ties to even; overflow goes to infinity; NaN to the canonical quiet NaN. */
uint32_t oracle_encode_rne(int fmt, double x) {
    int ebits, fbits;
    fmt_fields(fmt, &ebits, &fbits);
    const int bias = (1 << (ebits - 1)) - 1;
    const int emin = 1 - bias;          /* smallest normal exponent */
    const int emax = bias;              /* largest finite exponent */
    const uint32_t sign_bit = 1u << (ebits + fbits);
    const uint32_t exp_all = ((1u << ebits) - 1u) << fbits;
    if (isnan(x)) return exp_all | (1u << (fbits - 1));
    const uint32_t sign = signbit(x) ? sign_bit : 0u;
    double a = fabs(x);
    if (a == 0.0) return sign;
    if (isinf(a)) return sign | exp_all;
    /* a = fr * 2^ex with fr in [0.5, 1): the unbiased exponent is ex - 1 */
    int ex;
    (void)frexp(a, &ex);
    int E = ex - 1;
    if (E < emin) E = emin;             /* subnormal range shares emin's quantum */
    /* quantum (one unit in the last place) of the binade [2^E, 2^(E+1)) */
    const int qexp = E - fbits;
    const double n = ldexp(a, -qexp);   /* exact: scaling by a power of two */
    double r = floor(n);
    const double rem = n - r;           /* exact: n and r share the binade */
    if (rem > 0.5 || (rem == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
    /* r is an integer in [0, 2^(fbits+1)]; rounding up may carry into the
     * next binade, which the re-normalisation below absorbs. */
    if (r == 0.0) return sign;
    double v = ldexp(r, qexp);
    if (v >= ldexp(2.0 - ldexp(1.0, -fbits - 1), emax)) {
        /* at or beyond the halfway point past the largest finite value */
        return sign | exp_all;
    }
    (void)frexp(v, &ex);
    int Ev = ex - 1;
    if (Ev < emin) {
        /* subnormal: fraction = v / 2^(emin - fbits), exponent field 0 */
        const uint32_t f = (uint32_t)ldexp(v, -(emin - fbits));
        return sign | f;
    }
    const uint32_t f = (uint32_t)(ldexp(v, -(Ev - fbits)) - ldexp(1.0, fbits));
    return sign | ((uint32_t)(Ev + bias) << fbits) | f;
}

/* ULP(x) = 2^(E - M): E the unbiased exponent of |x| (clamped to the smallest
 * normal exponent for subnormals), M the stored fraction bits of the format. */
double oracle_ulp(int fmt, double x) {
    int ebits, fbits;
    fmt_fields(fmt, &ebits, &fbits);
    const int emin = 2 - (1 << (ebits - 1));
    double a = fabs(x);
    int E = emin;
    if (a != 0.0) {
        int ex;
        (void)frexp(a, &ex);
        E = ex - 1;
        if (E < emin) E = emin;
    }
    return ldexp(1.0, E - fbits);
}

/* ------------------------------------------------------------------------ */
/* The matrix product.                                                        */
/* ------------------------------------------------------------------------ */

static double g_bf16_value[65536];
static int g_bf16_ready = 0;

static void bf16_table_init(void) {
    if (g_bf16_ready) return;
    for (uint32_t h = 0; h < 65536u; ++h) g_bf16_value[h] = oracle_decode(ORACLE_FMT_BF16, h);
    g_bf16_ready = 1;
}

/*
 * A: bf16 bit patterns, row-major [M][lda] (row i, column k at A[i*lda + k]).
 * B: bf16 bit patterns, row-major [K][ldb] (row k, column j at B[k*ldb + j]).
 * rows: the nrows row indices of A to evaluate (NULL: rows 0 .. nrows-1).
 * C, D: binary64 outputs, [nrows][N] dense (row r of C holds row rows[r]).
 *
 * For every (i, j) the K terms are added to a binary64 accumulator that starts
 * at +0.0, in ascending k.  The loop nest walks k outside j so that B is read
 * row by row; that changes nothing about any single element's sum, whose
 * terms still arrive in ascending k into its own accumulator.
 *
 * Returns 0, or -1 on a bad argument.
 */
int oracle_gemm_rows(const uint16_t *A, const uint16_t *B,
                     int64_t M, int64_t N, int64_t K,
                     int64_t lda, int64_t ldb,
                     const int64_t *rows, int64_t nrows,
                     double *C, double *D) {
    if (M < 0 || N < 0 || K < 0 || nrows < 0) return -1;
    if (nrows > 0 && N > 0 && (C == NULL || D == NULL)) return -1;
    if (K > 0 && (lda < K || ldb < N)) return -1;
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t i = rows ? rows[r] : r;
        if (i < 0 || i >= M) return -1;
    }
    bf16_table_init();
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t i = rows ? rows[r] : r;
        double *c = C + r * N;
        double *d = D + r * N;
        for (int64_t j = 0; j < N; ++j) { c[j] = 0.0; d[j] = 0.0; }
        for (int64_t k = 0; k < K; ++k) {
            const double a = g_bf16_value[A[i * lda + k]];
            const uint16_t *brow = B + k * ldb;
            for (int64_t j = 0; j < N; ++j) {
                const double p = a * g_bf16_value[brow[j]];   /* exact */
                c[j] = c[j] + p;
                d[j] = d[j] + fabs(p);
            }
        }
    }
    return 0;
}

/* Serial split-K reduction in binary32: W is [S][count] dense; out[e] =
 * (((W[0][e] + W[1][e]) + W[2][e]) + ...), each '+' one binary32 addition. */
int oracle_splitk_reduce_f32(const float *W, int64_t S, int64_t count, float *out) {
    if (S < 1 || count < 0) return -1;
    for (int64_t e = 0; e < count; ++e) {
        float acc = W[e];
        for (int64_t s = 1; s < S; ++s) acc = acc + W[s * count + e];
        out[e] = acc;
    }
    return 0;
}

/*
 * A linear layer with 8-bit float operands: C_ij = sum_{k} A_ik * W_jk, in
 * binary64 with k ascending (each 8-bit x 8-bit product is exact), and the
 * scale D_ij = sum_k |A_ik * W_jk|.  A: [M][lda] bytes of format fmt_a, W:
 * [N][ldw] bytes (the weight layout, row j = output column j) of format fmt_b.
 * rows / nrows / C / D as in oracle_gemm_rows.  Returns 0 or -1.
 */
int oracle_linear8_rows(const uint8_t *A, const uint8_t *W, int fmt_a, int fmt_b,
                        int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldw,
                        const int64_t *rows, int64_t nrows, double *C, double *D) {
    if (M < 0 || N < 0 || K < 0 || nrows < 0) return -1;
    if (nrows > 0 && N > 0 && (C == NULL || D == NULL)) return -1;
    if (K > 0 && (lda < K || ldw < K)) return -1;
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t i = rows ? rows[r] : r;
        if (i < 0 || i >= M) return -1;
    }
    double va[256], vb[256];
    for (uint32_t h = 0; h < 256u; ++h) {
        va[h] = oracle_decode(fmt_a, h);
        vb[h] = oracle_decode(fmt_b, h);
    }
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t i = rows ? rows[r] : r;
        const uint8_t *arow = A + i * lda;
        for (int64_t j = 0; j < N; ++j) {
            const uint8_t *wrow = W + j * ldw;
            double c = 0.0, d = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const double p = va[arow[k]] * vb[wrow[k]];   /* exact */
                c = c + p;
                d = d + fabs(p);
            }
            C[r * N + j] = c;
            D[r * N + j] = d;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Ozaki scheme (cuTile article, "倍精度行列積エミュレーション": "Ozaki Scheme   */
/* について", "分解(Split)", "行列積の計算", "Fast Mode（GEMMの削減）",            */
/* "Fused Split Kernel（分割の融合）").                                        */
/*                                                                          */
/* Type1 = binary64 (m1 = 53 significand bits), Type2 = bfloat16 (m2 = 8),  */
/* Type3 = binary32 (m3 = 24), all counting the hidden bit.                 */
/* ------------------------------------------------------------------------ */

#define OZ_M1 53
#define OZ_M2 8
#define OZ_M3 24

/* The precision parameter rho = max(gamma, xi) of "分解(Split)":
 * gamma = ceil(m1 - (m3 - log2 k) / 2) and xi = m1 - m2, k the inner-product
 * length.  gamma = ceil(41 + log2(k) / 2) = 41 + t, t the least integer with
 * 4^t >= k -- evaluated in integers, with no logarithm to round.
 * Returns -1 for k < 1. */
int oracle_ozaki_rho(int64_t k) {
    if (k < 1) return -1;
    int t = 0;
    int64_t p = 1;
    while (p < k) {
        p *= 4;
        ++t;
    }
    const int gamma = (OZ_M1 - OZ_M3 / 2) + t;
    const int xi = OZ_M1 - OZ_M2;
    return gamma > xi ? gamma : xi;
}

/* Number of slice pairs (p, q), 0 <= p, q < slices, that Fast Mode keeps:
 * those with p + q < d. */
int64_t oracle_ozaki_pairs(int slices, int d) {
    int64_t n = 0;
    for (int p = 0; p < slices; ++p)
        for (int q = 0; q < slices; ++q)
            if (p + q < d) ++n;
    return n;
}

/* c = ceil(log2 m) for m > 0, exactly: m = f * 2^e with f in [0.5, 1). */
static int oz_ceil_log2(double m) {
    int e = 0;
    const double f = frexp(m, &e);
    return f == 0.5 ? e - 1 : e;
}

/*
 * The split of one vector x (n values at stride inc) into `slices` bfloat16
 * slices, eqs. (1)-(5):
 *   c^(1)   = ceil(log2 max_i |x_i|)                                     (1)
 *   sigma   = 0.75 * 2^(rho + c^(p))                                     (2)
 *   v_i     = fl((x_i^(p) + sigma) - sigma)                              (3)
 *   x^(p+1) = fl(x^(p) - v)                                              (4)
 *   xbar^(p)= cvt_bf16(fl(2^(-c^(p)) * v))                               (5)
 * The fused split computes every slice's exponent from the first maximum;
 * the one it uses here is the bound eq. (3) gives on the residual:
 * |x^(p+1)| <= ulp(sigma) / 2 = 2^(c^(p) - (m1 - rho) - 1), so
 *   c^(p+1) = c^(p) - (m1 - rho) - 1.
 * Every v is then a multiple of 2^(rho + c^(p) - m1) no larger than
 * 2^(c^(p)), so xbar^(p) has at most m1 - rho <= m2 significant bits and the
 * conversion to bfloat16 is exact; it is checked here (a failed check
 * returns -1).  out[p * p_stride + i * out_inc] = value of xbar^(p)_i,
 * *c1 = c^(1) (0 for an all-zero vector, whose slices are all zero), and
 * res[i * out_inc] = x^(slices+1)_i when res is not NULL.
 */
static int oz_split_vector(const double *x, int64_t n, int64_t inc, int rho, int slices,
                           double *out, int64_t p_stride, int64_t out_inc, int *c1, double *res) {
    double m = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        const double a = fabs(x[i * inc]);
        if (a > m) m = a;
    }
    if (m == 0.0) {
        *c1 = 0;
        for (int p = 0; p < slices; ++p)
            for (int64_t i = 0; i < n; ++i) out[p * p_stride + i * out_inc] = 0.0;
        if (res)
            for (int64_t i = 0; i < n; ++i) res[i * out_inc] = 0.0;
        return 0;
    }
    const int beta = OZ_M1 - rho;
    *c1 = oz_ceil_log2(m);
    for (int64_t i = 0; i < n; ++i) {
        double r = x[i * inc];                         /* x^(1) */
        int c = *c1;
        for (int p = 0; p < slices; ++p) {
            const double sigma = ldexp(0.75, rho + c);  /* (2) */
            const double t = r + sigma;
            const double v = t - sigma;                 /* (3) */
            r = r - v;                                  /* (4) */
            const double xb = ldexp(v, -c);             /* (5), before the conversion */
            if (g_bf16_value[oracle_encode_rne(ORACLE_FMT_BF16, xb)] != xb) return -1;
            out[p * p_stride + i * out_inc] = xb;
            c = c - beta - 1;
        }
        if (res) res[i * out_inc] = r;
    }
    return 0;
}

/*
 * Split every row (axis 0, the vectors of A in A B) or every column (axis 1,
 * the vectors of B) of X [rows][cols] (leading dimension ld) into `slices`
 * bfloat16 slices.  S: [slices][rows][cols] dense, the slice values; c1: one
 * c^(1) per vector (rows entries for axis 0, cols for axis 1); R: the final
 * residual [rows][cols] dense, or NULL.  Returns 0, or -1 on a bad argument
 * or an inexact conversion.
 */
int oracle_ozaki_split(const double *X, int64_t rows, int64_t cols, int64_t ld, int axis,
                       int rho, int slices, double *S, int *c1, double *R) {
    if (rows < 0 || cols < 0 || ld < cols || slices < 1 || rho < OZ_M1 - OZ_M2 || rho >= OZ_M1)
        return -1;
    if (axis != 0 && axis != 1) return -1;
    bf16_table_init();
    const int64_t plane = rows * cols;
    int bad = 0;
    if (axis == 0) {
        for (int64_t i = 0; i < rows; ++i)
            if (oz_split_vector(X + i * ld, cols, 1, rho, slices, S + i * cols, plane, 1, c1 + i,
                                R ? R + i * cols : NULL))
                bad = 1;
    } else {
        for (int64_t j = 0; j < cols; ++j)
            if (oz_split_vector(X + j, rows, ld, rho, slices, S + j, plane, cols, c1 + j,
                                R ? R + j : NULL))
                bad = 1;
    }
    return bad ? -1 : 0;
}

/*
 * Fast Mode's choice of d (cuTile article, "Fast Mode（GEMMの削減）": the
 * smallest d for which the pairs with p + q >= d may be skipped while
 * |fl(AB) - AB| <= 2 sqrt(k) u |A||B|, u = 2^-53).  The page states the bound
 * and not the procedure; the reading here is made per output element, from
 * its row of A and its column of B only, so that a row's bits stay
 * independent of the rest of the batch:
 *
 *   - The skipped pairs of element (i, j) add sum_{p+q>=d} 2^(c_x^(p) +
 *     c_y^(q)) xbar^(p) . ybar^(q).  Every slice entry is at most 1 and
 *     c^(p) = c^(1) - p (beta + 1), so with w = beta + 1, at most `slices`
 *     pairs per diagonal p + q = t and the page's probabilistic sqrt(k) for a
 *     k-term dot product, they amount to at most
 *       sqrt(k) 2^(c_x + c_y) sum_{t>=d} slices 2^(-t w)
 *         <= sqrt(k) 2^(c_x + c_y + 1 + L_s - d w),   L_s = ceil(log2 slices).
 *   - |A||B|_ij = sum_k |x_k| |y_k| is estimated by its mean-field value
 *     mu_x mu_y / k (mu the 1-norm of the vector), from below: mu_x >=
 *     T_x 2^(c_x - 40) with the integer mass T_x = sum_k floor(|x_k| 2^(40 -
 *     c_x)) (exact and order-free; < 2^62 for k <= 2^22), and k <= 2^kappa,
 *     kappa = ceil(log2 k).
 *   - So the skip is within the bound when 2^(1 + L_s - d w) <= 2^(-52) T_x
 *     T_y 2^(-80 - kappa), i.e. when T_x T_y >= 2^(133 + L_s + kappa - d w),
 *     which holds exactly when d w >= 134 + L_s + kappa - bitlen(T_x T_y)
 *     (bitlen of the 128-bit product).
 *   - d_ij = the least such d, at least 1 and at most `slices` (the
 *     deterministic default d: Fast Mode only ever removes pairs).
 * Element (i, j) then takes pair (p, q) iff p + q < d_ij, in the usual
 * order; every element takes pair (0, 0).
 */
static uint64_t oz_mass(const double *x, int64_t n, int64_t inc, int c) {
    uint64_t t = 0;
    for (int64_t i = 0; i < n; ++i) {
        const double a = fabs(x[i * inc]);
        if (a != 0.0) t += (uint64_t)floor(ldexp(a, 40 - c));  /* exact: a power-of-two scale */
    }
    return t;
}

static int oz_ceil_log2_int(int64_t v) {
    int l = 0;
    while (((int64_t)1 << l) < v) ++l;
    return l;
}

/* 134 + ceil(log2 slices) + ceil(log2 k) - bitlen(tx * ty): d_ij = the least
 * d >= 1 with d (beta + 1) >= this, capped at slices. */
static int oz_fast_need(uint64_t tx, uint64_t ty, int slices, int64_t k) {
    unsigned __int128 prod = (unsigned __int128)tx * ty;
    int bl = 0;
    while (prod != 0) {
        ++bl;
        prod >>= 1;
    }
    return 134 + oz_ceil_log2_int(slices) + oz_ceil_log2_int(k) - bl;
}

static int oz_fast_d(uint64_t tx, uint64_t ty, int slices, int beta, int64_t k) {
    const int need = oz_fast_need(tx, ty, slices, k), w = beta + 1;
    int d = need <= w ? 1 : (need + w - 1) / w;
    return d > slices ? slices : d;
}

/* The per-element d of Fast Mode for A B (see above): D [M][N] int32, and the
 * masses T of the rows of A and columns of B.  Returns 0 or -1. */
int oracle_ozaki_fast_d(const double *A, const double *B, int64_t M, int64_t N, int64_t K, int64_t lda,
                        int64_t ldb, int rho, int slices, int *D, uint64_t *Ta, uint64_t *Tb) {
    if (M < 0 || N < 0 || K < 1 || slices < 1 || lda < K || ldb < N) return -1;
    if (rho < OZ_M1 - OZ_M2 || rho >= OZ_M1) return -1;
    const int beta = OZ_M1 - rho;
    for (int64_t i = 0; i < M; ++i) {
        double m = 0.0;
        for (int64_t k = 0; k < K; ++k) if (fabs(A[i * lda + k]) > m) m = fabs(A[i * lda + k]);
        Ta[i] = m == 0.0 ? 0 : oz_mass(A + i * lda, K, 1, oz_ceil_log2(m));
    }
    for (int64_t j = 0; j < N; ++j) {
        double m = 0.0;
        for (int64_t k = 0; k < K; ++k) if (fabs(B[k * ldb + j]) > m) m = fabs(B[k * ldb + j]);
        Tb[j] = m == 0.0 ? 0 : oz_mass(B + j, K, ldb, oz_ceil_log2(m));
    }
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) D[i * N + j] = oz_fast_d(Ta[i], Tb[j], slices, beta, K);
    return 0;
}

/*
 * C = A B in the Ozaki scheme.  A: [M][lda], B: [K][ldb] binary64; C: [M][ldc].
 * A is split by rows and B by columns (each row of A and column of B is one
 * vector x, y of eq. (10)); then, for p = 0 .. slices-1 and, inside, q = 0 ..
 * slices-1, skipping the pairs with p + q >= d (Fast Mode):
 *   P = xbar^(p)T ybar^(q) = sum_k a_p[i][k] b_q[k][j]        (11), in binary64
 *   C[i][j] = C[i][j] + 2^(c_a^(p)[i] + c_b^(q)[j]) * P        (10), binary64
 * with C starting at +0.0.  P is exact: every term is a multiple of
 * 2^(2 (rho - m1)); *inexact (when not NULL) counts the (pair, i, j) whose
 * sum of |terms| exceeds 2^m3 such units, where a binary32 accumulation in
 * some order could round -- rho is chosen so that this count is 0
 * ("行列積の計算": no rounding error in the Type3 accumulation).  The scaling
 * by a power of two is exact (inputs within the normal range), so each pair
 * costs one binary64 rounding, in the addition.  d = -1: Fast Mode's
 * automatic choice, element by element (oracle_ozaki_fast_d): element (i, j)
 * takes the pairs with p + q < d_ij, in the same order.  Returns 0 or -1.
 */
int oracle_ozaki_gemm(const double *A, const double *B, int64_t M, int64_t N, int64_t K,
                      int64_t lda, int64_t ldb, int rho, int slices, int d, double *C, int64_t ldc,
                      int64_t *inexact) {
    if (M < 0 || N < 0 || K < 0 || slices < 1 || d < -1) return -1;
    if ((K > 0 && (lda < K || ldb < N)) || ldc < N) return -1;
    if (rho < OZ_M1 - OZ_M2 || rho >= OZ_M1) return -1;
    const int beta = OZ_M1 - rho;
    double *Sa = (double *)malloc(sizeof(double) * (size_t)(slices * M * (K > 0 ? K : 1)));
    double *Sb = (double *)malloc(sizeof(double) * (size_t)(slices * (K > 0 ? K : 1) * N));
    int *ca = (int *)malloc(sizeof(int) * (size_t)(M > 0 ? M : 1));
    int *cb = (int *)malloc(sizeof(int) * (size_t)(N > 0 ? N : 1));
    const int fast = (d == -1);
    int *Dij = fast ? (int *)malloc(sizeof(int) * (size_t)(M > 0 && N > 0 ? M * N : 1)) : NULL;
    uint64_t *Ta = fast ? (uint64_t *)malloc(sizeof(uint64_t) * (size_t)(M > 0 ? M : 1)) : NULL;
    uint64_t *Tb = fast ? (uint64_t *)malloc(sizeof(uint64_t) * (size_t)(N > 0 ? N : 1)) : NULL;
    int st = (Sa && Sb && ca && cb && (!fast || (Dij && Ta && Tb))) ? 0 : -1;
    if (st == 0 && K > 0) st = oracle_ozaki_split(A, M, K, lda, 0, rho, slices, Sa, ca, NULL);
    if (st == 0 && K > 0) st = oracle_ozaki_split(B, K, N, ldb, 1, rho, slices, Sb, cb, NULL);
    if (st == 0 && K > 0 && fast)
        st = oracle_ozaki_fast_d(A, B, M, N, K, lda, ldb, rho, slices, Dij, Ta, Tb);
    if (fast) d = slices;
    int64_t bad = 0;
    if (st == 0) {
        const double unit_bound = ldexp(1.0, OZ_M3 + 2 * (rho - OZ_M1));
        for (int64_t i = 0; i < M; ++i)
            for (int64_t j = 0; j < N; ++j) C[i * ldc + j] = 0.0;
        if (K > 0) {
            for (int p = 0; p < slices; ++p) {
                for (int q = 0; q < slices; ++q) {
                    if (p + q >= d) continue;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad)
#endif
                    for (int64_t i = 0; i < M; ++i) {
                        const double *ap = Sa + ((int64_t)p * M + i) * K;
                        for (int64_t j = 0; j < N; ++j) {
                            const double *bq = Sb + (int64_t)q * K * N + j;
                            double P = 0.0, D = 0.0;
                            for (int64_t k = 0; k < K; ++k) {
                                const double t = ap[k] * bq[k * N];
                                P = P + t;
                                D = D + fabs(t);
                            }
                            if (D > unit_bound) ++bad;
                            if (fast && p + q >= Dij[i * N + j]) continue;
                            const int e = (ca[i] - p * (beta + 1)) + (cb[j] - q * (beta + 1));
                            C[i * ldc + j] = C[i * ldc + j] + ldexp(P, e);
                        }
                    }
                }
            }
        }
    }
    if (inexact) *inexact = bad;
    free(Sa);
    free(Sb);
    free(ca);
    free(cb);
    free(Dij);
    free(Ta);
    free(Tb);
    return st;
}

/* Batch helpers for the Python side: decode / encode whole arrays. */
void oracle_decode_array(int fmt, const uint16_t *bits, int64_t n, double *out) {
    for (int64_t e = 0; e < n; ++e) out[e] = oracle_decode(fmt, bits[e]);
}

void oracle_encode_rne_array(int fmt, const double *x, int64_t n, uint16_t *out) {
    for (int64_t e = 0; e < n; ++e) out[e] = (uint16_t)oracle_encode_rne(fmt, x[e]);
}

/* Threads the row loop may use (1 without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
