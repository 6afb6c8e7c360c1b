// ozaki.cuh -- the split of the Ozaki scheme (cuTile article, "倍精度行列積
// エミュレーション": "分解(Split)" and "Fused Split Kernel（分割の融合）").
//
// A binary64 vector x (a row of A or a column of B) becomes `slices` bfloat16
// slices xbar^(p) with exponents c^(p), x = sum_p 2^(c^(p)) xbar^(p) + residual:
//   c^(1)    = ceil(log2 max_i |x_i|)                                   eq. (1)
//   v        = fl((x^(p) + sigma) - sigma), sigma = 0.75 * 2^(rho + c^(p))  (2)-(3)
//   x^(p+1)  = x^(p) - v                                                eq. (4)
//   xbar^(p) = 2^(-c^(p)) v, exactly a bfloat16                         eq. (5)
// and, as in the fused split kernel, every later exponent follows from the
// first maximum: c^(p+1) = c^(p) - beta - 1 with beta = 53 - rho, the bound
// eq. (3) puts on the residual (half a unit in the last place of sigma).
//
// Adding and subtracting sigma rounds x^(p) to the nearest multiple of
// 2^g, g = rho + c^(p) - 53 (the last place of sigma), ties to even: sigma =
// 3 * 2^(g + 51) is an even multiple of 2^g and x^(p) + sigma stays in
// sigma's binade.  The kernels below do exactly that rounding in 64-bit
// integers on the significand of x instead of two binary64 additions --
// binary64 arithmetic is scarce on this GPU -- so v = n 2^g with
//   n = round-half-even(x^(p) / 2^g),  |n| <= 2^beta,
// and xbar^(p) = n 2^(rho - 53).
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace bigemm {

// ceil(log2 m) for the bit pattern of a positive binary64 m; 0 for m = 0 (an
// all-zero vector, whose slices are all zero).
__device__ __forceinline__ int ozaki_ceil_log2_bits(uint64_t m) {
    if (m == 0) return 0;
    const int eb = static_cast<int>(m >> 52);
    const uint64_t frac = m & ((1ull << 52) - 1);
    if (eb != 0) return eb - 1023 + (frac != 0 ? 1 : 0);
    const int fl = 63 - __clzll(static_cast<long long>(frac));   // subnormal: frac * 2^-1074
    return fl - 1074 + ((frac & (frac - 1)) != 0 ? 1 : 0);
}

// One element's split state: x = R 2^E with R a signed integer of at most
// 53 bits.
struct OzakiElem {
    int64_t R;
    int E;
};

__device__ __forceinline__ OzakiElem ozaki_elem(double x) {
    const uint64_t bits = static_cast<uint64_t>(__double_as_longlong(x));
    const int eb = static_cast<int>((bits >> 52) & 0x7FF);
    const uint64_t frac = bits & ((1ull << 52) - 1);
    OzakiElem e;
    e.R = static_cast<int64_t>(eb != 0 ? (frac | (1ull << 52)) : frac);
    if (bits >> 63) e.R = -e.R;
    e.E = eb != 0 ? eb - 1075 : -1074;
    return e;
}

// The slices from single roundings.  With s_p = g_p - E the shift of slice
// p and F_p = n_0 2^(s_0) + ... + n_p 2^(s_p) (in units of 2^E), the
// sequential split gives F_p = round-half-even(R / 2^(s_p)) 2^(s_p): F_(p-1)
// is a multiple of 2^(s_(p-1)) = 2^(s_p + beta + 1), an even multiple of
// 2^(s_p), and rounding to a grid commutes with adding an even number of
// grid steps, ties included.  So
//   n_p = Q_p - 2^(beta+1) Q_(p-1),   Q_p = round-half-even(R / 2^(s_p)),
// Q_(-1) = 0 (|x| <= 2^(c^(1)) makes |Q_0| <= 2^beta).  |n_p| <= 2^beta, so
// the low 32 bits of each Q suffice (arithmetic modulo 2^32).
//
// Low 32 bits of round-half-even(R / 2^s): for s > 0 the quotient is
// floor((R + 2^(s-1)) / 2^s), round-half-up; a tie is exactly the case where
// R + 2^(s-1) is a multiple of 2^s, and there an odd result moves down by one
// to its even neighbour.  s >= 54 leaves 0 (|R| < 2^53 <= 2^(s-1)); s <= 0 is
// an exact left shift.
__device__ __forceinline__ uint32_t ozaki_round_lo32(int64_t R, int s) {
    if (s <= 0) return -s < 32 ? static_cast<uint32_t>(static_cast<uint64_t>(R) << (-s)) : 0u;
    if (s >= 54) return 0u;
    const int64_t t = R + (int64_t(1) << (s - 1));
    int64_t q = t >> s;  // arithmetic shift: floor
    if ((q & 1) && (t & ((int64_t(1) << s) - 1)) == 0) --q;
    return static_cast<uint32_t>(q);
}

// n 2^(rho - 53) in binary32, exactly: n (|n| <= 256) through the bit
// pattern of 1.5 * 2^23 + n (the integers of that binade are exact), then a
// power-of-two scale.
__device__ __forceinline__ float ozaki_slice_value(int n, float unit) {
    return (__int_as_float(0x4B400000 + n) - 12582912.0f) * unit;
}

__device__ __forceinline__ float ozaki_unit(int rho) {
    return __int_as_float((127 + rho - 53) << 23);  // 2^(rho - 53), exact in binary32
}

// The same Q_p through one window per element.  |R| is shifted once so that
// slice 0's unit sits at bit 96 of a 128-bit word W = |R| 2^(96 - s_0) (held
// as four 32-bit words); slice p's unit is then bit pos = 96 - p (beta + 1)
// for every element, and
//   Q_p = floor(W / 2^pos) + [bit pos-1 of W] * ([W has a 1 below bit pos-1]
//                                                 or floor(W / 2^pos) odd),
// round-half-even, with "a 1 below" read off W's trailing zero count.  RNE is
// odd-symmetric, so the slices of -|R| are the negated slices of |R|.  Exact
// when no bit of |R| falls below the window (s_0 <= 96) -- the element is
// not far below the vector's maximum -- and every slice's unit lies in it
// ((slices - 1)(beta + 1) <= 95); ozaki_window returns false otherwise and
// the caller keeps the per-slice rounding above.  One variable shift per
// element instead of one 64-bit rounding per slice.
struct OzakiWindow {
    uint32_t w0, w1, w2, w3;  // W, least significant word first
    int tz;                   // trailing zeros of W (a large value for W = 0)
    bool neg;
};

__device__ __forceinline__ bool ozaki_window(double x, int c1, int rho, OzakiWindow& W) {
    const uint64_t bits = static_cast<uint64_t>(__double_as_longlong(x));
    const int eb = static_cast<int>((bits >> 52) & 0x7FF);
    const uint64_t U = (bits & ((1ull << 52) - 1)) | (eb != 0 ? (1ull << 52) : 0ull);
    const int E = eb != 0 ? eb - 1075 : -1074;
    const int k = 96 - (c1 + rho - 53 - E);  // W = U 2^k; k <= 96 + beta when |x| <= 2^c1
    if (k < 0 || k > 104) return false;
    uint64_t lo, hi;
    if (k >= 64) {
        lo = 0;
        hi = U << (k - 64);
    } else if (k > 0) {
        lo = U << k;
        hi = U >> (64 - k);
    } else {
        lo = U;
        hi = 0;
    }
    W.w0 = static_cast<uint32_t>(lo);
    W.w1 = static_cast<uint32_t>(lo >> 32);
    W.w2 = static_cast<uint32_t>(hi);
    W.w3 = static_cast<uint32_t>(hi >> 32);
    W.tz = lo != 0 ? __ffsll(static_cast<long long>(lo)) - 1
                   : (hi != 0 ? 63 + __ffsll(static_cast<long long>(hi)) : (1 << 20));
    W.neg = (bits >> 63) != 0;
    return true;
}

// Low 32 bits of Q_p for the slice whose unit is bit pos (1 .. 96) of W.
__device__ __forceinline__ uint32_t ozaki_window_q(const OzakiWindow& W, int pos) {
    uint32_t a, h;
    if (pos >= 64) {
        a = __funnelshift_rc(W.w2, W.w3, pos - 64);
        h = pos > 64 ? (W.w2 >> (pos - 65)) : (W.w1 >> 31);
    } else if (pos >= 32) {
        a = __funnelshift_rc(W.w1, W.w2, pos - 32);
        h = pos > 32 ? (W.w1 >> (pos - 33)) : (W.w0 >> 31);
    } else {
        a = __funnelshift_r(W.w0, W.w1, pos);
        h = W.w0 >> (pos - 1);
    }
    return a + (h & 1u & ((W.tz < pos - 1 ? 1u : 0u) | a));
}

// Slice p of two adjacent elements: out[p * plane] and out[p * plane + 1],
// one 4-byte store when `paired`.
__device__ __forceinline__ void ozaki_store_two(__nv_bfloat16* out, int64_t plane, int p, int na, int nb,
                                                float unit, bool paired) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(ozaki_slice_value(na, unit), ozaki_slice_value(nb, unit));
    __nv_bfloat16* o = out + p * plane;
    if (paired) {
        *reinterpret_cast<__nv_bfloat162*>(o) = v;
    } else {
        o[0] = __low2bfloat16(v);
        o[1] = __high2bfloat16(v);
    }
}

// Splits two adjacent elements (vector exponents c1a, c1b) into `slices`
// slices each; slice p of the pair goes to out[p * plane] and out[p * plane
// + 1], as one 4-byte store when `paired`.  Every value is a bfloat16 exactly.
// Both elements through their windows when both fit, else both through the
// per-slice rounding (the same n_p either way).
__device__ __forceinline__ void ozaki_split_two(double xa, double xb, int c1a, int c1b, int rho,
                                                int slices, __nv_bfloat16* out, int64_t plane,
                                                bool paired) {
    const int w = 54 - rho;  // beta + 1
    const float unit = ozaki_unit(rho);
    OzakiWindow wa, wb;
    if ((slices - 1) * w <= 95 && ozaki_window(xa, c1a, rho, wa) && ozaki_window(xb, c1b, rho, wb)) {
        uint32_t pa = 0, pb = 0;
        for (int p = 0; p < slices; ++p) {
            const int pos = 96 - p * w;
            const uint32_t qa = ozaki_window_q(wa, pos), qb = ozaki_window_q(wb, pos);
            const int na = static_cast<int>(qa - (pa << w)), nb = static_cast<int>(qb - (pb << w));
            pa = qa;
            pb = qb;
            ozaki_store_two(out, plane, p, wa.neg ? -na : na, wb.neg ? -nb : nb, unit, paired);
        }
        return;
    }
    const OzakiElem a = ozaki_elem(xa), b = ozaki_elem(xb);
    int sa = c1a + rho - 53 - a.E, sb = c1b + rho - 53 - b.E;
    uint32_t pa = 0, pb = 0;
    for (int p = 0; p < slices; ++p, sa -= w, sb -= w) {
        const uint32_t qa = ozaki_round_lo32(a.R, sa), qb = ozaki_round_lo32(b.R, sb);
        const int na = static_cast<int>(qa - (pa << w)), nb = static_cast<int>(qb - (pb << w));
        pa = qa;
        pb = qb;
        ozaki_store_two(out, plane, p, na, nb, unit, paired);
    }
}

// ozaki_split_two for the slice width kW = beta + 1 = 54 - rho and slice
// count kS fixed at compile time (the common (K, slices) choices): the loop
// over slices unrolls and every window position is a constant.
template <int kW, int kS>
__device__ __forceinline__ void ozaki_split_two_fixed(double xa, double xb, int c1a, int c1b, int rho,
                                                      __nv_bfloat16* out, int64_t plane, bool paired) {
    static_assert(kW >= 1 && kS >= 1 && (kS - 1) * kW <= 95, "every slice's unit inside the window");
    OzakiWindow wa, wb;
    if (ozaki_window(xa, c1a, rho, wa) && ozaki_window(xb, c1b, rho, wb)) {
        const float unit = ozaki_unit(rho);
        uint32_t pa = 0, pb = 0;
#pragma unroll
        for (int p = 0; p < kS; ++p) {
            const uint32_t qa = ozaki_window_q(wa, 96 - p * kW), qb = ozaki_window_q(wb, 96 - p * kW);
            const int na = static_cast<int>(qa - (pa << kW)), nb = static_cast<int>(qb - (pb << kW));
            pa = qa;
            pb = qb;
            ozaki_store_two(out, plane, p, wa.neg ? -na : na, wb.neg ? -nb : nb, unit, paired);
        }
        return;
    }
    ozaki_split_two(xa, xb, c1a, c1b, rho, kS, out, plane, paired);
}

// kW = 0: the slice width and count from rho and slices at run time.
template <int kW, int kS>
__device__ __forceinline__ void ozaki_split_two_as(double xa, double xb, int c1a, int c1b, int rho, int slices,
                                                   __nv_bfloat16* out, int64_t plane, bool paired) {
    if constexpr (kW > 0)
        ozaki_split_two_fixed<kW, kS>(xa, xb, c1a, c1b, rho, out, plane, paired);
    else
        ozaki_split_two(xa, xb, c1a, c1b, rho, slices, out, plane, paired);
}

// One element alone (an odd vector's last element).
__device__ __forceinline__ void ozaki_split_one(double x, int c1, int rho, int slices,
                                                __nv_bfloat16* out, int64_t plane) {
    const int w = 54 - rho;
    const float unit = ozaki_unit(rho);
    const OzakiElem a = ozaki_elem(x);
    int s = c1 + rho - 53 - a.E;
    uint32_t prev = 0;
    for (int p = 0; p < slices; ++p, s -= w) {
        const uint32_t q = ozaki_round_lo32(a.R, s);
        out[p * plane] = __float2bfloat16_rn(ozaki_slice_value(static_cast<int>(q - (prev << w)), unit));
        prev = q;
    }
}

// Fast Mode's mass of a vector (its 1-norm from below, exactly and in any
// order): sum_k floor(|x_k| 2^(40 - c^(1))), each term at most 2^40 since
// |x_k| <= 2^(c^(1)), so the sum fits 64 bits for up to 2^23 terms.  The term
// of one element from its bit pattern: |x| = R 2^E, shifted by E + 40 - c.
__device__ __forceinline__ unsigned long long ozaki_mass_term(double x, int c1) {
    const OzakiElem a = ozaki_elem(x);
    const unsigned long long R = static_cast<unsigned long long>(a.R < 0 ? -a.R : a.R);
    if (R == 0) return 0ull;
    const int sh = a.E + 40 - c1;
    if (sh >= 0) return R << sh;  // < 2^41: |x| <= 2^c1
    return -sh >= 64 ? 0ull : (R >> -sh);
}

// Rows of X [rows][cols] (leading dimension ld): one block per row.  Each
// thread holds up to kOzakiRowCache elements (pairs of adjacent columns) in
// registers, so the row is read from memory once when cols <= 256 *
// kOzakiRowCache; the block finds the row's maximum (integer max of the
// magnitude bit patterns: exact and order-free), stores c^(1) in exps[row],
// and splits the row into out[p * plane + row * out_ld + k]; with `mass`
// not NULL it also stores the row's Fast Mode mass in mass[row].  A cache
// of 16 elements (rows up to 4096 read once) keeps three blocks per SM
// resident: at 4096 x 4096 the kernel took 187 us against 236 us with 32
// elements and two blocks, and 128 us with the slice shape fixed (kW, kS).
constexpr int kOzakiRowThreads = 256;
constexpr int kOzakiRowCache = 16;  // elements per thread kept in registers

__device__ __forceinline__ uint64_t ozaki_abs_bits(double x) {
    return static_cast<uint64_t>(__double_as_longlong(x)) & 0x7FFFFFFFFFFFFFFFull;
}

template <int kW = 0, int kS = 0>
__global__ void __launch_bounds__(kOzakiRowThreads, 3)
    ozaki_split_rows_kernel(const double* __restrict__ X, int64_t rows, int64_t cols, int64_t ld,
                            int rho, int slices, __nv_bfloat16* __restrict__ out, int64_t out_ld,
                            int64_t plane, int* __restrict__ exps, unsigned long long* __restrict__ mass) {
    __shared__ uint64_t wmax[kOzakiRowThreads / 32];
    const int tid = threadIdx.x;
    const int64_t pairs = cols / 2;
    const bool paired = (out_ld % 2 == 0) && ((reinterpret_cast<uintptr_t>(out) & 3u) == 0);
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const double* x = X + r * ld;
        double cache[kOzakiRowCache];
        uint64_t m = 0;
#pragma unroll
        for (int i = 0; i < kOzakiRowCache / 2; ++i) {
            const int64_t pr = tid + static_cast<int64_t>(i) * kOzakiRowThreads;
            cache[2 * i] = pr < pairs ? x[2 * pr] : 0.0;
            cache[2 * i + 1] = pr < pairs ? x[2 * pr + 1] : 0.0;
            m = max(m, max(ozaki_abs_bits(cache[2 * i]), ozaki_abs_bits(cache[2 * i + 1])));
        }
        // the rest of a long row (read again for the split)
        for (int64_t pr = tid + static_cast<int64_t>(kOzakiRowCache / 2) * kOzakiRowThreads; pr < pairs;
             pr += kOzakiRowThreads)
            m = max(m, max(ozaki_abs_bits(x[2 * pr]), ozaki_abs_bits(x[2 * pr + 1])));
        if ((cols & 1) && tid == 0) m = max(m, ozaki_abs_bits(x[cols - 1]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        if ((tid & 31) == 0) wmax[tid >> 5] = m;
        __syncthreads();
        m = wmax[0];
#pragma unroll
        for (int w = 1; w < kOzakiRowThreads / 32; ++w) m = max(m, wmax[w]);
        __syncthreads();  // wmax is reused by the next row
        const int c1 = ozaki_ceil_log2_bits(m);
        if (tid == 0) exps[r] = c1;
        if (mass != nullptr) {
            // integer sums: the same total in any order
            unsigned long long t = 0;
#pragma unroll
            for (int i = 0; i < kOzakiRowCache / 2; ++i) {
                const int64_t pr = tid + static_cast<int64_t>(i) * kOzakiRowThreads;
                if (pr < pairs) t += ozaki_mass_term(cache[2 * i], c1) + ozaki_mass_term(cache[2 * i + 1], c1);
            }
            for (int64_t pr = tid + static_cast<int64_t>(kOzakiRowCache / 2) * kOzakiRowThreads; pr < pairs;
                 pr += kOzakiRowThreads)
                t += ozaki_mass_term(x[2 * pr], c1) + ozaki_mass_term(x[2 * pr + 1], c1);
            if ((cols & 1) && tid == 0) t += ozaki_mass_term(x[cols - 1], c1);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xFFFFFFFFu, t, o);
            if ((tid & 31) == 0) wmax[tid >> 5] = t;
            __syncthreads();
            if (tid == 0) {
                for (int w = 1; w < kOzakiRowThreads / 32; ++w) t += wmax[w];
                mass[r] = t;
            }
            __syncthreads();  // wmax is reused by the next row
        }
        __nv_bfloat16* orow = out + r * out_ld;
#pragma unroll
        for (int i = 0; i < kOzakiRowCache / 2; ++i) {
            const int64_t pr = tid + static_cast<int64_t>(i) * kOzakiRowThreads;
            if (pr < pairs)
                ozaki_split_two_as<kW, kS>(cache[2 * i], cache[2 * i + 1], c1, c1, rho, slices, orow + 2 * pr, plane,
                                paired);
        }
        for (int64_t pr = tid + static_cast<int64_t>(kOzakiRowCache / 2) * kOzakiRowThreads; pr < pairs;
             pr += kOzakiRowThreads)
            ozaki_split_two_as<kW, kS>(x[2 * pr], x[2 * pr + 1], c1, c1, rho, slices, orow + 2 * pr, plane,
                                       paired);
        if ((cols & 1) && tid == 0) ozaki_split_one(x[cols - 1], c1, rho, slices, orow + cols - 1, plane);
    }
}

// Column maxima of X [rows][cols]: block (32 columns) x (8 row phases) over a
// chunk of `chunk` rows (blockIdx.y; at least kOzakiColChunk, a multiple of
// 8); each thread scans every eighth
// row of its column in the chunk, the block combines the eight, and the
// chunk's ceil(log2(max)) is merged into exps[j] with an integer atomicMax
// (ceil(log2) is monotone, so the merged value is ceil(log2) of the column
// maximum whatever the order).  exps must hold kOzakiNoExp beforehand; a
// chunk of zeros merges nothing, and an all-zero column keeps kOzakiNoExp
// (read as 0 by the split below).
constexpr int kOzakiColChunk = 256;
constexpr int kOzakiNoExp = static_cast<int>(0x80808080u);  // every byte 0x80: below any c^(1)

__global__ void __launch_bounds__(256)
    ozaki_col_exps_kernel(const double* __restrict__ X, int64_t rows, int64_t cols, int64_t ld,
                          int64_t chunk, int* __restrict__ exps) {
    __shared__ uint64_t part[8][32];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const int64_t j = static_cast<int64_t>(blockIdx.x) * 32 + tx;
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * chunk;
    const int64_t r1 = min(rows, r0 + chunk);
    uint64_t m = 0;
    if (j < cols) {
#pragma unroll 8
        for (int64_t r = r0 + ty; r < r1; r += 8) m = max(m, ozaki_abs_bits(X[r * ld + j]));
    }
    part[ty][tx] = m;
    __syncthreads();
    if (ty == 0 && j < cols) {
        for (int t = 1; t < 8; ++t) m = max(m, part[t][tx]);
        if (m != 0) atomicMax(exps + j, ozaki_ceil_log2_bits(m));
    }
}

// The column split: element (r, j) of X [rows][cols] goes to
// out[p * plane + r * out_ld + j]; rows rows .. out_rows-1 of every slice
// (the padding up to a whole K block) are written as zeros.  A thread takes
// two adjacent columns (one 4-byte store per slice when out_ld is even),
// blocks along y step through the rows.  Blocks with blockIdx.y == 0 also
// turn an all-zero column's kOzakiNoExp into its c^(1) = 0.  With `mass` not
// NULL (zero beforehand) every thread adds its rows' Fast Mode mass terms
// into mass[j] with one integer atomic addition per column: order-free.
template <int kW = 0, int kS = 0>
__global__ void __launch_bounds__(256)
    ozaki_split_cols_kernel(const double* __restrict__ X, int64_t rows, int64_t cols, int64_t ld,
                            int64_t out_rows, int rho, int slices, __nv_bfloat16* __restrict__ out,
                            int64_t out_ld, int64_t plane, int* __restrict__ exps,
                            unsigned long long* __restrict__ mass) {
    const int64_t j = 2 * (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x);
    if (j >= cols) return;
    const bool two = j + 1 < cols;
    const bool paired = two && (out_ld % 2 == 0) && ((reinterpret_cast<uintptr_t>(out) & 3u) == 0);
    int ea = exps[j];
    int eb = two ? exps[j + 1] : 0;
    ea = ea == kOzakiNoExp ? 0 : ea;
    eb = eb == kOzakiNoExp ? 0 : eb;
    if (blockIdx.y == 0) {
        exps[j] = ea;
        if (two) exps[j + 1] = eb;
    }
    unsigned long long ta = 0, tb = 0;
    for (int64_t r = blockIdx.y; r < out_rows; r += gridDim.y) {
        __nv_bfloat16* o = out + r * out_ld + j;
        if (two) {
            const double xa = r < rows ? X[r * ld + j] : 0.0;
            const double xb = r < rows ? X[r * ld + j + 1] : 0.0;
            ozaki_split_two_as<kW, kS>(xa, xb, ea, eb, rho, slices, o, plane, paired);
            if (mass != nullptr) {
                ta += ozaki_mass_term(xa, ea);
                tb += ozaki_mass_term(xb, eb);
            }
        } else {
            const double xa = r < rows ? X[r * ld + j] : 0.0;
            ozaki_split_one(xa, ea, rho, slices, o, plane);
            if (mass != nullptr) ta += ozaki_mass_term(xa, ea);
        }
    }
    if (mass != nullptr) {
        if (ta != 0) atomicAdd(mass + j, ta);
        if (two && tb != 0) atomicAdd(mass + j + 1, tb);
    }
}

}  // namespace bigemm
