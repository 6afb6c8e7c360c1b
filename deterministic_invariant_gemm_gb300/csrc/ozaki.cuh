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

// Writes the `slices` bfloat16 slices of x (vector exponent c1) to
// out[0], out[plane], out[2 plane], ...
__device__ __forceinline__ void ozaki_split_value(double x, int c1, int rho, int slices,
                                                  __nv_bfloat16* out, int64_t plane) {
    const int beta = 53 - rho;
    const uint64_t bits = static_cast<uint64_t>(__double_as_longlong(x));
    const int eb = static_cast<int>((bits >> 52) & 0x7FF);
    const uint64_t frac = bits & ((1ull << 52) - 1);
    // x = R 2^E with R a signed integer of at most 53 bits
    int64_t R = static_cast<int64_t>(eb != 0 ? (frac | (1ull << 52)) : frac);
    if (bits >> 63) R = -R;
    const int E = eb != 0 ? eb - 1075 : -1074;
    const float unit = __int_as_float((127 + rho - 53) << 23);   // 2^(rho - 53), exact in binary32
    for (int p = 0; p < slices; ++p) {
        const int g = c1 - p * (beta + 1) + rho - 53;   // exponent of sigma's last place
        int64_t n = 0;
        if (R != 0) {
            if (E >= g) {
                // x^(p) is a multiple of 2^g already: no rounding, nothing left
                n = R * (int64_t(1) << (E - g));
                R = 0;
            } else if (g - E <= 60) {
                const int shift = g - E;
                int64_t q = R >> shift;                            // floor
                const int64_t rem = R - q * (int64_t(1) << shift); // in [0, 2^shift)
                const int64_t half = int64_t(1) << (shift - 1);
                if (rem > half || (rem == half && (q & 1))) ++q;   // to nearest, ties to even
                n = q;
                R -= n * (int64_t(1) << shift);
            }
            // g - E > 60: |x^(p)| < 2^(g - 7), n = 0
        }
        out[p * plane] = __float2bfloat16_rn(static_cast<float>(n) * unit);
    }
}

// Rows of X [rows][cols] (leading dimension ld): one warp per row finds the
// row's maximum (integer max of the magnitude bit patterns: exact and
// order-free), stores c^(1) in exps[row], then splits the row into
// out[p * plane + row * out_ld + k].
constexpr int kOzakiRowWarps = 8;

__global__ void __launch_bounds__(kOzakiRowWarps * 32)
    ozaki_split_rows_kernel(const double* __restrict__ X, int64_t rows, int64_t cols, int64_t ld,
                            int rho, int slices, __nv_bfloat16* __restrict__ out, int64_t out_ld,
                            int64_t plane, int* __restrict__ exps) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * kOzakiRowWarps;
    for (int64_t r = static_cast<int64_t>(blockIdx.x) * kOzakiRowWarps + (threadIdx.x >> 5); r < rows;
         r += warps) {
        const double* x = X + r * ld;
        uint64_t m = 0;
        for (int64_t k = lane; k < cols; k += 32) {
            const uint64_t a = static_cast<uint64_t>(__double_as_longlong(x[k])) & 0x7FFFFFFFFFFFFFFFull;
            m = a > m ? a : m;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const uint64_t b = __shfl_xor_sync(0xFFFFFFFFu, m, o);
            m = b > m ? b : m;
        }
        const int c1 = ozaki_ceil_log2_bits(m);
        if (lane == 0) exps[r] = c1;
        for (int64_t k = lane; k < cols; k += 32)
            ozaki_split_value(x[k], c1, rho, slices, out + r * out_ld + k, plane);
    }
}

// Column maxima of X [rows][cols]: block (32 columns) x (8 row phases); each
// thread scans every eighth row of its column, the block combines the eight.
__global__ void __launch_bounds__(256)
    ozaki_col_exps_kernel(const double* __restrict__ X, int64_t rows, int64_t cols, int64_t ld,
                          int* __restrict__ exps) {
    __shared__ uint64_t part[8][32];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const int64_t j = static_cast<int64_t>(blockIdx.x) * 32 + tx;
    uint64_t m = 0;
    if (j < cols)
        for (int64_t r = ty; r < rows; r += 8) {
            const uint64_t a = static_cast<uint64_t>(__double_as_longlong(X[r * ld + j])) & 0x7FFFFFFFFFFFFFFFull;
            m = a > m ? a : m;
        }
    part[ty][tx] = m;
    __syncthreads();
    if (ty == 0 && j < cols) {
        for (int t = 1; t < 8; ++t) m = part[t][tx] > m ? part[t][tx] : m;
        exps[j] = ozaki_ceil_log2_bits(m);
    }
}

// The column split: element (r, j) of X [rows][cols] goes to
// out[p * plane + r * out_ld + j]; rows rows .. out_rows-1 of every slice
// (the padding up to a whole K block) are written as zeros.  Threads run
// along a row (coalesced), blocks along y step through the rows.
__global__ void __launch_bounds__(256)
    ozaki_split_cols_kernel(const double* __restrict__ X, int64_t rows, int64_t cols, int64_t ld,
                            int64_t out_rows, int rho, int slices, __nv_bfloat16* __restrict__ out,
                            int64_t out_ld, int64_t plane, const int* __restrict__ exps) {
    const int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (j >= cols) return;
    const int c1 = exps[j];
    for (int64_t r = blockIdx.y; r < out_rows; r += gridDim.y) {
        const double x = r < rows ? X[r * ld + j] : 0.0;
        ozaki_split_value(x, c1, rho, slices, out + r * out_ld + j, plane);
    }
}

}  // namespace bigemm
