/*
 * bigemm.h -- C ABI of libbigemm.so: a deterministic, batch-invariant BF16
 * matrix multiply C = A * B with FP32 accumulation, for NVIDIA GB300 (sm_103a).
 *
 * The operation (Tencent AI-infra article "腾讯エンジニア：大規模モデルの出力を
 * 確定させるための AI インフラ手法", section "Batch Invariance の由来"):
 *     A is [M, K], B is [K, N], C is [M, N],   C_ij = sum_{k=0}^{K-1} A_ik * B_kj.
 * Each output element's K-reduction order is fixed by K and the split-K count
 * alone: it never depends on M, on the other rows of the batch, on where a row
 * sits in the batch, or on run-to-run scheduling.  Concretely, for every (i, j):
 *   - the K axis is cut into blocks of BIGEMM_BLOCK_K = 64 ("Tiling": the
 *     per-CTA K loop in fixed steps; "Batch Invariance の由来": BLOCK_K fixes the
 *     reduction tree), consumed in ascending order by one tensor-core
 *     accumulator in FP32;
 *   - with split_k = S > 1 the blocks are dealt into S contiguous segments,
 *     each segment's FP32 partial goes to its own workspace slice, and a
 *     separate kernel adds the slices in the fixed order s = 0, 1, ..., S-1
 *     ("Split-K": workspace [split_k, M, N], partial GEMM kernel, reduction
 *     kernel) -- no atomics.  A product large enough to fill the GPU with
 *     whole tiles (bigemm_split_is_folded) instead has the CTA that owns a
 *     tile compute its S segment partials one after another and add them in
 *     the same order with the same FP32 additions; a smaller one (S <= 8),
 *     and every batch of at most 32 rows (the few-row kernel), may have the
 *     S CTAs of a thread-block cluster compute one segment each and add the
 *     partials through distributed shared memory, again in that order with
 *     those additions (bigemm_split_path).  The same bits every way, with no
 *     workspace traffic and no second kernel;
 *   - the M and N tile sizes and the order in which tiles run (a GROUP_M
 *     swizzle, "GROUP_M - Swizzle L2 Cache") change no sum.
 * So row i of C is bit-for-bit a function of (row i of A, B, K, split_k,
 * output type) only.
 *
 * Layouts.  All matrices are row-major with explicit leading dimensions in
 * elements: A[i*lda + k] (bf16), B[k*ldb + j] (bf16), C[i*ldc + j].  The
 * workspace of the split-K path holds S slices of M rows of
 * bigemm_workspace_ld(N) fp32 values: slice s, row i, column j at
 * ws[(s*M + i) * bigemm_workspace_ld(N) + j].
 *
 * Ownership and synchronisation.  The caller owns every buffer and the stream.
 * The library allocates no device memory, never synchronises, and returns as
 * soon as the work is enqueued on `stream` (a cudaStream_t; NULL is the legacy
 * default stream).  Buffers must stay valid until that work completes.  Calls
 * that share a workspace must be ordered (same stream or explicit events).
 * C must not overlap A, B or the workspace.
 *
 * Errors.  Every argument is checked before anything is enqueued; a failed
 * check returns an error code and enqueues nothing:
 *   BIGEMM_ERR_ARG        negative size, NULL pointer, ld smaller than the row
 *                         length, split_k outside [0, ceil(K/64)], sizes past
 *                         the int32 limits of the tile scheduler
 *   BIGEMM_ERR_ALIGN      a base pointer not 16-byte aligned, lda or ldb not a
 *                         multiple of 8 elements (16-byte rows for the tensor
 *                         memory accelerator), ldc not a multiple of 4 (fp32
 *                         C) or 8 (bf16 C)
 *   BIGEMM_ERR_WORKSPACE  workspace NULL, misaligned or smaller than
 *                         bigemm_workspace_bytes(M, N, K, split_k)
 *   BIGEMM_ERR_UNSUPPORTED the current device is not sm_103 / sm_100 class
 *   BIGEMM_ERR_CUDA       a CUDA runtime or driver call failed
 *   BIGEMM_ERR_TIMEOUT    reported by bigemm_device_status(): a kernel's
 *                         bounded wait expired; the kernel stopped early,
 *                         released its tensor memory and returned (its output
 *                         is then undefined)
 *   BIGEMM_ERR_STATIC_LIMIT bigemm_run_splitk_static only: the product needs
 *                         more split-K scratch than the built-in array holds
 * Empty products are valid: M == 0 or N == 0 enqueue nothing, K == 0 writes
 * zeros to C.
 */
#ifndef BIGEMM_H
#define BIGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define BIGEMM_API __attribute__((visibility("default")))
#else
#define BIGEMM_API
#endif

typedef enum {
    BIGEMM_OK = 0,
    BIGEMM_ERR_ARG = 1,
    BIGEMM_ERR_ALIGN = 2,
    BIGEMM_ERR_WORKSPACE = 3,
    BIGEMM_ERR_UNSUPPORTED = 4,
    BIGEMM_ERR_CUDA = 5,
    BIGEMM_ERR_TIMEOUT = 6,
    BIGEMM_ERR_STATIC_LIMIT = 7
} bigemm_status;

/* A cudaStream_t passed through the C ABI. */
typedef void *bigemm_stream;

/* K step of the tensor-core mainloop (elements).  Fixed: it is part of the
 * reduction order, so it never varies with the shape (Tencent article,
 * "Batch Invariance の由来": a different BLOCK_K gives a different but still
 * deterministic result). */
#define BIGEMM_BLOCK_K 64

/* Output tile of one work unit: BIGEMM_TILE_M rows x BIGEMM_TILE_N columns. */
#define BIGEMM_TILE_M 128
#define BIGEMM_TILE_N 256

/* A split product is folded (its segments summed inside the CTA, no
 * workspace) when it has at least BIGEMM_FOLD_MIN_ROWS rows and at least
 * BIGEMM_FOLD_MIN_TILES output tiles; see bigemm_split_is_folded. */
#define BIGEMM_FOLD_MIN_ROWS 97
#define BIGEMM_FOLD_MIN_TILES 128

/* A bf16 product (bigemm_run, bigemm_run_bf16out, bigemm_linear) of 1 ..
 * BIGEMM_SKINNY_MAX_ROWS rows whose effective split is at most
 * BIGEMM_SKINNY_MAX_SPLIT runs the few-row kernel: the S CTAs of each
 * 128 x 256 output tile form a thread-block cluster, one K segment each, and
 * add their partials through distributed shared memory (one launch, no
 * workspace); see BIGEMM_PATH_SKINNY. */
#define BIGEMM_SKINNY_MAX_ROWS 32
#define BIGEMM_SKINNY_MAX_SPLIT 8

/* Library version, (major << 16) | minor. */
BIGEMM_API int bigemm_version(void);

/* Human-readable name of a status code (static storage, never NULL). */
BIGEMM_API const char *bigemm_status_string(bigemm_status status);

/* max(1, ceil(K / BIGEMM_BLOCK_K)): the number of K blocks (at least 1),
 * and the largest split_k; 0 for K < 0. */
BIGEMM_API int bigemm_max_split_k(int64_t K);

/* The split-K count used when split_k = 0 is passed: a function of K alone,
 * never of M or N ("Split-K" is enabled for long K; "Batch Invariance の由来":
 * a split that varies with the batch breaks invariance).  It is the largest
 * power of two <= min(16, floor(K / 512)), and at least 1:
 * K < 1024 -> 1, K = 4096 -> 8, K >= 8192 -> 16. */
BIGEMM_API int bigemm_default_split_k(int64_t K);

/* Number of non-empty K segments for (K, split_k): with L = ceil(KB / S)
 * blocks per segment (KB = ceil(K/64)), this is ceil(KB / L) <= S.  The
 * reduction order depends on (K, split_k) only through this count and L.
 * split_k = 0 means bigemm_default_split_k(K).  Returns 0 for an invalid
 * split_k. */
BIGEMM_API int bigemm_effective_split_k(int64_t K, int split_k);

/* Row stride (elements) of the fp32 workspace slices: N rounded up to a
 * multiple of 4, so that every row starts 16-byte aligned. */
BIGEMM_API int64_t bigemm_workspace_ld(int64_t N);

/* 1 when a product of this shape with effective split S > 1 sums its
 * segments inside the CTA rather than through the workspace: M >=
 * BIGEMM_FOLD_MIN_ROWS and ceil(M / 128) * ceil(N / 256) >=
 * BIGEMM_FOLD_MIN_TILES, so that whole tiles alone occupy most SMs.  The
 * choice is one of speed only: both ways form every sum the same way (the
 * same segment partials, added in the order 0..S-1, each addition one FP32
 * addition rounded to nearest even), so row i of C has the same bits either
 * way.  A shape test only, for any K and split_k (8-bit products too); 0 for
 * invalid arguments or an effective split of 1. */
BIGEMM_API int bigemm_split_is_folded(int64_t M, int64_t N, int64_t K, int split_k);

/* How bigemm_run, bigemm_run_bf16out, bigemm_linear (fp8 = 0) or
 * bigemm_linear_fp8 (fp8 = 1) execute a product of this shape on the current
 * device -- a matter of speed only, every way forms each sum identically:
 *   BIGEMM_PATH_UNSPLIT    effective split 1 (or K = 0): one kernel;
 *   BIGEMM_PATH_WORKSPACE  partial kernel into the workspace, then
 *                          splitk_reduce_kernel (two kernels);
 *   BIGEMM_PATH_FOLDED     segments summed inside the CTA (one kernel);
 *   BIGEMM_PATH_CLUSTER    effective split S in 2..8 and every tile's cluster
 *                          of S CTAs resident at once: each CTA computes one
 *                          segment and the cluster adds the partials through
 *                          distributed shared memory in the order 0..S-1
 *                          (one kernel);
 *   BIGEMM_PATH_SKINNY     a bf16 product of 1 .. BIGEMM_SKINNY_MAX_ROWS rows
 *                          with effective split 2 .. BIGEMM_SKINNY_MAX_SPLIT:
 *                          the few-row kernel, clusters of S CTAs of a
 *                          footprint small enough that the next product's
 *                          CTAs start beside them and warm L2 with their
 *                          weights (one kernel, no workspace).  It also
 *                          serves such products unsplit (reported as
 *                          BIGEMM_PATH_UNSPLIT).
 * The choice is by shape alone except between CLUSTER and WORKSPACE, which
 * depends on the device's cluster capacity.
 * -1 for invalid arguments or when the device cannot be queried. */
/* Number of clusters of `splits` GEMM CTAs (one CTA per SM) the current
 * device can hold at once, as the CUDA occupancy calculator reports it; a
 * product clusters when its tiles are no more than this.  0 for splits
 * outside 2..8, -1 when the device cannot be queried. */
BIGEMM_API int bigemm_cluster_capacity(int splits);

#define BIGEMM_PATH_UNSPLIT 0
#define BIGEMM_PATH_WORKSPACE 1
#define BIGEMM_PATH_FOLDED 2
#define BIGEMM_PATH_CLUSTER 3
#define BIGEMM_PATH_SKINNY 4
BIGEMM_API int bigemm_split_path(int64_t M, int64_t N, int64_t K, int split_k, int fp8);

/* 1 when bigemm_run, bigemm_run_bf16out, bigemm_linear (fp8 = 0) or
 * bigemm_linear_fp8 (fp8 = 1) runs a product of this shape on CTA pairs, 0
 * when on single CTAs, -1 for invalid arguments or when the device cannot be
 * queried.  The 2-SM kernel serves products of at least 256 rows with
 * 256-wide tiles (bigemm_tile_n) that are unsplit (effective split 1) or
 * folded (bigemm_split_is_folded): a thread-block cluster of two CTAs on two
 * SMs computes a 256 x 256 output tile with tcgen05.mma.cta_group::2 (M =
 * 256, N = 256, K = 16 for bf16, 32 for 8-bit floats); each CTA loads its own
 * 128 rows of A and its own 128 columns of B (rows of W) with plain TMA loads
 * and holds its 128 rows of the FP32 sums in its TMEM; a folded split keeps
 * one sum per K segment and adds them in the order 0..S-1, as on one CTA.  By default (bigemm_set_pair_mode 1) it takes such a product
 * when its 256 x 256 tiles number at least twice bigemm_pair_capacity(): a
 * pair's lighter loads then outweigh its costlier start and finish.  A
 * choice of speed only (Tencent AI-infra article, "Tiling"): every output
 * element is the same FP32 accumulation chain over K, 16 k (bf16) or 32 k
 * (8-bit) per instruction in ascending order, as on one CTA -- the GPU tests
 * compare the two bit for bit. */
BIGEMM_API int bigemm_uses_pair(int64_t M, int64_t N, int64_t K, int split_k, int fp8);

/* When the 2-SM kernel runs, for products launched afterwards in this
 * process: 0 never, 1 by the rule above (the default), 2 for every product
 * it can serve (at least 256 rows, unsplit or folded, 256-wide tiles) -- for
 * comparisons and tests.  Returns the previous mode, or -1 for a mode
 * outside 0..2 (nothing changes). */
BIGEMM_API int bigemm_set_pair_mode(int mode);

/* CTA pairs of the 2-SM kernel the current device holds at once (the
 * occupancy calculator's count of 2-CTA clusters): the persistent grid's
 * size.  0 disables the 2-SM kernel; -1 when the device cannot be queried. */
BIGEMM_API int bigemm_pair_capacity(void);

/* Width in columns of the output tiles a product of this shape runs with on
 * the current device: BIGEMM_TILE_N (256), or 128 / 64 for a bf16 product
 * whose 256-wide work units (tiles x K segments) would occupy fewer than half
 * of the SMs while each unit streams at least 32 K blocks (small M and N,
 * long K: "Split-K" on the Tencent page names exactly this case, few output
 * tiles and a long K).  Narrow tiles put more SMs to work on such a product;
 * they never run on the folded or cluster paths (a split product with narrow
 * tiles takes BIGEMM_PATH_WORKSPACE).  Speed only: the tile width sets the N
 * extent of each 128-row tensor-core instruction, never which K blocks an
 * element sums or in what order, so every width gives the same bits (the GPU
 * tests compare rows computed at widths 64, 128 and 256).  fp8 = 1 asks for
 * bigemm_linear_fp8, always 256.  -1 for invalid arguments or when the device
 * cannot be queried. */
BIGEMM_API int bigemm_tile_n(int64_t M, int64_t N, int64_t K, int split_k, int fp8);

/* Workspace bytes bigemm_run / bigemm_run_bf16out / bigemm_linear need for
 * (M, N, K, split_k): effective_split * M * bigemm_workspace_ld(N) * 4 when
 * the effective split is > 1 and the product is neither folded
 * (bigemm_split_is_folded) nor a few-row one (M <= BIGEMM_SKINNY_MAX_ROWS
 * and effective split <= BIGEMM_SKINNY_MAX_SPLIT), else 0.  A function of the shape alone: the
 * workspace is required even when the product then runs on the cluster path,
 * which leaves it untouched.  Returns 0 for invalid arguments too. */
BIGEMM_API size_t bigemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int split_k);

/* Workspace bytes bigemm_run_partial needs: effective_split * M *
 * bigemm_workspace_ld(N) * 4, also when the effective split is 1. */
BIGEMM_API size_t bigemm_partial_workspace_bytes(int64_t M, int64_t N, int64_t K, int split_k);

/* C (fp32) = A * B.  A: bf16 [M, K] (lda), B: bf16 [K, N] (ldb), C: fp32
 * [M, N] (ldc).  split_k: 1 = no split, 0 = bigemm_default_split_k(K), S > 1 =
 * S segments whose FP32 partials are added in the order 0..S-1: through the
 * workspace and the reduction kernel, inside the CTA for products that fill
 * the GPU with tiles, or inside a thread-block cluster for small ones
 * (bigemm_split_path names the way; all give the same bits).  workspace /
 * workspace_bytes may be NULL / 0 when bigemm_workspace_bytes is 0. */
BIGEMM_API bigemm_status bigemm_run(const void *A, const void *B, float *C,
                         int64_t M, int64_t N, int64_t K,
                         int64_t lda, int64_t ldb, int64_t ldc,
                         int split_k, void *workspace, size_t workspace_bytes,
                         bigemm_stream stream);

/* As bigemm_run, but C is bf16: the FP32 result (after the split-K reduction
 * when split_k > 1) is rounded once to bf16, to nearest even. */
BIGEMM_API bigemm_status bigemm_run_bf16out(const void *A, const void *B, void *C,
                                 int64_t M, int64_t N, int64_t K,
                                 int64_t lda, int64_t ldb, int64_t ldc,
                                 int split_k, void *workspace, size_t workspace_bytes,
                                 bigemm_stream stream);

/* The split-K partial-product kernel alone ("Split-K": each segment writes
 * its partial to workspace[k_idx, m, n] without atomics).  Writes
 * bigemm_effective_split_k(K, split_k) slices (one slice when that is 1);
 * workspace_bytes must be >= bigemm_partial_workspace_bytes(M, N, K, split_k). */
BIGEMM_API bigemm_status bigemm_run_partial(const void *A, const void *B,
                                 int64_t M, int64_t N, int64_t K,
                                 int64_t lda, int64_t ldb, int split_k,
                                 void *workspace, size_t workspace_bytes,
                                 bigemm_stream stream);

/* The split-K reduction kernel alone ("Split-K": a separate light kernel sums
 * the workspace along the split axis).  For every (i, j):
 *     acc = ws[0][i][j];  acc = acc + ws[s][i][j] for s = 1 .. splits-1
 * each '+' one FP32 addition rounded to nearest even, in exactly that order;
 * then C[i*ldc + j] = acc (c_is_bf16 = 0) or acc rounded to bf16, nearest
 * even (c_is_bf16 = 1).  workspace layout as above, splits >= 1. */
BIGEMM_API bigemm_status bigemm_splitk_reduce(const float *workspace, int splits,
                                   int64_t M, int64_t N,
                                   void *C, int64_t ldc, int c_is_bf16,
                                   bigemm_stream stream);

/* Batch-invariant linear layer: C = A * W^T + bias, i.e.
 *     C_ij = sum_{k=0}^{K-1} A_ik * W_jk + bias_j
 * with the weight matrix in the layout linear layers keep it: W bf16 [N, K]
 * row-major (ldw >= K, a multiple of 8).  This is the call the Tencent
 * article's serving path routes a linear layer to when batch invariance is
 * on ("vLLM における GEMM の Batch Invariance サポート": linear_batch_invariant(x,
 * weight, bias)).  A bf16 [M, K] (lda), C [M, N] fp32 (c_is_bf16 = 0, ldc % 4
 * == 0) or bf16 (c_is_bf16 = 1, ldc % 8 == 0); bias bf16 [N], 16-byte
 * aligned, or NULL.
 * The reduction order is that of bigemm_run for the same K and split_k -- K
 * blocks of 64 in ascending order, S contiguous segments summed in the order
 * 0..S-1 -- and the bias is added last, one FP32 addition per element (in the
 * epilogue when S = 1, in the reduction kernel when S > 1).  Row i of C is
 * bit-for-bit a function of (row i of A, W, bias, K, split_k, output type).
 * The weight is read K-major, so the bits may differ from bigemm_run with B =
 * W^T; each entry point is batch-invariant on its own.  Workspace and errors
 * as in bigemm_run. */
BIGEMM_API bigemm_status bigemm_linear(const void *A, const void *W, const void *bias, void *C,
                                       int64_t M, int64_t N, int64_t K,
                                       int64_t lda, int64_t ldw, int64_t ldc,
                                       int split_k, int c_is_bf16,
                                       void *workspace, size_t workspace_bytes,
                                       bigemm_stream stream);

/* 8-bit float formats of bigemm_linear_fp8 (the values of the instruction
 * descriptor's format fields). */
#define BIGEMM_FP8_E4M3 0   /* 4 exponent, 3 fraction bits, no infinity ("fn") */
#define BIGEMM_FP8_E5M2 1   /* 5 exponent, 2 fraction bits, IEEE-style */

/* Number of non-empty K segments of an 8-bit float product: as
 * bigemm_effective_split_k, but a K block is 128 elements (128 bytes per row,
 * like 64 BF16 elements).  0 for an invalid split_k. */
BIGEMM_API int bigemm_fp8_effective_split_k(int64_t K, int split_k);

/* Workspace bytes bigemm_linear_fp8 needs: as bigemm_workspace_bytes with
 * the 8-bit effective split (0 when it is 1 or the product is folded). */
BIGEMM_API size_t bigemm_fp8_workspace_bytes(int64_t M, int64_t N, int64_t K, int split_k);

/* Batch-invariant linear layer with 8-bit float operands:
 *     C_ij = scale * (sum_{k=0}^{K-1} A_ik * W_jk) + bias_j
 * A: [M, K] bytes in format fmt_a (lda a multiple of 16), W: [N, K] bytes in
 * format fmt_w (ldw a multiple of 16), BIGEMM_FP8_E4M3 or BIGEMM_FP8_E5M2
 * (either may be mixed); scale: one FP32 factor, e.g. the product of per-tensor
 * quantisation scales; bias: bf16 [N] or NULL; C fp32 or bf16 as in
 * bigemm_linear.  The products are exact and accumulate in FP32 on the tensor
 * cores (tcgen05.mma.kind::f8f6f4, K = 32 per instruction), K blocks of 128
 * in ascending order, split-K segments summed in the order 0..S-1; then one
 * FP32 multiply by scale and one FP32 addition of the bias.  Row i of C is
 * bit-for-bit a function of (row i of A, W, formats, scale, bias, K, split_k,
 * output type) -- the pages' batch invariance carried to the FP8 products
 * they benchmark (cuTile article, "TileGymで行列積ベンチマーク"; Tencent
 * article, "vLLM における…": FP8 goes to other kernels there).  The workspace
 * holds bigemm_fp8_effective_split_k slices (bigemm_fp8_workspace_bytes). */
BIGEMM_API bigemm_status bigemm_linear_fp8(const void *A, const void *W, int fmt_a, int fmt_w,
                                           float scale, const void *bias, void *C,
                                           int64_t M, int64_t N, int64_t K,
                                           int64_t lda, int64_t ldw, int64_t ldc,
                                           int split_k, int c_is_bf16,
                                           void *workspace, size_t workspace_bytes,
                                           bigemm_stream stream);

/* Workspace bytes bigemm_run_fp8 needs: B transposed, N rows of
 * round_up(K, 16) bytes rounded up to 256, then bigemm_fp8_workspace_bytes.
 * 0 for invalid arguments. */
BIGEMM_API size_t bigemm_fp8_kn_workspace_bytes(int64_t M, int64_t N, int64_t K, int split_k);

/* The 8-bit float product with B in the [K, N] layout of bigemm_run:
 *     C_ij = scale * (sum_{k=0}^{K-1} A_ik * B_kj) + bias_j
 * B: [K, N] bytes in format fmt_b, ldb >= N a multiple of 16, 16-byte
 * aligned; everything else as in bigemm_linear_fp8.  The tensor cores read
 * 8-bit operands K-major, so a first kernel copies B transposed into the
 * workspace (N rows of round_up(K, 16) bytes, zero past K) and the product
 * then runs as bigemm_linear_fp8 with W = B^T: the same bits, row i of C a
 * function of (row i of A, B, formats, scale, bias, K, split_k, output
 * type).  One launch more than bigemm_linear_fp8 (bigemm_last_launch_count).
 * Workspace: bigemm_fp8_kn_workspace_bytes, 256-byte aligned. */
BIGEMM_API bigemm_status bigemm_run_fp8(const void *A, const void *B, int fmt_a, int fmt_b,
                                        float scale, const void *bias, void *C,
                                        int64_t M, int64_t N, int64_t K,
                                        int64_t lda, int64_t ldb, int64_t ldc,
                                        int split_k, int c_is_bf16,
                                        void *workspace, size_t workspace_bytes,
                                        bigemm_stream stream);

/* ------------------------------------------------------------------------
 * Binary64 matrix product by the Ozaki scheme on the bfloat16 tensor cores
 * (cuTile article, "倍精度行列積エミュレーション": "Ozaki Schemeについて",
 * "分解(Split)", "行列積の計算", "Fast Mode（GEMMの削減）", "Fused Split
 * Kernel（分割の融合）").  The pages give no API; these calls are this
 * library's.
 *
 * Every row of A and every column of B (a vector x) is split into `slices`
 * bfloat16 slices by the Veltkamp split, eqs. (1)-(5):
 *   c^(1) = ceil(log2 max_i |x_i|),  sigma = 0.75 * 2^(rho + c^(p)),
 *   v = fl((x^(p) + sigma) - sigma),  x^(p+1) = x^(p) - v,  xbar^(p) = 2^(-c^(p)) v,
 * with c^(p+1) = c^(p) - (53 - rho) - 1 (the residual's bound, so that every
 * exponent follows from the first maximum, as in the fused split) and
 *   rho = max(ceil(53 - (24 - log2 K) / 2), 53 - 8),
 * the value that makes every slice-pair product over all of K exact in FP32
 * (eq. (11)).  Each vector is scaled by its own maximum -- per row of A, per
 * column of B -- so row i of C depends on row i of A and on B only: the
 * product is batch-invariant like the rest of the library.  Then
 *   C_ij = sum over (p, q) with p + q < d, p outer and q inner, of
 *          2^(c_a^(p)_i + c_b^(q)_j) * (xbar_a^(p)_i . ybar_b^(q)_j)      eq. (10)
 * each term one binary64 addition in that fixed order, the products on the
 * tensor cores (exact).  Inputs must be finite, with every scaled term a
 * normal binary64 (|values| roughly within 2^-900 .. 2^900).
 * ---------------------------------------------------------------------- */

/* rho for inner length K (1 <= K <= 2^22), or -1. */
BIGEMM_API int bigemm_ozaki_rho(int64_t K);

/* The default number of slices for inner length K: the least s with
 * s * (54 - rho) - 1 >= 53, enough to carry every vector to binary64
 * precision below its maximum; -1 for K outside 1 .. 2^22. */
BIGEMM_API int bigemm_ozaki_default_slices(int64_t K);

/* Slice pairs (p, q), 0 <= p, q < slices, with p + q < d: the number of
 * tensor-core products bigemm_ozaki_dgemm runs per output tile.  -1 for
 * invalid arguments. */
BIGEMM_API int64_t bigemm_ozaki_pairs(int slices, int d);

/* Workspace bytes of bigemm_ozaki_dgemm (slices = 0: the default): the
 * slices of A [s][M][round_up(K, 8)] and of B [s][round_up(K, 64)]
 * [round_up(N, 8)] in bf16, then c^(1) of every row of A and every column
 * of B (int32), then one int32 per 128 x 256 tile of C (how many slice
 * pairs the tile has taken so far) and one more (set when a wait gives up),
 * then Fast Mode's masses of the rows of A and the columns of B (uint64),
 * each part 256-byte aligned.  0 for invalid arguments. */
BIGEMM_API size_t bigemm_ozaki_workspace_bytes(int64_t M, int64_t N, int64_t K, int slices);

/* The split alone.  X: binary64 [rows][ld].  axis 0: every row is a vector,
 * slice p of row r goes to out[p * rows * out_ld + r * out_ld + k]; axis 1:
 * every column, slice p of element (r, j) to out[p * out_rows * out_ld +
 * r * out_ld + j], rows rows .. out_rows-1 of every slice written as zeros
 * (out_rows >= rows).  out: bf16; exps: c^(1) per vector (int32).  rho in
 * 45 .. 52, slices in 1 .. 32. */
BIGEMM_API bigemm_status bigemm_ozaki_split(const double *X, int64_t rows, int64_t cols, int64_t ld,
                                            int axis, int rho, int slices, void *out, int64_t out_ld,
                                            int64_t out_rows, int *exps, bigemm_stream stream);

/* C = A * B in binary64.  A [M][lda], B [K][ldb] binary64 (8-byte aligned),
 * C [M][ldc] binary64 (16-byte aligned, ldc even).  slices: 0 = the default
 * (bigemm_ozaki_default_slices), else 1 .. 32; d: 0 = slices (the deterministic
 * binary64 bound: every skipped pair is below 2^-54 of its vectors' maxima),
 * smaller for Fast Mode's trade of accuracy for speed, or -1 for Fast Mode's
 * automatic d ("Fast Mode（GEMMの削減）": the smallest d meeting
 * |fl(AB) - AB| <= 2 sqrt(k) u |A||B|).  The page gives that bound, not its
 * procedure; here each element (i, j) takes its own d_ij, from row i of A
 * and column j of B only (so rows stay batch-invariant): with the vectors'
 * masses T = sum_k floor(|x_k| 2^(40 - c^(1))) (exact integers), d_ij is the
 * least d >= 1 with d (54 - rho) >= 134 + ceil(log2 slices) + ceil(log2 K) -
 * bitlen(T_a[i] T_b[j]), at most `slices` -- the skipped pairs' probabilistic
 * size (at most `slices` pairs per diagonal, sqrt(K) per dot product) against
 * 2 sqrt(K) 2^-53 times a mean-field estimate T_a T_b 2^(c_a + c_b - 80) / K
 * of |A||B|_ij.  The element adds the pairs with p + q < d_ij, in the usual
 * order; the kernel runs the pairs up to the largest d_ij.  K <= 2^22.  Four
 * launches: the row split of A, the column maxima and column split of B, and
 * one tensor-core kernel that runs every kept slice pair of each output tile
 * and keeps the binary64 sum in C (plus one memset of the tile counts).  The
 * kernel deals the (slice pair, tile) products over the SMs pair by pair, so
 * the pairs of one tile may run on different SMs at once; each element of C
 * still takes its pairs' terms one after another in the fixed pair order (a
 * tile's epilogue waits, bounded, for its count to show the previous pair).
 * With at least 256 rows and K < 4096 (and enough items for two waves) the
 * products run on CTA pairs (256 x 256 tiles, tcgen05.mma.cta_group::2; see
 * bigemm_uses_pair and bigemm_set_pair_mode), each CTA adding its 128 rows
 * under its 128 x 256 tile's count -- the same additions in the same order.
 * The kernel is a cooperative launch: CUDA starts it only when all of its
 * CTAs (at most one per SM) can be resident together, so those waits end
 * whatever else runs on the device, concurrent Ozaki products included.
 * Workspace: bigemm_ozaki_workspace_bytes, 256-byte aligned. */
BIGEMM_API bigemm_status bigemm_ozaki_dgemm(const double *A, const double *B, double *C,
                                            int64_t M, int64_t N, int64_t K,
                                            int64_t lda, int64_t ldb, int64_t ldc,
                                            int slices, int d,
                                            void *workspace, size_t workspace_bytes,
                                            bigemm_stream stream);

/* Measured contrast only -- NOT deterministic.  Same arguments as bigemm_run
 * without a workspace: C (fp32) is zeroed on the stream, then every K
 * segment's partial is added into C with atomic adds ("Split-K": atomic_add;
 * "Batch Invariance の由来": the hardware decides the order of the atomic
 * additions, so the bits vary from run to run). */
BIGEMM_API bigemm_status bigemm_run_atomic_splitk(const void *A, const void *B, float *C,
                                       int64_t M, int64_t N, int64_t K,
                                       int64_t lda, int64_t ldb, int64_t ldc,
                                       int split_k, bigemm_stream stream);

/* Size of the scratch array built into the library for
 * bigemm_run_splitk_static: 16 MiB of device memory on every GPU that loads
 * the library, held until the process exits. */
#define BIGEMM_STATIC_SCRATCH_BYTES (16u << 20)

/* Split-K product without a caller workspace and without any allocation.
 * The pages have no counterpart to this call: it exists for callers that
 * cannot allocate device memory or hand the library a scratch buffer -- for
 * example a serving loop that forbids allocation after start-up (cudaMalloc
 * may synchronise the whole device and stall unrelated streams), or a plugin
 * inside a host framework that owns all device memory through its own
 * allocator and does not expose it over a C interface.
 *
 * Arguments and result are those of bigemm_run (C fp32 [M, N]); the split-K
 * partial sums go to a BIGEMM_STATIC_SCRATCH_BYTES array compiled into the
 * library instead of a caller workspace, and the same two kernels run, so the
 * bits equal bigemm_run's for the same split_k.  It calls no cudaMalloc,
 * cudaFree or allocating library routine.
 *   - Products whose bigemm_workspace_bytes(M, N, K, split_k) exceeds
 *     BIGEMM_STATIC_SCRATCH_BYTES return BIGEMM_ERR_STATIC_LIMIT and enqueue
 *     nothing; use bigemm_run with a workspace, or a smaller split_k.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and keeps it; make
 *     that first call before any stream capture on the device.  The kept
 *     address belongs to the device's primary context: it does not survive
 *     cudaDeviceReset (or any teardown of that context), after which this
 *     call must not be used again in the process.
 *   - Every call on a device shares the one array, which keeps the last
 *     call's contents.  Nothing in it needs to start at zero: each call's
 *     partial kernel writes every element its reduction reads.  Calls that
 *     can overlap on the GPU (other streams, no ordering event) race on it
 *     and corrupt each other's results; order them. */
BIGEMM_API bigemm_status bigemm_run_splitk_static(const void *A, const void *B, float *C,
                                                  int64_t M, int64_t N, int64_t K,
                                                  int64_t lda, int64_t ldb, int64_t ldc,
                                                  int split_k, bigemm_stream stream);

/* Reads (and, if reset != 0, clears) the device-side error word the kernels
 * set when a bounded wait expires.  Synchronises the current device.
 * Returns BIGEMM_OK, BIGEMM_ERR_TIMEOUT or BIGEMM_ERR_CUDA. */
BIGEMM_API bigemm_status bigemm_device_status(int reset);

/* Self-test of the failure path; the pages have no counterpart.  Enqueues one
 * split-K partial kernel (16 x 256 x 512, operands in the built-in scratch
 * array of bigemm_run_splitk_static) whose producer issues no loads, so its
 * MMA issuer's bounded wait gives up after 2 s: the kernel raises its abort
 * flag, the other roles leave their waits, nothing is loaded or stored, TMEM
 * is freed and the kernel ends with the wait's bit set in the device error
 * word.  A later bigemm_device_status() then returns BIGEMM_ERR_TIMEOUT, and
 * the context stays usable.  Shares the scratch array with
 * bigemm_run_splitk_static (calls must not overlap). */
BIGEMM_API bigemm_status bigemm_selftest_timeout(bigemm_stream stream);

/* Self-test of the Ozaki kernel's failure path; the pages have no counterpart.
 * Enqueues a 256 x 256 x 128 binary64 product of zero matrices, with its
 * operands, output and workspace in the built-in scratch array, whose tile
 * counts start far below zero, so that no epilogue's bounded wait for the
 * previous slice pair of its tile is ever met.  The first wait to give up
 * after 2 s sets the launch's abort word, and every other CTA then leaves its
 * waits at once (rather than each running out its own 2 s); the kernel ends
 * with the wait's bit in the device error word, so a later
 * bigemm_device_status() returns BIGEMM_ERR_TIMEOUT, and the context stays
 * usable.  Shares the scratch array with bigemm_run_splitk_static (calls
 * must not overlap). */
BIGEMM_API bigemm_status bigemm_selftest_ozaki_order_timeout(bigemm_stream stream);

/* Number of kernels the most recent successful call on this host thread
 * enqueued (0 to 4). */
BIGEMM_API int bigemm_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* BIGEMM_H */
