// kernels.cuh -- the device side of the deterministic, batch-invariant BF16 GEMM.
//
// Work decomposition (Tencent AI-infra article "腾讯エンジニア：大規模モデルの出力を
// 確定させるための AI インフラ手法"):
//   * "Tiling": one work unit computes a kBM x kBN tile of C over one K segment;
//     its accumulator lives in tensor memory (TMEM) and is fed by a K loop in
//     fixed steps of kBK = 64, each step four tcgen05.mma of K = 16, in
//     ascending k.
//   * "Split-K": with S > 1 segments the K blocks are dealt into S contiguous
//     segments; each unit writes its FP32 partial to workspace slice s with plain
//     stores, and splitk_reduce_kernel adds the slices in the order 0..S-1.
//   * "GROUP_M - Swizzle L2 Cache": units are ordered in groups of GROUP_M tile
//     rows; a persistent grid of at most one CTA per SM takes units
//     blockIdx.x, blockIdx.x + gridDim.x, ... -- a static schedule.
// None of the three changes the order in which any single C element's terms
// are added, so the bits of row i depend only on (row i of A, B, K, S).  The
// same 128-row, K = 16 MMA instruction and operand roles are used for every M:
// short batches are padded by the TMA unit's zero fill, never served by a
// different code path.  The instruction's N extent is the tile width, 256,
// or 128 / 64 for small products with long K (Tile<kTN> below); it sets which
// columns an instruction covers, not how any column's sum is formed.
//
// CTA roles (384 threads = three warpgroups, one CTA per SM):
//   warp 0       TMA producer: fills a kStages-deep shared-memory ring.
//   warp 1       allocates TMEM; one lane issues the MMAs and commits.
//   warps 2, 3   set-up only (barrier initialisation).
//   warps 4..11  epilogue, two warps per TMEM lane quarter, each taking half
//                of the tile's columns: TMEM -> registers -> swizzled
//                shared-memory boxes -> TMA stores; two TMEM accumulators let
//                the epilogue of tile t overlap the mainloop of tile t + 1.
// The first warpgroup gives most of its registers to the two epilogue
// warpgroups, which hold up to a 32 x 256 FP32 block per warp (a folded
// tile's running sum).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace bigemm {

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kUmmaK = 16;
constexpr int kNumThreads = 384;       // warp 0 TMA, warp 1 MMA, warps 4..11 epilogue
constexpr int kEpilogueThreads = 256;
constexpr int kEpilogueWarps = kEpilogueThreads / 32;
constexpr int kEpilogueWarp0 = 4;      // first epilogue warp: the second warpgroup

// Register split.  The block is launched with kLaunchRegs registers per thread
// (65536 over 384 threads, in steps of 8: what ptxas assigns to a 384-thread,
// one-block-per-SM kernel; the host checks it before the first launch).  The
// producer / MMA warpgroup drops to kFrontRegs and the two epilogue
// warpgroups take the rest -- never more than the launch provided, or the
// increase would wait for registers that never come free.
constexpr int kLaunchRegs = 168;
constexpr int kFrontRegs = 56;
constexpr int kEpilogueRegs = 224;
static_assert(128 * kFrontRegs + 256 * kEpilogueRegs <= kNumThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
static_assert(kNumThreads * kLaunchRegs <= 65536, "one block per SM");

constexpr uint32_t kABytes = kBM * kBK * 2;       // 16 KiB: 128 rows x 128 B
constexpr uint32_t kBChunkCols = 64;              // one 128-byte swizzle span of N
constexpr uint32_t kBChunkBytes = kBK * kBChunkCols * 2;  // 8 KiB: 64 k-rows x 128 B
constexpr uint32_t kBBytes = kBK * kBN * 2;       // 32 KiB
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr uint32_t kStageBufBytes = 32 * 128;     // one epilogue staging box
constexpr int kPrefetchRows = 256;                // K rows per L2-prefetch box of B

// Pipeline depth, TMEM accumulators and epilogue staging.  One CTA per SM: a
// 4-stage ring of 48 KiB stages, two 128 x 256 FP32 accumulators (all 512 TMEM
// columns) so that the epilogue of one tile overlaps the mainloop of the next,
// and eight staging boxes, the sources of the epilogue's TMA stores (fp32: 32
// rows x 128 bytes, 128-byte swizzle; bf16: 32 rows x 64 bytes, 64-byte
// swizzle).  The epilogue warps that have rows split the boxes evenly.
constexpr int kStages = 4;
constexpr int kAccStages = 2;
constexpr int kTmemCols = kAccStages * kBN;
constexpr int kNumBoxes = 8;
constexpr int kMaxBatch = 4;  // 32-column blocks per TMEM load
constexpr int kNumBarriers = 2 * kStages + 2 * kAccStages + 1;
constexpr uint32_t kStagingBytes = kNumBoxes * kStageBufBytes;
// The dynamic shared memory base is 1024-byte aligned (checked at run time).
constexpr uint32_t kSmemBytes = kStages * kStageBytes + kStagingBytes + kNumBarriers * 8 + 16;
static_assert(kSmemBytes <= 232448, "shared memory budget of one sm_103 CTA");

// Epilogue layout for M rows: two warps per TMEM lane quarter with rows
// (ceil(M / 32) quarters, at most 4) share the staging boxes (4, 2 or 1 each);
// each reads `batch` 32-column blocks per TMEM load.
__host__ __device__ constexpr int epi_boxes_for(int M) {
    return kNumBoxes / (2 * ((M + 31) / 32 <= 1 ? 1 : ((M + 31) / 32 == 2 ? 2 : 4)));
}
__host__ __device__ constexpr int epi_batch_for(int M) {
    return epi_boxes_for(M) < kMaxBatch ? epi_boxes_for(M) : kMaxBatch;
}

// B [K, N] row-major is read N-major; the weight layout W [N, K] of a linear
// layer is read K-major, like A.
constexpr uint32_t kIdescBN = idesc_bf16_f32(kBM, kBN, /*A MN-major*/ false, /*B MN-major*/ true);
constexpr uint32_t kIdescWt = idesc_bf16_f32(kBM, kBN, /*A MN-major*/ false, /*B MN-major*/ false);

// Tile widths.  kBN = 256 columns is the default.  A product whose 256-wide
// units would leave most SMs idle (few tiles and few K segments: small N,
// small M, long K) runs with 128- or 64-column tiles instead, so that more
// SMs stream its operands.  Every output element is still formed by the same
// 128-row instructions over the same K blocks in ascending order -- the tile
// width sets only the N extent of each instruction -- and the GPU tests check
// that every width gives the same bits.  A narrower tile has a smaller B
// stage, so the ring holds more stages in the same shared memory: 4 stages of
// 48 KiB (256), 6 of 32 KiB (128), 8 of 24 KiB (64).
template <int kTN>
struct Tile {
    static_assert(kTN == 256 || kTN == 128 || kTN == 64, "tile width");
    static constexpr uint32_t kBBytes = kBK * kTN * 2;
    static constexpr uint32_t kStageBytes = kABytes + kBBytes;
    static constexpr int kStages = static_cast<int>((4u * (kABytes + kBK * kBN * 2)) / kStageBytes);
    static constexpr int kTmemCols = kAccStages * kTN;
    static constexpr int kNumBarriers = 2 * kStages + 2 * kAccStages + 1;
    static constexpr uint32_t kSmemBytes =
        kStages * kStageBytes + kStagingBytes + kNumBarriers * 8 + 16;
    static constexpr int kHalfBlocks = kTN / 64;  // 32-column blocks per epilogue warp
    static constexpr uint32_t kIdescBN = idesc_bf16_f32(kBM, kTN, false, true);
    static constexpr uint32_t kIdescWt = idesc_bf16_f32(kBM, kTN, false, false);
    static_assert(kSmemBytes <= 232448, "shared memory budget of one sm_103 CTA");
    static_assert(kBBytes % 1024 == 0, "B stages on 1024-byte boundaries (128-byte swizzle)");
};
static_assert(Tile<kBN>::kStages == kStages && Tile<kBN>::kSmemBytes == kSmemBytes &&
                  Tile<kBN>::kTmemCols == kTmemCols && Tile<kBN>::kIdescBN == kIdescBN,
              "the default tile width keeps the default layout");

// A wait that gives up: 2 s of global time, checked every 256 polls.
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;

// Bits of the device error word.
constexpr unsigned kErrWaitProducer = 1u;
constexpr unsigned kErrWaitMma = 2u;
constexpr unsigned kErrWaitEpilogue = 4u;
constexpr unsigned kErrWaitDrain = 8u;
constexpr unsigned kErrSmemAlign = 16u;
constexpr unsigned kErrWaitOzakiOrder = 32u;

enum OutKind : int {
    kOutF32 = 0,     // C fp32, plain stores
    kOutBF16 = 1,    // C bf16 (round to nearest even), plain stores
    kOutSlices = 2,  // fp32 split-K partial to workspace slice `seg`
    kOutAtomic = 3,  // fp32 atomic add into C (nondeterministic contrast)
    kOutOzaki = 4,   // binary64 C += 2^e * (slice-pair product), Ozaki scheme
};

struct GemmParams {
    void* out;              // C, or the workspace for kOutSlices
    int64_t ld_out;         // row stride of `out`, elements
    int64_t slice_stride;   // elements between workspace slices (M * ld_out)
    unsigned* status;       // device error word
    int M, N;
    int m_tiles, n_tiles;
    int splits;             // effective number of K segments
    int kb_total;           // ceil(K / kBK)
    int kb_per_split;       // K blocks per segment
    int units;              // m_tiles * n_tiles * splits
    // Epilogue layout, a function of M only (see the epilogue below).
    int epi_boxes;          // staging boxes owned by each epilogue warp with rows
    int epi_batch;          // 32-column blocks read from TMEM and stored together (1, 2 or 4)
    int grouped;            // 1: tmC views the output as {32 columns, rows, column groups
                            //    [, slices]} with boxes of epi_batch groups, one store per batch
    int prefetch_rows;      // K rows of B warmed in L2 before the dependency wait
    int group_m;            // tile rows per GROUP_M swizzle group
    const __nv_bfloat16* bias;  // [N] added to every row by the direct (unsplit)
                                // epilogue, or nullptr
    float scale;            // the direct epilogue multiplies the sum by this (1: none)
    uint32_t idesc_fp8;     // instruction descriptor of the 8-bit float product
    int fold;               // 1: a unit is a whole tile whose `splits` K segments are
                            //    summed in the CTA (splits > 1, direct output)
    int cluster;            // 1: clusters of `splits` CTAs, one per K segment of a tile,
                            //    sum their partials through distributed shared memory
                            //    (splits in 2..8, direct output, one unit per CTA)
    // Ozaki scheme (kOutOzaki): A is `oz_slices` bfloat16 slices of M rows each
    // (slice p at rows p * M), B the same number of slices of oz_kpad rows.
    // The work items are (slice pair, tile) pairs, pair-major: item L is pair
    // L / units of tile L % units, for the pairs (p, q) with p + q < oz_d, and
    // CTA c takes items c, c + grid, ...  A tile's pairs may run on different
    // CTAs; oz_count[tile] (zero at launch) counts the epilogue warps that have
    // added a pair into the tile's C (kEpilogueWarps per pair), and pair k's
    // warps wait until it reaches k * kEpilogueWarps, so every element of C
    // still takes its pairs in order.
    const int* oz_ca;       // c^(1) of every row of A
    const int* oz_cb;       // c^(1) of every column of B
    int* oz_count;          // per tile, then the grid's abort word (oz_count[units])
    int oz_slices, oz_d, oz_beta, oz_pairs, oz_kpad;
    // Fast Mode's automatic d (oz_fast): element (i, j) takes the pairs with
    // p + q < d_ij, d_ij the least d >= 1 with d (beta + 1) >= oz_need0 -
    // bitlen(T_a[i] T_b[j]) (at most oz_slices), T the vectors' integer masses;
    // the kernel enumerates the pairs with p + q < the largest d_ij.
    const unsigned long long* oz_ta;  // mass of every row of A
    const unsigned long long* oz_tb;  // mass of every column of B
    int oz_fast, oz_need0;
    int oz_c32;             // 1: C and its row stride are 32-byte aligned (wide C accesses)
    int selftest_stall;     // 1 (the failure self-test only): the producer issues no
                            //    loads, so the MMA issuer's bounded wait must give up
    int a_rows;             // rows of A each stage loads (32, 64 or 128: the batch
                            //    rounded up); the stage's other rows stay zero
};

// The slice pairs of the Ozaki scheme in the order of the binary64
// accumulation: p outer, q inner, skipping p + q >= d (Fast Mode).
__device__ __forceinline__ void ozaki_next_pair(const GemmParams& p, int d, int& a, int& b) {
    ++b;
    if (b >= p.oz_slices || a + b >= d) {
        ++a;
        b = 0;
    }
}

// Bit length of the 128-bit product x y.
__device__ __forceinline__ int ozaki_bitlen_product(unsigned long long x, unsigned long long y) {
    const unsigned long long hi = __umul64hi(x, y), lo = x * y;
    if (hi != 0) return 128 - __clzll(static_cast<long long>(hi));
    return lo != 0 ? 64 - __clzll(static_cast<long long>(lo)) : 0;
}

// Fast Mode's d for masses (tx, ty): the least d >= 1 with d (beta + 1) >=
// need0 - bitlen(tx ty), at most the slice count.
__device__ __forceinline__ int ozaki_fast_d(const GemmParams& p, unsigned long long tx,
                                            unsigned long long ty) {
    const int need = p.oz_need0 - ozaki_bitlen_product(tx, ty), w = p.oz_beta + 1;
    const int d = need <= w ? 1 : (need + w - 1) / w;
    return d < p.oz_slices ? d : p.oz_slices;
}

// Unit u -> (tile row, tile column, K segment).  All tiles of segment 0 come
// first, then segment 1, ...; inside a segment the tiles follow the GROUP_M
// swizzle: groups of p.group_m tile rows, column-major inside a group.  With
// clusters the segments of one tile are consecutive instead (a cluster is
// consecutive CTAs).  The order decides only which CTA computes a tile, never
// how a sum is formed.
__device__ __forceinline__ void unit_coords(const GemmParams& p, int u, int& mt, int& nt,
                                            int& seg) {
    const int tiles = p.m_tiles * p.n_tiles;
    int tile;
    if (p.cluster) {
        tile = u / p.splits;
        seg = u - tile * p.splits;
    } else {
        seg = u / tiles;
        tile = u - seg * tiles;
    }
    const int per_group = p.group_m * p.n_tiles;
    const int g = tile / per_group;
    const int first_m = g * p.group_m;
    const int gm = min(p.m_tiles - first_m, p.group_m);
    const int r = tile - g * per_group;
    mt = first_m + r % gm;
    nt = r / gm;
}

// The scheduling parameters the producer thread needs, read from the kernel
// parameters in one batch: each first read of a parameter line misses the
// constant cache (the parameters are new at every launch), and read one after
// another as they are needed these misses lay end to end on the way to every
// CTA's first load.
struct Sched {
    int units, m_tiles, n_tiles, group_m, splits, cluster;
    int fold, kb_total, kb_per_split, prefetch_rows, a_rows, selftest_stall;
};

__device__ __forceinline__ Sched load_sched(const GemmParams& p) {
    Sched s;
    s.units = p.units;
    s.m_tiles = p.m_tiles;
    s.n_tiles = p.n_tiles;
    s.group_m = p.group_m;
    s.splits = p.splits;
    s.cluster = p.cluster;
    s.fold = p.fold;
    s.kb_total = p.kb_total;
    s.kb_per_split = p.kb_per_split;
    s.prefetch_rows = p.prefetch_rows;
    s.a_rows = p.a_rows;
    s.selftest_stall = p.selftest_stall;
    // all twelve values arrive together here
    asm volatile("" ::"r"(s.units), "r"(s.m_tiles), "r"(s.n_tiles), "r"(s.group_m), "r"(s.splits),
                 "r"(s.cluster), "r"(s.fold), "r"(s.kb_total), "r"(s.kb_per_split), "r"(s.prefetch_rows),
                 "r"(s.a_rows), "r"(s.selftest_stall));
    return s;
}

// unit_coords on the preloaded values (the same mapping).
__device__ __forceinline__ void unit_coords(const Sched& p, int u, int& mt, int& nt, int& seg) {
    const int tiles = p.m_tiles * p.n_tiles;
    int tile;
    if (p.cluster) {
        tile = u / p.splits;
        seg = u - tile * p.splits;
    } else {
        seg = u / tiles;
        tile = u - seg * tiles;
    }
    const int per_group = p.group_m * p.n_tiles;
    const int g = tile / per_group;
    const int first_m = g * p.group_m;
    const int gm = min(p.m_tiles - first_m, p.group_m);
    const int r = tile - g * per_group;
    mt = first_m + r % gm;
    nt = r / gm;
}

// Bounded wait on an mbarrier phase.  Gives up when another role has aborted
// (shared flag) or after kWaitTimeoutNs; a timeout raises the abort flag and
// records `why` in the device error word.  Never traps.
// kCluster: acquire at cluster scope (a barrier the other CTA of a pair
// arrives on).
template <bool kCluster = false>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity,
                                             volatile int* abort_flag, unsigned* status,
                                             unsigned why, bool honour_abort = true) {
    const auto done = [&]() {
        return kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
    };
    if (done()) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1; it != 0u; ++it) {
        if (done()) return true;
        if ((it & 255u) == 0u) {
            if (honour_abort && *abort_flag) return false;
            if (global_timer_ns() - t0 > kWaitTimeoutNs) break;
        }
    }
    *abort_flag = 1;
    atomicOr(status, why);
    return false;
}

// Bounded wait until *count >= want (an acquire load per poll).  Gives up
// like wait_bounded: when another role of this CTA has aborted, when another
// CTA of the grid has given up (*grid_abort, a word of the launch's
// workspace, zero at launch), or after kWaitTimeoutNs; a timeout raises the
// CTA's abort flag, the grid's abort word and the error bit, so that the
// CTAs waiting behind this one stop at once instead of each running out its
// own time.
__device__ __forceinline__ bool wait_count_bounded(const int* count, int want, volatile int* abort_flag,
                                                   int* grid_abort, unsigned* status) {
    if (ld_acquire_gpu(count) >= want) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1; it != 0u; ++it) {
        if (ld_acquire_gpu(count) >= want) return true;
        if ((it & 63u) == 0u) {
            if (*abort_flag || *reinterpret_cast<volatile int*>(grid_abort)) {
                *abort_flag = 1;
                return false;
            }
            if (global_timer_ns() - t0 > kWaitTimeoutNs) break;
        }
    }
    *abort_flag = 1;
    atomicExch(grid_abort, 1);
    atomicOr(status, kErrWaitOzakiOrder);
    return false;
}

// Thread `lane` holds row `lane` of a 32 x 32 fp32 block (32 registers).  The
// staging writers put it into a shared-memory box in the layout the TMA store
// expects: fp32 rows of 128 bytes whose 16-byte chunks are permuted by the
// 128-byte swizzle (chunk j of row r at j ^ (r % 8)); bf16 rows of 64 bytes
// with the 64-byte swizzle (chunk j of row r at j ^ ((r / 2) % 4)).  Both
// permutations also spread a quarter-warp's 16-byte stores over all banks.
__device__ __forceinline__ void stage_f32(uint32_t buf, int lane, const uint32_t (&r)[32]) {
    const uint32_t row = buf + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
    for (int j = 0; j < 8; ++j)
        st_shared_v4(row + ((static_cast<uint32_t>(j) ^ (lane & 7)) << 4), r[4 * j], r[4 * j + 1],
                     r[4 * j + 2], r[4 * j + 3]);
}

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo, uint32_t hi) {
    __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(lo), __uint_as_float(hi));
    return *reinterpret_cast<uint32_t*>(&b2);
}

__device__ __forceinline__ void stage_bf16(uint32_t buf, int lane, const uint32_t (&r)[32]) {
    const uint32_t row = buf + static_cast<uint32_t>(lane) * 64u;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        st_shared_v4(row + ((static_cast<uint32_t>(j) ^ ((lane >> 1) & 3)) << 4),
                     pack_bf16x2(r[8 * j], r[8 * j + 1]), pack_bf16x2(r[8 * j + 2], r[8 * j + 3]),
                     pack_bf16x2(r[8 * j + 4], r[8 * j + 5]), pack_bf16x2(r[8 * j + 6], r[8 * j + 7]));
}

// A row's 32 values stored element by element, columns >= N skipped.
template <int kOut>
__device__ __forceinline__ void store_row_masked(const GemmParams& p, int row, int col,
                                                 const uint32_t (&r)[32]) {
    const int valid = min(32, p.N - col);
    if constexpr (kOut == kOutBF16) {
        __nv_bfloat16* dst =
            static_cast<__nv_bfloat16*>(p.out) + static_cast<int64_t>(row) * p.ld_out + col;
#pragma unroll
        for (int c = 0; c < 32; ++c)
            if (c < valid) dst[c] = __float2bfloat16_rn(__uint_as_float(r[c]));
    } else {
        float* dst = static_cast<float*>(p.out) + static_cast<int64_t>(row) * p.ld_out + col;
#pragma unroll
        for (int c = 0; c < 32; ++c)
            if (c < valid) dst[c] = __uint_as_float(r[c]);
    }
}

// Adds bias[col .. col+31] (bf16, every lane the same values) to a thread's
// 32 FP32 accumulators, one FP32 addition each, rounded to nearest even.
// Columns >= N are left alone.
__device__ __forceinline__ void add_bias_block(const __nv_bfloat16* bias, int col, int N,
                                               uint32_t* r) {
    if (col + 32 <= N) {
        const uint4* b4 = reinterpret_cast<const uint4*>(bias + col);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const uint4 w = __ldg(b4 + v);
            const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                // a bf16 value is the upper half of the FP32 with the same value
                const float lo = __uint_as_float(wv[h] << 16);
                const float hi = __uint_as_float(wv[h] & 0xFFFF0000u);
                r[8 * v + 2 * h] = __float_as_uint(__fadd_rn(__uint_as_float(r[8 * v + 2 * h]), lo));
                r[8 * v + 2 * h + 1] =
                    __float_as_uint(__fadd_rn(__uint_as_float(r[8 * v + 2 * h + 1]), hi));
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (col + j < N)
                r[j] = __float_as_uint(__fadd_rn(__uint_as_float(r[j]), __bfloat162float(bias[col + j])));
    }
}

// The atomic contrast: every thread adds its row's 32 values into C.
__device__ __forceinline__ void atomic_add_row_chunk(const GemmParams& p, int row, int col,
                                                     const uint32_t (&r)[32]) {
    const int valid = min(32, p.N - col);
    float* dst = static_cast<float*>(p.out) + static_cast<int64_t>(row) * p.ld_out + col;
#pragma unroll
    for (int c = 0; c < 32; ++c)
        if (c < valid) atomicAdd(dst + c, __uint_as_float(r[c]));
}

// The epilogue's last step for nb (<= kNbMax) 32-column blocks of one warp's
// 32 rows, held in r: the output scale and the bias (direct outputs), then
// either the atomic additions of the contrast or swizzled staging boxes and
// their TMA stores.  Blocks ending in a partial 16-byte chunk of a C row are
// written element by element instead (the TMA unit clips the innermost
// dimension at 16-byte granularity; the workspace owns its padding).  `nbat`
// counts the batches this warp has handed to the TMA unit; the slot a batch
// reuses must have been read by its earlier store, so at most slots - 1 may
// pend.
template <int kOut, int kNbMax>
__device__ __forceinline__ void emit_blocks(const GemmParams& p, const CUtensorMap* tmC, uint32_t* r,
                                            int nb, int c0, int n0, int m0, int seg, int lane,
                                            uint32_t my_boxes, int batch, int slots, uint32_t& nbat) {
    constexpr uint32_t kBox = (kOut == kOutBF16) ? kStageBufBytes / 2 : kStageBufBytes;
    if constexpr (kOut == kOutF32 || kOut == kOutBF16) {
        if (p.scale != 1.0f) {  // uniform: one FP32 multiply per element
#pragma unroll
            for (int i = 0; i < kNbMax * 32; ++i)
                if (i < nb * 32) r[i] = __float_as_uint(__fmul_rn(__uint_as_float(r[i]), p.scale));
        }
        if (p.bias != nullptr) {  // uniform
#pragma unroll
            for (int i = 0; i < kNbMax; ++i)
                if (i < nb) add_bias_block(p.bias, n0 + (c0 + i) * 32, p.N, r + 32 * i);
        }
    }
    if constexpr (kOut == kOutAtomic) {
#pragma unroll
        for (int i = 0; i < kNbMax; ++i)
            if (i < nb && m0 + lane < p.M)
                atomic_add_row_chunk(p, m0 + lane, n0 + (c0 + i) * 32,
                                     *reinterpret_cast<const uint32_t(*)[32]>(r + 32 * i));
    } else {
        const uint32_t box0 = my_boxes + (nbat % static_cast<uint32_t>(slots)) * batch * kBox;
        if (nbat >= static_cast<uint32_t>(slots)) {
            if (lane == 0) bulk_wait_group_read_dyn(slots - 1);
            __syncwarp();
        }
        constexpr int kVec = (kOut == kOutBF16) ? 8 : 4;
        int staged = 0;
#pragma unroll
        for (int i = 0; i < kNbMax; ++i) {
            if (i >= nb) break;
            const int col = n0 + (c0 + i) * 32;
            const uint32_t(&ri)[32] = *reinterpret_cast<const uint32_t(*)[32]>(r + 32 * i);
            const bool ragged = kOut != kOutSlices && col + 32 > p.N && (p.N % kVec) != 0;
            if (ragged) {
                if (m0 + lane < p.M) store_row_masked<kOut>(p, m0 + lane, col, ri);
            } else {
                const uint32_t box = box0 + static_cast<uint32_t>(i) * kBox;
                if constexpr (kOut == kOutBF16) stage_bf16(box, lane, ri);
                else stage_f32(box, lane, ri);
                ++staged;
            }
        }
        if (staged > 0) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                const int g0 = (n0 + c0 * 32) / 32;
                if (p.grouped) {
                    if constexpr (kOut == kOutSlices) tma_store_4d(tmC, box0, 0, m0, g0, seg);
                    else tma_store_3d(tmC, box0, 0, m0, g0);
                } else {
                    for (int i = 0; i < staged; ++i) {
                        const uint32_t box = box0 + static_cast<uint32_t>(i) * kBox;
                        const int col = n0 + (c0 + i) * 32;
                        if constexpr (kOut == kOutSlices) tma_store_3d(tmC, box, col, m0, seg);
                        else tma_store_2d(tmC, box, col, m0);
                    }
                }
                bulk_commit_group();
            }
            ++nbat;
        }
    }
}

// The in-cluster split-K sum of one tile.  CTA rank s of the cluster holds
// the FP32 partial of K segment s (layout: row r at r * 1 KiB, 16-byte chunk c
// at c ^ (r % 8)).  The tile's valid rows x 64 chunks are dealt to the ranks
// in equal contiguous shares; for each chunk: acc = w_0, then acc = acc + w_s
// for s = 1 .. splits-1 (FP32, round to nearest even), then acc * scale and
// acc + bias -- splitk_reduce_kernel's arithmetic in its order, so the bits
// equal the workspace path's.  `e` is the thread's index among the 256
// epilogue threads.
template <int kOut>
__device__ __forceinline__ void cluster_reduce(const GemmParams& p, uint32_t part_base, int e) {
    int mt, nt, seg;
    unit_coords(p, blockIdx.x, mt, nt, seg);
    const int m0 = mt * kBM, n0 = nt * kBN;
    const int rows = min(kBM, p.M - m0);
    const int items = rows * (kBN / 4);
    const int S = p.splits;
    const int per = (items + S - 1) / S;
    const int lo = static_cast<int>(cluster_ctarank()) * per;
    const int hi = min(items, lo + per);
    uint32_t src[8];
#pragma unroll
    for (int s = 0; s < 8; ++s) src[s] = s < S ? map_shared_rank(part_base, static_cast<uint32_t>(s)) : 0u;
    for (int v = lo + e; v < hi; v += kEpilogueThreads) {
        const int row = v >> 6, c = v & 63;
        const int col = n0 + c * 4;
        if (col >= p.N) continue;
        const uint32_t off = static_cast<uint32_t>(row) * 1024u +
                             ((static_cast<uint32_t>(c) ^ (static_cast<uint32_t>(row) & 7u)) << 4);
        float4 w[8];
#pragma unroll
        for (int s = 0; s < 8; ++s)
            if (s < S) w[s] = ld_shared_cluster_f32x4(src[s] + off);
        float4 acc = w[0];
#pragma unroll
        for (int s = 1; s < 8; ++s) {
            if (s < S) {
                acc.x = __fadd_rn(acc.x, w[s].x);
                acc.y = __fadd_rn(acc.y, w[s].y);
                acc.z = __fadd_rn(acc.z, w[s].z);
                acc.w = __fadd_rn(acc.w, w[s].w);
            }
        }
        const int valid = min(4, p.N - col);
        if (p.scale != 1.0f) {
            acc.x = __fmul_rn(acc.x, p.scale);
            acc.y = __fmul_rn(acc.y, p.scale);
            acc.z = __fmul_rn(acc.z, p.scale);
            acc.w = __fmul_rn(acc.w, p.scale);
        }
        if (p.bias != nullptr) {
            float* a = &acc.x;
            for (int k = 0; k < valid; ++k) a[k] = __fadd_rn(a[k], __bfloat162float(p.bias[col + k]));
        }
        const int64_t grow = m0 + row;
        if constexpr (kOut == kOutBF16) {
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + grow * p.ld_out + col;
            if (valid == 4) {
                __nv_bfloat162 lo2 = __floats2bfloat162_rn(acc.x, acc.y);
                __nv_bfloat162 hi2 = __floats2bfloat162_rn(acc.z, acc.w);
                *reinterpret_cast<uint2*>(dst) =
                    make_uint2(*reinterpret_cast<uint32_t*>(&lo2), *reinterpret_cast<uint32_t*>(&hi2));
            } else {
                const float a[4] = {acc.x, acc.y, acc.z, acc.w};
                for (int k = 0; k < valid; ++k) dst[k] = __float2bfloat16_rn(a[k]);
            }
        } else {
            float* dst = static_cast<float*>(p.out) + grow * p.ld_out + col;
            if (valid == 4) {
                *reinterpret_cast<float4*>(dst) = acc;
            } else {
                const float a[4] = {acc.x, acc.y, acc.z, acc.w};
                for (int k = 0; k < valid; ++k) dst[k] = a[k];
            }
        }
    }
}

// One step of the Ozaki scheme's binary64 sum for 32 columns of one row:
// c[j] = c[j] + 2^(e_pair + cb[j]) * P[j], P[j] the FP32 slice-pair product
// (an exact integer multiple of its unit, so the scaling by a power of two
// is exact and one rounding remains: a fused multiply-add with the power of
// two is that addition).  first: the sum starts here from +0.0 and C is not
// read.  valid < 32 at the right edge of C.
__device__ __forceinline__ double ozaki_term(double c, uint32_t pbits, int e) {
    const double P = static_cast<double>(__uint_as_float(pbits));
    if (e >= -1022 && e <= 1023)
        return __fma_rn(P, __longlong_as_double(static_cast<long long>(e + 1023) << 52), c);
    return __dadd_rn(c, ldexp(P, e));
}

// 2^e * P for the bit pattern of a binary32 P that is zero or normal, with
// e + exponent(P) inside the normal binary64 range: sign kept, exponent
// moved by e and rebiased, the 23 fraction bits widened to 52.
__device__ __forceinline__ double ozaki_scaled(uint32_t pbits, int e) {
    const uint32_t mag = pbits & 0x7FFFFFFFu;
    const uint64_t bits = (static_cast<uint64_t>(pbits >> 31) << 63) |
                          (static_cast<uint64_t>(static_cast<int>(mag >> 23) - 127 + e + 1023) << 52) |
                          (static_cast<uint64_t>(mag & 0x7FFFFFu) << 29);
    return mag != 0u ? __longlong_as_double(static_cast<long long>(bits)) : 0.0;
}

// Fast Mode's per-element choice (fast.tb not NULL): element j takes the
// pair iff t == 0 or t (beta + 1) < need0 - bitlen(ta tb[j]) (t = p + q),
// i.e. iff p + q < its d; an element that does not keep C unchanged (no
// addition of zero, which would turn -0.0 into +0.0).  For t > 0 and
// E = need0 - t (beta + 1) - 1 >= 0 the test is ta tb[j] < 2^E, i.e. (for
// ta > 0) tb[j] <= lim = floor((2^E - 1) / ta): one comparison per element
// against a limit the row computes once per pair.
struct OzakiFastRow {
    const unsigned long long* tb;  // masses of the block's columns, or NULL: every element
    unsigned long long lim;        // the largest column mass that takes the pair
    bool none;                     // no element of the row takes it
};

// The row's limit for diagonal t of the pairs (tw = t (beta + 1)): none
// passes when E < 0; every column mass passes (lim = 2^64 - 1) when t == 0,
// ta == 0 or 2^E / ta >= 2^64; otherwise floor((2^E - 1) / ta) by restoring
// division, starting after the bits of 2^E - 1 that stay below ta (at most
// 64 steps).
__device__ __forceinline__ OzakiFastRow ozaki_fast_row(const unsigned long long* tb,
                                                       unsigned long long ta, int tw, int need0) {
    OzakiFastRow f;
    f.tb = tb;
    f.lim = ~0ull;
    f.none = false;
    if (tb == nullptr || tw == 0) return f;
    const int E = need0 - tw - 1;
    if (E < 0) {  // bitlen(ta tb) < 0: never
        f.none = true;
        return f;
    }
    if (ta == 0) return f;  // a zero product: bitlen 0 <= E
    const int la = 64 - __clzll(static_cast<long long>(ta));
    if (E - la >= 64) return f;  // ta tb < 2^(la + 64) <= 2^E for every tb
    if (E < la - 1) {            // 2^E - 1 < ta: only a zero mass
        f.lim = 0;
        return f;
    }
    // 2^E - 1 is E one bits; its first la - 1 leave a remainder 2^(la-1) - 1 < ta
    unsigned long long rem = (la == 64) ? 0x7FFFFFFFFFFFFFFFull : ((1ull << (la - 1)) - 1);
    unsigned long long q = 0;
    for (int pos = E - la; pos >= 0; --pos) {
        const bool carry = (rem >> 63) != 0;
        const unsigned long long r2 = (rem << 1) | 1ull;
        if (carry || r2 >= ta) {
            rem = r2 - ta;  // the true difference is below ta < 2^64
            q |= 1ull << pos;
        } else {
            rem = r2;
        }
    }
    f.lim = q;
    return f;
}

__device__ __forceinline__ bool ozaki_takes(const OzakiFastRow& f, int j) {
    if (f.tb == nullptr) return true;
    return !f.none && __ldg(f.tb + j) <= f.lim;
}

__device__ __forceinline__ void ozaki_accumulate_block(double* crow, const int* cb, int valid,
                                                       int e_pair, const uint32_t (&r)[32],
                                                       bool first, const OzakiFastRow& fast, bool c32) {
    if (valid == 32) {
        // all loads first (C and the column exponents), then the arithmetic,
        // then the stores: 32 independent memory operations in flight
        int e[32];
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
            const int4 v = __ldg(reinterpret_cast<const int4*>(cb + j));
            e[j] = e_pair + v.x;
            e[j + 1] = e_pair + v.y;
            e[j + 2] = e_pair + v.z;
            e[j + 3] = e_pair + v.w;
        }
        double2 c[16];
        if (first) {
#pragma unroll
            for (int j = 0; j < 16; ++j) c[j] = make_double2(0.0, 0.0);
        } else if (c32) {
            // 32 bytes per lane and instruction: a whole sector, half the
            // instructions (each lane's row is another line)
#pragma unroll
            for (int j = 0; j < 8; ++j)
                ld_global_v4f64(crow + 4 * j, c[2 * j].x, c[2 * j].y, c[2 * j + 1].x, c[2 * j + 1].y);
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) c[j] = *reinterpret_cast<const double2*>(crow + 2 * j);
        }
        int lo = e[0], hi = e[0];
#pragma unroll
        for (int j = 1; j < 32; ++j) {
            lo = min(lo, e[j]);
            hi = max(hi, e[j]);
        }
        if (lo >= -1006 && hi <= 1001) {
            // P is a nonzero multiple of 2^-16 below 2^24, or zero, so 2^e P is a
            // normal binary64 for e in this range: build it from P's bits
            // (exponent rebiased, fraction widened) -- exact, integer work only
            // -- and spend one binary64 addition per element.
            if (fast.tb == nullptr || fast.lim == ~0ull) {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    c[j].x = __dadd_rn(c[j].x, ozaki_scaled(r[2 * j], e[2 * j]));
                    c[j].y = __dadd_rn(c[j].y, ozaki_scaled(r[2 * j + 1], e[2 * j + 1]));
                }
            } else if (!fast.none) {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const ulonglong2 t = __ldg(reinterpret_cast<const ulonglong2*>(fast.tb) + j);
                    if (t.x <= fast.lim) c[j].x = __dadd_rn(c[j].x, ozaki_scaled(r[2 * j], e[2 * j]));
                    if (t.y <= fast.lim) c[j].y = __dadd_rn(c[j].y, ozaki_scaled(r[2 * j + 1], e[2 * j + 1]));
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                if (ozaki_takes(fast, 2 * j)) c[j].x = ozaki_term(c[j].x, r[2 * j], e[2 * j]);
                if (ozaki_takes(fast, 2 * j + 1)) c[j].y = ozaki_term(c[j].y, r[2 * j + 1], e[2 * j + 1]);
            }
        }
        if (c32) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                st_global_v4f64(crow + 4 * j, c[2 * j].x, c[2 * j].y, c[2 * j + 1].x, c[2 * j + 1].y);
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) *reinterpret_cast<double2*>(crow + 2 * j) = c[j];
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (j < valid && ozaki_takes(fast, j))
                crow[j] = ozaki_term(first ? 0.0 : crow[j], r[j], e_pair + __ldg(cb + j));
    }
}

// C rows at least this many elements apart take the staged form below: at
// 8192^3 (rows 64 KiB apart) it took 31.9 against 33.7 ms; at 4096^3 (32
// KiB) it was no faster and read 17.3 against 9.6 GB from DRAM, so narrower
// rows keep the direct per-lane accesses.
constexpr int64_t kOzStagedMinLd = 8192;

// ozaki_accumulate_block for a warp's full 32 x 32 block (32 columns inside
// N), with the loads and stores of C coalesced through the warp's 4 KiB of
// shared memory: per half of 16 columns, the warp reads the block's rows four
// at a time (8 lanes x 16 bytes per row: 512 contiguous-per-row bytes per
// instruction) into buf, each lane then takes its own row from buf (16-byte
// chunk c of row i at chunk c ^ (i % 8): no bank conflict), adds exactly as
// ozaki_accumulate_block does, puts the row back, and the warp writes the
// rows out four at a time.  rows: the block's rows inside C (lanes past it
// compute but nothing of theirs is read or written).  Every lane calls it.
__device__ __forceinline__ void ozaki_accumulate_block_staged(double* crow0, int64_t ldc, int rows, const int* cb,
                                                              int e_pair, const uint32_t (&r)[32], bool first,
                                                              const OzakiFastRow& fast, double* buf, int lane) {
    const int quarter = lane >> 3, chunk = lane & 7;
    const auto slot = [](int i, int c) { return i * 16 + ((c ^ (i & 7)) << 1); };  // chunk c of row i
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {  // unrolled: r is indexed by constants
        double* const ch = crow0 + hb * 16;
        if (!first) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int i = 4 * k + quarter;
                const double2 v = i < rows ? *reinterpret_cast<const double2*>(ch + static_cast<int64_t>(i) * ldc + 2 * chunk)
                                           : make_double2(0.0, 0.0);
                *reinterpret_cast<double2*>(buf + slot(i, chunk)) = v;
            }
            __syncwarp();
        }
        int e[16];
#pragma unroll
        for (int j = 0; j < 16; j += 4) {
            const int4 v = __ldg(reinterpret_cast<const int4*>(cb + hb * 16 + j));
            e[j] = e_pair + v.x;
            e[j + 1] = e_pair + v.y;
            e[j + 2] = e_pair + v.z;
            e[j + 3] = e_pair + v.w;
        }
        double c[16];
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
            if (first) {
                c[j] = 0.0;
                c[j + 1] = 0.0;
            } else {
                const double2 v = *reinterpret_cast<const double2*>(buf + slot(lane, j >> 1));
                c[j] = v.x;
                c[j + 1] = v.y;
            }
        }
        int lo = e[0], hi = e[0];
#pragma unroll
        for (int j = 1; j < 16; ++j) {
            lo = min(lo, e[j]);
            hi = max(hi, e[j]);
        }
        // the per-element choice of ozaki_accumulate_block (Fast Mode: the
        // column masses from hb * 16; an element that does not take the pair
        // keeps its C)
        const bool all = fast.tb == nullptr || fast.lim == ~0ull;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const uint32_t pbits = r[hb * 16 + j];
            bool takes = all;
            if (!all) takes = !fast.none && __ldg(fast.tb + hb * 16 + j) <= fast.lim;
            if (takes)
                c[j] = (lo >= -1006 && hi <= 1001) ? __dadd_rn(c[j], ozaki_scaled(pbits, e[j]))
                                                   : ozaki_term(c[j], pbits, e[j]);
        }
#pragma unroll
        for (int j = 0; j < 16; j += 2)
            *reinterpret_cast<double2*>(buf + slot(lane, j >> 1)) = make_double2(c[j], c[j + 1]);
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int i = 4 * k + quarter;
            if (i < rows)
                *reinterpret_cast<double2*>(ch + static_cast<int64_t>(i) * ldc + 2 * chunk) =
                    *reinterpret_cast<const double2*>(buf + slot(i, chunk));
        }
        __syncwarp();  // buf is refilled by the next half
    }
}

// kWt: the second operand is the weight matrix W [N, K] (K-major); otherwise
// B [K, N] (N-major).  Both products run the same K = 16 instruction sequence.
// kFp8: 8-bit float operands (both K-major, kWt): a K block is 128 elements,
// still 128 bytes per row, consumed by four tcgen05.mma.kind::f8f6f4 of K = 32;
// the shared-memory layout and descriptors are byte for byte those of BF16.
template <int kOut, bool kWt, bool kFp8, int kTN = kBN>
__global__ void __launch_bounds__(kNumThreads, 1)
    bigemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmBp, const __grid_constant__ CUtensorMap tmC,
                     const GemmParams p) {
    static_assert(!kFp8 || kWt, "8-bit operands are read K-major only");
    static_assert(kTN == kBN || (!kFp8 && kOut != kOutOzaki),
                  "narrow tiles serve the bf16 products only");
    // this tile width's ring, accumulators and barriers
    using TileT = Tile<kTN>;
    constexpr int kRing = TileT::kStages;
    constexpr uint32_t kRingB = TileT::kBBytes;
    constexpr uint32_t kRingStage = TileT::kStageBytes;
    constexpr int kBars = TileT::kNumBarriers;
    constexpr int kHB = TileT::kHalfBlocks;
    constexpr int kKB = kFp8 ? 128 : kBK;  // elements per K block (128 bytes per row)
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 128-byte-swizzled tiles must start on 1024-byte boundaries; the layout
    // below assumes the base is.  Should it not be, stop before touching
    // anything (no barrier, no TMEM yet) and report it.
    const uint32_t base = smem_addr(smem_raw);
    if (base & 1023u) {
        if (threadIdx.x == 0) atomicOr(p.status, kErrSmemAlign);
        return;
    }
    uint8_t* gbase = smem_raw;
    const uint32_t sA = base;                                // stage s: sA + s * kABytes
    const uint32_t sB = base + kRing * kABytes;              // stage s: sB + s * kRingB
    const uint32_t sOut = base + kRing * kRingStage;         // epilogue staging boxes
    uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + kRing * kRingStage + kStagingBytes);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const uint32_t bar0 = smem_addr(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kRing + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * kRing + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * kRing + kAccStages + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * kRing + 2 * kAccStages);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (warp == 2 && lane == 0) {
        for (int s = 0; s < kRing; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < kAccStages; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), kEpilogueThreads);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    // The coordinates of this CTA's first unit, found by the producer thread
    // while the previous kernel in the stream finishes and reused for its first
    // loads (working them out after the dependency wait put some 0.5 us between
    // the wait and the first load of every CTA).
    int first_mt = 0, first_nt = 0, first_seg = 0;
    Sched sc{};
    if (warp == 0 && lane == 0) {
        sc = load_sched(p);
        // Warm L2 with the weights of this CTA's first unit (its first
        // p.prefetch_rows K rows) while the previous kernel in the stream
        // finishes.  An L2 prefetch writes no shared memory and L2 is the
        // device's point of coherence, so it cannot expose data older than the
        // dependency wait below.
        tma_prefetch_desc(&tmBp);
        if (static_cast<int>(blockIdx.x) < sc.units) {
            unit_coords(sc, blockIdx.x, first_mt, first_nt, first_seg);
            const int nt = first_nt, seg = first_seg;
            const int k0 = seg * sc.kb_per_split * kKB;
            const int seg_rows = (sc.fold ? sc.kb_total : sc.kb_per_split) * kKB;
            const int k1 = min(k0 + sc.prefetch_rows, min(k0 + seg_rows, sc.kb_total * kKB));
            for (int k = k0; k < k1; k += kPrefetchRows) {
                if constexpr (kWt) tma_prefetch_l2_2d(&tmBp, k, nt * kTN);
                else tma_prefetch_l2_2d(&tmBp, nt * kTN, k);
            }
            // and the tile's bias values, which the epilogue adds (one line
            // per 64 columns, none past N)
            if constexpr (kOut == kOutF32 || kOut == kOutBF16) {
                if (p.bias != nullptr)
                    for (int c = nt * kTN; c < min(nt * kTN + kTN, p.N); c += 64) prefetch_l2(p.bias + c);
            }
        }
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if constexpr (kOut != kOutAtomic && kOut != kOutOzaki) tma_prefetch_desc(&tmC);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), TileT::kTmemCols);
        tmem_relinquish();
    }
    if (p.a_rows < kBM) {
        // A short batch loads only its first a_rows rows of A per stage; the
        // MMA still reads all 128 (one instruction shape for every M), so the
        // rest of every A stage is zeroed once here and never written again.
        // Those rows feed only output rows >= M, which are never stored.
        // (by the epilogue warps, idle until the first tile is done, so that
        // the producer thread's prologue stays short)
        const uint32_t tail = static_cast<uint32_t>(p.a_rows) * 128u;
        const uint32_t per_stage = (kABytes - tail) / 16u;
        for (uint32_t i = threadIdx.x - kEpilogueWarp0 * 32; threadIdx.x >= kEpilogueWarp0 * 32 &&
                                                          i < kRing * per_stage;
             i += kEpilogueThreads) {
            const uint32_t s_ = i / per_stage, c = i - s_ * per_stage;
            st_shared_v4(sA + s_ * kABytes + tail + c * 16u, 0u, 0u, 0u, 0u);
        }
        if (threadIdx.x >= kEpilogueWarp0 * 32)
            fence_proxy_async_smem();  // visible to the tensor core's (async-proxy) reads
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    // Everything above overlaps the previous kernel in the stream; from here on
    // global memory is read and written only after it has completed.
    grid_dependency_wait();

    // The slice pairs this product enumerates: p + q < oz_d.  With Fast Mode's
    // automatic d, oz_d is the largest per-element d of the product, that of
    // the least row mass and the least column mass (d_ij falls as the masses
    // grow), found by every CTA from the split kernels' masses.
    int oz_d = 0, oz_pairs = 0;
    if constexpr (kOut == kOutOzaki) {
        oz_d = p.oz_d;
        oz_pairs = p.oz_pairs;
        if (p.oz_fast) {
            __shared__ unsigned long long oz_min[2];
            if (threadIdx.x == 0) {
                oz_min[0] = ~0ull;
                oz_min[1] = ~0ull;
            }
            __syncthreads();
            unsigned long long ma = ~0ull, mb = ~0ull;
            for (int i = threadIdx.x; i < p.M; i += kNumThreads) ma = min(ma, p.oz_ta[i]);
            for (int j = threadIdx.x; j < p.N; j += kNumThreads) mb = min(mb, p.oz_tb[j]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                ma = min(ma, __shfl_xor_sync(0xffffffffu, ma, o));
                mb = min(mb, __shfl_xor_sync(0xffffffffu, mb, o));
            }
            if (lane == 0) {
                atomicMin(&oz_min[0], ma);
                atomicMin(&oz_min[1], mb);
            }
            __syncthreads();
            oz_d = ozaki_fast_d(p, oz_min[0], oz_min[1]);
            oz_pairs = 0;
            for (int a = 0; a < p.oz_slices; ++a) oz_pairs += max(0, min(p.oz_slices, oz_d - a));
        }
    }

    // Only the direct-output epilogues (the folded running sum) and the Ozaki
    // epilogue need more than the launch's 168 registers per thread; the
    // others skip the re-division (it sits between the dependency wait and
    // the first load).
    constexpr bool kSplitRegs = (kOut == kOutF32 || kOut == kOutBF16 || kOut == kOutOzaki);
    if (warp < kEpilogueWarp0) {
      if constexpr (kSplitRegs) regs_release_to<kFrontRegs>();
      if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer --
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued_mask = 0, issued_parity = 0;
            bool ok = !sc.selftest_stall;  // the failure self-test issues nothing
            if constexpr (kOut == kOutOzaki) {
                // Items pair-major: all CTAs work on the same one or two slice
                // pairs at a time and share their A and B panels in L2.  Per
                // item: rows pa * M + m0 of the A slices, rows pb * oz_kpad + k
                // of the B slices.
                int pa = 0, pb = 0, pk = 0;  // pair pk is (pa, pb)
                const int items = p.units * oz_pairs;
                for (int L = blockIdx.x; ok && L < items; L += gridDim.x) {
                    const int pair = L / p.units, u = L - pair * p.units;
                    for (; pk < pair; ++pk) ozaki_next_pair(p, oz_d, pa, pb);
                    {
                        int mt, nt, seg;
                        unit_coords(p, u, mt, nt, seg);
                        const int n0 = nt * kBN;
                        const int a_row = mt * kBM + pa * p.M;
                        const int b_row = pb * p.oz_kpad;
                        for (int kb = 0; kb < p.kb_total; ++kb) {
                            if (!wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, p.status,
                                              kErrWaitProducer)) {
                                ok = false;
                                break;
                            }
                            const uint32_t fb = full_bar(stage);
                            mbar_arrive_expect_tx(fb, kRingStage);
                            tma_load_2d(sA + stage * kABytes, &tmA, fb, kb * kBK, a_row);
#pragma unroll
                            for (int c = 0; c < kBN / static_cast<int>(kBChunkCols); ++c)
                                tma_load_2d(sB + stage * kRingB + c * kBChunkBytes, &tmB, fb,
                                            n0 + c * static_cast<int>(kBChunkCols), b_row + kb * kBK);
                            issued_mask |= 1u << stage;
                            issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                            if (++stage == kRing) {
                                stage = 0;
                                phase ^= 1u;
                            }
                        }
                    }
                }
            } else {
            for (int u = blockIdx.x; ok && u < sc.units; u += gridDim.x) {
                int mt = first_mt, nt = first_nt, seg = first_seg;
                if (u != static_cast<int>(blockIdx.x)) unit_coords(sc, u, mt, nt, seg);
                // a folded unit streams all of K; its segments follow one another
                const int kb0 = sc.fold ? 0 : seg * sc.kb_per_split;
                const int kb1 = sc.fold ? sc.kb_total : min(kb0 + sc.kb_per_split, sc.kb_total);
                const int m0 = mt * kBM, n0 = nt * kTN;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, p.status,
                                      kErrWaitProducer)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = full_bar(stage);
                    mbar_arrive_expect_tx(fb, static_cast<uint32_t>(sc.a_rows) * 128u + kRingB);
                    tma_load_2d(sA + stage * kABytes, &tmA, fb, kb * kKB, m0);
                    if constexpr (kWt) {
                        // one box: 256 weight rows x 64 k (128 bytes each)
                        tma_load_2d(sB + stage * kRingB, &tmB, fb, kb * kKB, n0);
                    } else {
#pragma unroll
                        for (int c = 0; c < kTN / static_cast<int>(kBChunkCols); ++c)
                            tma_load_2d(sB + stage * kRingB + c * kBChunkBytes, &tmB, fb,
                                        n0 + c * static_cast<int>(kBChunkCols), kb * kBK);
                    }
                    issued_mask |= 1u << stage;
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == kRing) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            }
            // Every load of this CTA is issued: the next kernel in the stream may
            // be scheduled from now on (it waits for this grid to complete before
            // touching memory; this CTA already holds its TMEM, so a dependent
            // cannot take it first).  Triggering here rather than at the start
            // keeps the next kernel's blocks from starting while this one is
            // still streaming.
            grid_launch_dependents();
            // No copy may still be in flight when the CTA exits: wait (bounded)
            // for the last load issued into every stage.
            for (int s = 0; s < kRing; ++s)
                if (issued_mask & (1u << s))
                    wait_bounded(full_bar(s), (issued_parity >> s) & 1u, abort_flag, p.status,
                                 kErrWaitDrain, /*honour_abort=*/false);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------- MMA issuer --
            int stage = 0;
            uint32_t phase = 0;
            int t = 0;  // accumulators filled so far (one per segment)
            bool ok = true;
            // an Ozaki item is one (slice pair, tile), over all of K
            const int n_items = (kOut == kOutOzaki) ? p.units * oz_pairs : p.units;
            for (int u = blockIdx.x; ok && u < n_items; u += gridDim.x) {
                int mt = 0, nt = 0, seg0 = 0;
                if constexpr (kOut != kOutOzaki) unit_coords(p, u, mt, nt, seg0);
                // A folded unit fills one accumulator per K segment, in order; the
                // epilogue adds them.  Otherwise the unit is the single segment seg0.
                const int nseg = (kOut != kOutOzaki && p.fold) ? p.splits : 1;
                for (int sg = 0; ok && sg < nseg; ++sg, ++t) {
                    const int seg = p.fold ? sg : seg0;
                    const int kb0 = seg * p.kb_per_split;
                    const int kb1 = min(kb0 + p.kb_per_split, p.kb_total);
                    const int acc = t % kAccStages;
                    const uint32_t acc_phase = static_cast<uint32_t>(t / kAccStages) & 1u;
                    if (!wait_bounded(tempty_bar(acc), acc_phase ^ 1u, abort_flag, p.status,
                                      kErrWaitMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kTN);
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!wait_bounded(full_bar(stage), phase, abort_flag, p.status, kErrWaitMma)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a0 = sA + stage * kABytes;
                        const uint32_t b0 = sB + stage * kRingB;
    #pragma unroll
                        for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
                            // A: K-major, 128-byte rows; advance 16 elements = 32 bytes.
                            const uint64_t ad = smem_desc_sw128(a0 + kk * kUmmaK * 2, 16, 1024);
                            uint64_t bd;
                            if constexpr (kWt) {
                                // W: K-major like A, 256 rows of 128 bytes.
                                bd = smem_desc_sw128(b0 + kk * kUmmaK * 2, 16, 1024);
                            } else {
                                // B: N-major; 16 k-rows of 128 bytes = 2048 bytes per step.
                                // LBO = distance between 64-column chunks, SBO = 8 k-rows.
                                bd = smem_desc_sw128(b0 + kk * kUmmaK * 128, kBChunkBytes, 1024);
                            }
                            if constexpr (kFp8)
                                mma_fp8(d_tmem, ad, bd, p.idesc_fp8, (kb > kb0 || kk > 0) ? 1u : 0u);
                            else
                                mma_bf16(d_tmem, ad, bd, kWt ? TileT::kIdescWt : TileT::kIdescBN,
                                         (kb > kb0 || kk > 0) ? 1u : 0u);
                        }
                        mma_commit(empty_bar(stage));
                        if (++stage == kRing) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (!ok) break;
                    mma_commit(tfull_bar(acc));
                }
            }
            // Every MMA this thread issued completes before TMEM is released.
            mma_commit(drain_bar);
            wait_bounded(drain_bar, 0, abort_flag, p.status, kErrWaitDrain, /*honour_abort=*/false);
        }
      }
      // The cluster's two barriers (see the epilogue): every thread of every
      // CTA passes both, on every path.
      if constexpr ((kOut == kOutF32 || kOut == kOutBF16) && kTN == kBN) {
          if (p.cluster) {
              cluster_arrive_release();
              cluster_wait_acquire();
              cluster_arrive_release();
              cluster_wait_acquire();
          }
      }
    } else {
        if constexpr (kSplitRegs) regs_grow_to<kEpilogueRegs>();
        // ------------------------------------------------------ epilogue --
        // Warp w reads TMEM lanes 32 (w % 4) .. +31, i.e. tile rows q*32 .. q*32+31,
        // and the columns of half h = (w - 4) / 4 of the tile (128 each).
        // Blocks of 32 x 32 go TMEM -> registers -> swizzled staging boxes -> TMA
        // stores (coalesced, asynchronous; rows >= M and columns >= N fall outside
        // the tensor map and are not written).  A batch of epi_batch blocks is
        // read from TMEM with one load, staged, fenced once and stored with one
        // TMA store (or one per block when the output is not viewed as column
        // groups); each batch is one bulk group.  The warps that have rows split
        // the eight boxes evenly -- a split that depends on M alone, so every
        // warp owns its boxes for the whole launch and recycles them batch by
        // batch.
        const int q = warp & 3;
        const int h = (warp - kEpilogueWarp0) >> 2;
        const int per_warp = p.epi_boxes;
        const int batch = p.epi_batch;
        const int slots = per_warp / batch;  // batches in flight per warp (2 or 1)
        // fp32 boxes are 32 rows x 128 bytes; bf16 boxes 32 rows x 64 bytes, packed
        // at 2 KiB so that a batch of them is one contiguous grouped box.
        // (Warps whose rows are always past M never use their box range.)
        constexpr uint32_t kBox = (kOut == kOutBF16) ? kStageBufBytes / 2 : kStageBufBytes;
        const uint32_t my_boxes = sOut + static_cast<uint32_t>((q * 2 + h) * per_warp) * kBox;
        uint32_t nbat = 0;  // batches this warp has handed to the TMA unit
        int t = 0;          // accumulators drained so far (one per segment)
        bool folded = false;
        if constexpr (kOut == kOutOzaki) {
            // ---- Ozaki scheme: for the item's slice pair (pa, pb), C[row][col] +=
            // 2^e * P with P the FP32 slice-pair product (exact) and e =
            // c_a^(pa)[row] + c_b^(pb)[col]; the first pair starts the sum at
            // +0.0.  A warp adds pair k into its 32 rows x 128 columns only
            // once the tile's count shows that all warps have added pair k - 1
            // (whichever CTA ran it), then raises the count: every element
            // takes its pairs in the order of the binary64 sum.  Each lane's
            // acquiring read of the count orders its reads of C after the
            // stores that raised it (each writer lane fences before the count
            // is raised).
            folded = true;
            double* C = static_cast<double*>(p.out);
            const int step = p.oz_beta + 1;
            bool ok = true;
            // the producer's order: items pair-major
            int pa = 0, pb = 0, pk = 0;
            const int items = p.units * oz_pairs;
            for (int L = blockIdx.x; ok && L < items; L += gridDim.x) {
                const int pair = L / p.units, u = L - pair * p.units;
                for (; pk < pair; ++pk) ozaki_next_pair(p, oz_d, pa, pb);
                {
                    int mt, nt, seg;
                    unit_coords(p, u, mt, nt, seg);
                    const int m0 = mt * kBM + q * 32, n0 = nt * kBN;
                    const int row = m0 + lane;
                    const bool row_ok = row < p.M;
                    const int acc = t % kAccStages;
                    const uint32_t acc_phase = static_cast<uint32_t>(t / kAccStages) & 1u;
                    if (!wait_bounded(tfull_bar(acc), acc_phase, abort_flag, p.status, kErrWaitEpilogue)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (pair > 0) {
                        // wait (bounded) for pair - 1 of this tile in every warp
                        bool in_order = true;
                        if (lane == 0)
                            in_order = wait_count_bounded(p.oz_count + u, pair * kEpilogueWarps,
                                                          abort_flag, p.oz_count + p.units, p.status);
                        in_order = __shfl_sync(0xffffffffu, in_order ? 1 : 0, 0) != 0;
                        if (!in_order) {
                            tc_fence_before();
                            mbar_arrive(tempty_bar(acc));
                            ok = false;
                            break;
                        }
                        // every lane acquires the count itself, so that its own
                        // loads of C below come after the previous pair's stores
                        (void)ld_acquire_gpu(p.oz_count + u);
                    }
                    if (m0 < p.M) {
                        const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                               static_cast<uint32_t>(acc * kBN);
                        const int e_pair = row_ok ? (p.oz_ca[row] - pa * step) - pb * step : 0;
                        // Fast Mode: the row's limit on the column masses for this pair
                        OzakiFastRow fast = ozaki_fast_row(p.oz_fast ? p.oz_tb : nullptr,
                                                           (p.oz_fast && row_ok) ? p.oz_ta[row] : 0ull,
                                                           (pa + pb) * step, p.oz_need0);
#pragma unroll 1
                        for (int i = 0; i < 4; ++i) {
                            uint32_t r[32];
                            tmem_ld_32x32b_x32(tbase + (h * 4 + i) * 32, r);
                            tmem_ld_wait();
                            if (i == 3) {  // the accumulator is no longer needed
                                tc_fence_before();
                                mbar_arrive(tempty_bar(acc));
                            }
                            const int col0 = n0 + (h * 4 + i) * 32;
                            if (p.oz_fast) fast.tb = p.oz_tb + col0;  // 256-byte aligned: col0 % 32 == 0
                            if (col0 + 32 <= p.N && p.ld_out >= kOzStagedMinLd)
                                ozaki_accumulate_block_staged(
                                    C + static_cast<int64_t>(m0) * p.ld_out + col0, p.ld_out, min(32, p.M - m0),
                                    p.oz_cb + col0, e_pair, r, pair == 0, fast,
                                    reinterpret_cast<double*>(gbase + (sOut - base)) + (q * 2 + h) * 512, lane);
                            else if (row_ok && col0 < p.N)
                                ozaki_accumulate_block(C + static_cast<int64_t>(row) * p.ld_out + col0,
                                                       p.oz_cb + col0, min(32, p.N - col0), e_pair, r,
                                                       pair == 0, fast, p.oz_c32 != 0);
                        }
                    } else {
                        tc_fence_before();
                        mbar_arrive(tempty_bar(acc));
                    }
                    // this warp's part of the pair is in C: count it
                    __threadfence();
                    __syncwarp();
                    if (lane == 0) atomicAdd(p.oz_count + u, 1);
                    ++t;
                }
            }
        }
        if constexpr ((kOut == kOutF32 || kOut == kOutBF16) && kTN == kBN) {
            if (p.cluster) {
                // ---- one K segment of a clustered tile: the FP32 partial goes
                // to this CTA's shared memory (the pipeline stages, idle once
                // the last MMA has completed), row r of the tile at r * 1 KiB,
                // its 16-byte chunk c at c ^ (r % 8).
                folded = true;
                if (static_cast<int>(blockIdx.x) < p.units) {
                    int mt, nt, seg;
                    unit_coords(p, blockIdx.x, mt, nt, seg);
                    if (wait_bounded(tfull_bar(0), 0, abort_flag, p.status, kErrWaitEpilogue)) {
                        tc_fence_after();
                        // the tensor core's reads of the stages are complete
                        fence_proxy_async_smem();
                        if (mt * kBM + q * 32 < p.M) {
                            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
                            const uint32_t row = static_cast<uint32_t>(q * 32 + lane);
                            const uint32_t prow = sA + row * 1024u;
#pragma unroll 1
                            for (int i = 0; i < 4; ++i) {
                                uint32_t r[32];
                                tmem_ld_32x32b_x32(tbase + (h * 4 + i) * 32, r);
                                tmem_ld_wait();
#pragma unroll
                                for (int j = 0; j < 8; ++j) {
                                    const uint32_t c = static_cast<uint32_t>(h * 32 + i * 8 + j);
                                    st_shared_v4(prow + ((c ^ (row & 7u)) << 4), r[4 * j], r[4 * j + 1],
                                                 r[4 * j + 2], r[4 * j + 3]);
                                }
                            }
                        }
                        tc_fence_before();
                        mbar_arrive(tempty_bar(0));
                    }
                }
                // The first barrier publishes the partials to the cluster; the
                // second keeps each CTA's shared memory alive until the others
                // have read it.  Every thread of every CTA of the cluster
                // passes both, on every path (the first warpgroup included).
                cluster_arrive_release();
                cluster_wait_acquire();
                if (static_cast<int>(blockIdx.x) < p.units)
                    cluster_reduce<kOut>(p, sA, static_cast<int>(threadIdx.x) - kEpilogueWarp0 * 32);
                cluster_arrive_release();
                cluster_wait_acquire();
            } else if (p.fold) {
                // ---- folded tiles: sum = w_0, then sum = sum + w_s for s = 1 ..
                // splits-1 (FP32, round to nearest even) -- the additions
                // splitk_reduce_kernel makes, in the same order, on the same
                // partials, so the bits agree with the workspace path.  The
                // host folds only when every warp with rows stores one block per
                // batch (p.epi_batch == 1).  The sum lives in 128 registers.
                folded = true;
                for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
                    int mt, nt, seg;
                    unit_coords(p, u, mt, nt, seg);
                    const int m0 = mt * kBM + q * 32, n0 = nt * kBN;
                    const int nchunks = min(h * 4 + 4, min(kBN / 32, (p.N - n0 + 31) / 32));
                    uint32_t sum[128];
                    bool ok = true;
#pragma unroll 1
                    for (int sg = 0; sg < p.splits; ++sg, ++t) {
                        const int acc = t % kAccStages;
                        const uint32_t acc_phase = static_cast<uint32_t>(t / kAccStages) & 1u;
                        if (!wait_bounded(tfull_bar(acc), acc_phase, abort_flag, p.status,
                                          kErrWaitEpilogue)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        if (m0 < p.M) {
                            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                                   static_cast<uint32_t>(acc * kBN);
                            if (sg == 0) {  // sum = w_0 itself (a -0.0 stays -0.0)
#pragma unroll
                                for (int i = 0; i < 4; ++i)
                                    if (h * 4 + i < nchunks)
                                        tmem_ld_32x32b_x32(tbase + (h * 4 + i) * 32,
                                                           *reinterpret_cast<uint32_t(*)[32]>(sum + 32 * i));
                                tmem_ld_wait();
                            } else {
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    if (h * 4 + i < nchunks) {
                                        uint32_t w[32];
                                        tmem_ld_32x32b_x32(tbase + (h * 4 + i) * 32, w);
                                        tmem_ld_wait();
#pragma unroll
                                        for (int j = 0; j < 32; ++j)
                                            sum[32 * i + j] = __float_as_uint(__fadd_rn(
                                                __uint_as_float(sum[32 * i + j]), __uint_as_float(w[j])));
                                    }
                                }
                            }
                        }
                        tc_fence_before();
                        mbar_arrive(tempty_bar(acc));
                    }
                    if (!ok) break;
                    if (m0 < p.M) {
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            if (h * 4 + i < nchunks)
                                emit_blocks<kOut, 1>(p, &tmC, sum + 32 * i, 1, h * 4 + i, n0, m0, seg,
                                                     lane, my_boxes, 1, slots, nbat);
                    }
                }
            }
        }
        if (!folded) {
            for (int u = blockIdx.x; u < p.units; u += gridDim.x, ++t) {
                int mt, nt, seg;
                unit_coords(p, u, mt, nt, seg);
                const int m0 = mt * kBM + q * 32, n0 = nt * kTN;
                // this warp's 32-column blocks: [h * kHB, nchunks)
                const int nchunks = min(h * kHB + kHB, min(kTN / 32, (p.N - n0 + 31) / 32));
                const int acc = t % kAccStages;
                const uint32_t acc_phase = static_cast<uint32_t>(t / kAccStages) & 1u;
                if (!wait_bounded(tfull_bar(acc), acc_phase, abort_flag, p.status, kErrWaitEpilogue))
                    break;
                tc_fence_after();
                bool released = false;
                if (m0 < p.M) {  // uniform per warp: a warp whose rows are all past M skips
                    const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                           static_cast<uint32_t>(acc * kTN);
#pragma unroll 1
                    for (int c0 = h * kHB; c0 < nchunks; c0 += batch) {
                        const int nb = min(batch, nchunks - c0);
                        uint32_t r[kMaxBatch * 32];
                        if (batch == 4) tmem_ld_32x32b_x128(tbase + c0 * 32, r);
                        else if (batch == 2) tmem_ld_32x32b_x64(tbase + c0 * 32, r);
                        else tmem_ld_32x32b_x32(tbase + c0 * 32, *reinterpret_cast<uint32_t(*)[32]>(r));
                        tmem_ld_wait();
                        if (c0 + nb >= nchunks) {  // the accumulator is no longer needed
                            tc_fence_before();
                            mbar_arrive(tempty_bar(acc));
                            released = true;
                        }
                        emit_blocks<kOut, kMaxBatch>(p, &tmC, r, nb, c0, n0, m0, seg, lane, my_boxes,
                                                     batch, slots, nbat);
                    }
                }
                if (!released) {
                    tc_fence_before();
                    mbar_arrive(tempty_bar(acc));
                }
            }
        }
        // All of this warp's stores complete before the CTA exits.
        if (lane == 0) bulk_wait_group<0>();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TileT::kTmemCols);
    }
}

// Split-K reduction: for every element, acc = w_0, then acc = acc + w_s for
// s = 1 .. S-1 in that order (FP32, round to nearest even), then acc * scale
// and acc + bias[n] when given; starting from w_0
// rather than 0.0f keeps a lone -0.0 partial intact.  One thread handles four
// adjacent columns of one row (16-byte loads, coalesced along N); the loads of
// up to eight slices are issued before their additions.
constexpr int kReduceThreads = 128;

// kBias: a linear layer's bias[N] is added (the pointer is then non-null);
// the products without one run the kernel without any of that code.
template <bool kBF16Out, bool kBias>
__global__ void __launch_bounds__(kReduceThreads)
    splitk_reduce_kernel(const float* __restrict__ ws, void* __restrict__ C, int M, int N,
                         int64_t ldc, int64_t ws_ld, int S, const __nv_bfloat16* __restrict__ bias,
                         float scale) {
    // The next kernel in the stream may be scheduled at once: it waits for
    // this grid to complete before touching memory, and this kernel holds no
    // tensor memory a dependent could need.
    grid_launch_dependents();
    const int64_t vec_per_row = ws_ld / 4;
    if constexpr (kBias) {
        // Warm L2 with this thread's first bias values while the partial
        // kernel finishes: a linear layer's bias is read once per product and
        // is usually gone from L2 by then, and its trip from DRAM would
        // otherwise come after the slices'.  An L2 prefetch fills nothing in
        // the SM and L2 is the device's point of coherence, so it cannot
        // expose data older than the dependency wait below.
        const int64_t v0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
        if (v0 < static_cast<int64_t>(M) * vec_per_row)
            prefetch_l2(bias + static_cast<int>(v0 % vec_per_row) * 4);
    }
    grid_dependency_wait();
    const int64_t total = static_cast<int64_t>(M) * vec_per_row;
    const int64_t slice = static_cast<int64_t>(M) * ws_ld;
    for (int64_t v = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; v < total;
         v += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t m = v / vec_per_row;
        const int col = static_cast<int>(v - m * vec_per_row) * 4;
        const float* src = ws + m * ws_ld + col;
        int valid = 0;
        uint2 bw = make_uint2(0u, 0u);
        if constexpr (kBias) {
            // four bf16 values in one 8-byte load (col is a multiple of 4 and
            // the bias 16-byte aligned), issued before the slices' loads so
            // that the two latencies overlap: this kernel's time is the
            // latency of its loads
            valid = min(4, N - col);
            if (valid == 4) bw = __ldg(reinterpret_cast<const uint2*>(bias + col));
        }
        // S == 0: no slices (an empty K); the sum is +0.0 and only a bias remains
        float4 acc = S > 0 ? __ldcs(reinterpret_cast<const float4*>(src)) : make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s0 = 1; s0 < S; s0 += 8) {
            float4 w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (s0 + i < S) w[i] = __ldcs(reinterpret_cast<const float4*>(src + (s0 + i) * slice));
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (s0 + i < S) {
                    acc.x = __fadd_rn(acc.x, w[i].x);
                    acc.y = __fadd_rn(acc.y, w[i].y);
                    acc.z = __fadd_rn(acc.z, w[i].z);
                    acc.w = __fadd_rn(acc.w, w[i].w);
                }
            }
        }
        if constexpr (!kBias) valid = min(4, N - col);
        if (valid <= 0) continue;
        if (scale != 1.0f) {  // an 8-bit product's output scale, after the split sum
            acc.x = __fmul_rn(acc.x, scale);
            acc.y = __fmul_rn(acc.y, scale);
            acc.z = __fmul_rn(acc.z, scale);
            acc.w = __fmul_rn(acc.w, scale);
        }
        if constexpr (kBias) {  // added after the split sum (and the scale)
            if (valid == 4) {
                // a bf16 value is the upper half of the FP32 with the same value
                acc.x = __fadd_rn(acc.x, __uint_as_float(bw.x << 16));
                acc.y = __fadd_rn(acc.y, __uint_as_float(bw.x & 0xFFFF0000u));
                acc.z = __fadd_rn(acc.z, __uint_as_float(bw.y << 16));
                acc.w = __fadd_rn(acc.w, __uint_as_float(bw.y & 0xFFFF0000u));
            } else {
                float* a = &acc.x;
                for (int c = 0; c < valid; ++c) a[c] = __fadd_rn(a[c], __bfloat162float(bias[col + c]));
            }
        }
        if constexpr (kBF16Out) {
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(C) + m * ldc + col;
            if (valid == 4) {
                __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
                __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
                uint2 pk = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
                *reinterpret_cast<uint2*>(dst) = pk;
            } else {
                const float a[4] = {acc.x, acc.y, acc.z, acc.w};
                for (int c = 0; c < valid; ++c) dst[c] = __float2bfloat16_rn(a[c]);
            }
        } else {
            float* dst = static_cast<float*>(C) + m * ldc + col;
            if (valid == 4) {
                *reinterpret_cast<float4*>(dst) = acc;
            } else {
                const float a[4] = {acc.x, acc.y, acc.z, acc.w};
                for (int c = 0; c < valid; ++c) dst[c] = a[c];
            }
        }
    }
}

// Bt[n][k] = B[k][n] for 8-bit operands: B [K, N] (ldb bytes per row) copied
// K-major into Bt [N, ldt] (ldt a multiple of 16, >= K), the layout the 8-bit
// tensor-core path reads; columns k in [K, ldt) of Bt are written as zeros.
// One 64 x 64 byte tile per block through shared memory, 4-byte accesses on
// both sides (byte accesses at a ragged right edge of B).  A byte copy: the
// values, and so every product formed from them, are unchanged.
constexpr int kTrTile = 64;
constexpr int kTrThreads = 256;

__global__ void __launch_bounds__(kTrThreads)
    fp8_transpose_kernel(const uint8_t* __restrict__ B, int64_t ldb, uint8_t* __restrict__ Bt, int64_t ldt,
                         int K, int N) {
    __shared__ uint8_t tile[kTrTile][kTrTile + 4];
    const int k0 = static_cast<int>(blockIdx.y) * kTrTile, n0 = static_cast<int>(blockIdx.x) * kTrTile;
    for (int i = threadIdx.x; i < kTrTile * (kTrTile / 4); i += kTrThreads) {
        const int r = i / (kTrTile / 4), w = i % (kTrTile / 4);
        const int k = k0 + r, n = n0 + 4 * w;
        uint32_t v = 0;
        if (k < K && n < N) {
            const uint8_t* src = B + static_cast<int64_t>(k) * ldb + n;
            if (n + 4 <= N) {
                v = *reinterpret_cast<const uint32_t*>(src);  // 4-byte aligned: ldb % 16 == 0, n % 4 == 0
            } else {
                for (int j = 0; j < N - n; ++j) v |= static_cast<uint32_t>(src[j]) << (8 * j);
            }
        }
        tile[r][4 * w] = static_cast<uint8_t>(v);
        tile[r][4 * w + 1] = static_cast<uint8_t>(v >> 8);
        tile[r][4 * w + 2] = static_cast<uint8_t>(v >> 16);
        tile[r][4 * w + 3] = static_cast<uint8_t>(v >> 24);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kTrTile * (kTrTile / 4); i += kTrThreads) {
        const int r = i / (kTrTile / 4), w = i % (kTrTile / 4);
        const int n = n0 + r, k = k0 + 4 * w;
        if (n < N && k < ldt) {
            const uint32_t v = static_cast<uint32_t>(tile[4 * w][r]) | (static_cast<uint32_t>(tile[4 * w + 1][r]) << 8) |
                               (static_cast<uint32_t>(tile[4 * w + 2][r]) << 16) |
                               (static_cast<uint32_t>(tile[4 * w + 3][r]) << 24);
            *reinterpret_cast<uint32_t*>(Bt + static_cast<int64_t>(n) * ldt + k) = v;  // ldt % 16 == 0
        }
    }
}

}  // namespace bigemm
