// skinny.cuh -- products with few rows (decode-shaped batches, M <= 32), their
// split-K sum formed inside one launch.
//
// The arithmetic is that of bigemm_tc_kernel, instruction for instruction:
// every element C[i][j] is the sum of its K segments' FP32 partials in the
// order 0..S-1, each partial one TMEM accumulator fed by the segment's K
// blocks of 64 in ascending order, four tcgen05.mma (M = 128, N = 256,
// K = 16) per block, with the same operand roles and instruction descriptors
// ("Tiling", "Split-K" and "Batch Invariance の由来" on the Tencent AI-infra page
// "腾讯エンジニア：大規模モデルの出力を確定させるための AI インフラ手法").  So the
// bits are those of the other paths by construction.  What changes is the
// shape of the work around the instructions, to suit a batch of a few rows
// against a large weight matrix:
//
//   * One CTA computes one K segment of one 128 x 256 output tile, and the S
//     CTAs of a tile form a thread-block cluster (S <= 8).  After the last
//     instruction every CTA writes the batch rows of its partial into its own
//     shared memory; the cluster then adds them through distributed shared
//     memory in the order 0..S-1 with the FP32 additions of
//     splitk_reduce_kernel and stores C.  No workspace, no second kernel.
//   * A stage holds only the batch's rows of A (16 or 32 rows of 128
//     bytes).  The instruction still reads 128 rows; the descriptor's rows
//     past the stage's run on into the next shared-memory bytes, which feed
//     only output rows >= M: each output row of a tensor-core product is
//     formed from its own row of A and from B alone, and rows >= M are
//     never stored.
//   * A CTA takes under half of an SM (at most 112 KiB of shared memory, 192
//     threads, 256 TMEM columns), so the next product's CTAs can be resident
//     while this one runs.  Under programmatic launch they may start once
//     this grid has issued its last loads, and before their own wait their
//     idle epilogue warps warm L2 with their weight segment (an L2 prefetch
//     fills no shared memory, and L2 is the device's point of coherence, so
//     it cannot expose data older than the wait).  The next product's
//     weights then stream from HBM during this product's last loads, its
//     split sum and the kernel boundary.
#pragma once

#include "kernels.cuh"

namespace bigemm {

constexpr int kSkMaxM = 32;               // batch rows served
constexpr int kSkMaxCluster = 8;          // segments (one CTA each) per tile
constexpr int kSkThreads = 192;           // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kSkEpiWarp0 = 2;
constexpr int kSkEpiThreads = 128;
constexpr int kSkMaxStages = 8;
constexpr int kSkPullItems = 2;           // (row, four-column group) items per thread per round
constexpr uint32_t kSkBBytes = kBK * kBN * 2;             // 32 KiB of weights per K block
constexpr int kSkBarriers = 2 * kSkMaxStages + 2;         // full, empty, accumulator done, drain
// Ring bytes that leave room for a second CTA on the SM (228 KiB of shared
// memory per SM, 1 KiB of it reserved per CTA).
constexpr uint32_t kSkHalfSmBytes = 112u * 1024u;
static_assert(2 * (kSkHalfSmBytes + kSkBarriers * 8 + 16 + 1024) <= 228u * 1024u, "two CTAs per SM");

// Rows of A a stage holds: the batch rounded up to 16 or 32.
__host__ __device__ constexpr int sk_a_rows(int M) { return M <= 16 ? 16 : 32; }
__host__ __device__ constexpr uint32_t sk_a_bytes(int M) { return static_cast<uint32_t>(sk_a_rows(M)) * 128u; }
__host__ __device__ constexpr uint32_t sk_stage_bytes(int M) { return sk_a_bytes(M) + kSkBBytes; }
// Layout: the A slots of all stages, then the B slots, then the barriers.
// The instruction reads 16 KiB from an A slot's start, which always stays
// inside the ring (the B slots follow).
__host__ __device__ constexpr uint32_t sk_smem_bytes(int M, int stages) {
    return static_cast<uint32_t>(stages) * sk_stage_bytes(M) + kSkBarriers * 8 + 16;
}
// The partials a CTA writes for the split sum: M rows of 256 fp32 values.
__host__ __device__ constexpr uint32_t sk_partial_bytes(int M) { return static_cast<uint32_t>(M) * kBN * 4u; }
static_assert(sk_partial_bytes(kSkMaxM) <= 2 * sk_stage_bytes(kSkMaxM), "partials fit in a 2-stage ring");
static_assert(3 * sk_stage_bytes(kSkMaxM) <= kSkHalfSmBytes, "three stages beside a second CTA");
static_assert(kABytes <= kSkBBytes, "an A slot's 128-row read stays inside the ring");

struct SkinnyParams {
    void* out;              // C [M, N], fp32 or bf16
    int64_t ldc;
    const __nv_bfloat16* w; // the weights: B [K, N] (ldw = ldb) or W [N, K] (ldw)
    int64_t ldw;
    unsigned* status;       // device error word
    const __nv_bfloat16* bias;  // [N] or nullptr: added after the split sum
    int M, N, K;
    int stages;             // ring depth (<= kSkMaxStages)
    int splits;             // effective K segments S = CTAs per cluster (<= 8)
    int kb_total;           // ceil(K / 64)
    int kb_per_split;       // K blocks per segment L
};

// Warms L2 with the K blocks [kb0, kb1) of this CTA's weights (output
// columns n0 .. n0 + 255, none past N), one prefetch instruction per 128-byte
// line, dealt over the 128 epilogue threads (thread `e`).  Plain prefetch
// instructions, not the TMA unit's: the TMA unit of an SM serves both CTAs
// on it, and tensor prefetches queued there delay the other CTA's loads.
template <bool kWt>
__device__ __forceinline__ void sk_warm_l2(const SkinnyParams& p, int n0, int kb0, int kb1, int e) {
    const int k0 = kb0 * kBK, k1 = min(kb1 * kBK, p.K);
    const int c1 = min(n0 + kBN, p.N);
    if (k0 >= k1 || n0 >= c1) return;
    // rows of the region and the byte span each row covers
    const int rows = kWt ? (c1 - n0) : (k1 - k0);
    const int64_t first = kWt ? static_cast<int64_t>(n0) * p.ldw + k0 : static_cast<int64_t>(k0) * p.ldw + n0;
    const int span = 2 * (kWt ? (k1 - k0) : (c1 - n0));
    const char* base = reinterpret_cast<const char*>(p.w + first);
    const int64_t stride = 2 * p.ldw;
    // lines per row: enough for the span from any 16-byte-aligned start
    const int lines = (span + 127 + 112) / 128;
    for (int v = e; v < rows * lines; v += kSkEpiThreads) {
        const int r = v / lines, l = v - r * lines;
        const char* row = base + r * stride;
        const uintptr_t a = (reinterpret_cast<uintptr_t>(row) & ~static_cast<uintptr_t>(127)) +
                            static_cast<uintptr_t>(l) * 128u;
        if (a < reinterpret_cast<uintptr_t>(row) + static_cast<uintptr_t>(span))
            prefetch_l2(reinterpret_cast<const void*>(a));
    }
}

// One four-column group of one row of C: acc = w_0, then acc + w_s for s = 1
// .. S-1 (FP32, round to nearest even; starting from w_0 itself keeps a lone
// -0.0), then + bias, then the store (fp32, or bf16 rounded to nearest even).
template <int kOut>
__device__ __forceinline__ void sk_finish(const SkinnyParams& p, const float4 (&w)[kSkMaxCluster], int S,
                                          int row, int col) {
    float4 acc = w[0];
#pragma unroll
    for (int s = 1; s < kSkMaxCluster; ++s) {
        if (s < S) {
            acc.x = __fadd_rn(acc.x, w[s].x);
            acc.y = __fadd_rn(acc.y, w[s].y);
            acc.z = __fadd_rn(acc.z, w[s].z);
            acc.w = __fadd_rn(acc.w, w[s].w);
        }
    }
    const int valid = min(4, p.N - col);
    if (p.bias != nullptr) {
        float* a = &acc.x;
        if (valid == 4) {
            const uint2 bw = __ldg(reinterpret_cast<const uint2*>(p.bias + col));
            // a bf16 value is the upper half of the FP32 with the same value
            a[0] = __fadd_rn(a[0], __uint_as_float(bw.x << 16));
            a[1] = __fadd_rn(a[1], __uint_as_float(bw.x & 0xFFFF0000u));
            a[2] = __fadd_rn(a[2], __uint_as_float(bw.y << 16));
            a[3] = __fadd_rn(a[3], __uint_as_float(bw.y & 0xFFFF0000u));
        } else {
            for (int k = 0; k < valid; ++k) a[k] = __fadd_rn(a[k], __bfloat162float(p.bias[col + k]));
        }
    }
    if constexpr (kOut == kOutBF16) {
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + static_cast<int64_t>(row) * p.ldc + col;
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
        float* dst = static_cast<float*>(p.out) + static_cast<int64_t>(row) * p.ldc + col;
        if (valid == 4) {
            *reinterpret_cast<float4*>(dst) = acc;
        } else {
            const float a[4] = {acc.x, acc.y, acc.z, acc.w};
            for (int k = 0; k < valid; ++k) dst[k] = a[k];
        }
    }
}

template <int kOut, bool kWt>
__global__ void __launch_bounds__(kSkThreads, 1)
    bigemm_skinny_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         const SkinnyParams p) {
    static_assert(kOut == kOutF32 || kOut == kOutBF16, "direct outputs only");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const bool clustered = p.splits > 1;  // uniform; the layout check below uses it
    const uint32_t base = smem_addr(smem_raw);
    if (base & 1023u) {
        // The swizzled layout needs a 1024-byte base.  Report it, touch
        // nothing, and still pass the cluster's two barriers, which every
        // thread of every CTA of the cluster must reach.
        if (threadIdx.x == 0) atomicOr(p.status, kErrSmemAlign);
        if (clustered) {
            cluster_arrive_release();
            cluster_wait_acquire();
            cluster_arrive_release();
            cluster_wait_acquire();
        }
        return;
    }
    // The scalars every role needs after the dependency wait, read here, in
    // the prologue that overlaps the previous kernel, and kept in registers:
    // the parameters are new at every launch, and their first reads miss the
    // constant cache.
    int stages = p.stages, S = p.splits, kb_total = p.kb_total, L = p.kb_per_split, M = p.M;
    asm volatile("" : "+r"(stages), "+r"(S), "+r"(kb_total), "+r"(L), "+r"(M));
    const uint32_t a_bytes = sk_a_bytes(M);
    const uint32_t sB = base + static_cast<uint32_t>(stages) * a_bytes;  // B slot s: sB + s * 32 KiB
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw + stages * (a_bytes + kSkBBytes));
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kSkBarriers);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const uint32_t bar0 = smem_addr(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kSkMaxStages + s); };
    const uint32_t done_bar = bar0 + 8u * (2 * kSkMaxStages);
    const uint32_t drain_bar = done_bar + 8u;

    // This CTA: tile `tile` (columns n0 .. n0 + 255), K segment `seg` (its
    // rank in the tile's cluster), K blocks kb0 .. kb1 - 1.
    const int tile = static_cast<int>(blockIdx.x) / S;
    const int seg = static_cast<int>(blockIdx.x) - tile * S;
    const int n0 = tile * kBN;
    const int kb0 = seg * L;
    const int kb1 = min(kb0 + L, kb_total);

    if (warp == 1 && lane == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(done_bar, 1);
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 2) {
        tmem_alloc(smem_addr(tmem_slot), static_cast<uint32_t>(kBN));
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp >= kSkEpiWarp0) {
        // Idle until the accumulator is complete: warm L2 with this CTA's
        // weights and bias meanwhile (while the previous kernel in the stream
        // finishes, when this CTA started early).
        const int e = static_cast<int>(threadIdx.x) - kSkEpiWarp0 * 32;
        sk_warm_l2<kWt>(p, n0, kb0, kb1, e);
        if (p.bias != nullptr && e * 64 < min(kBN, p.N - n0)) prefetch_l2(p.bias + n0 + e * 64);
    }

    // From here on global memory is read and written only after the previous
    // kernel in the stream has completed.
    grid_dependency_wait();

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer --
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued_mask = 0, issued_parity = 0;
            const uint32_t tx = static_cast<uint32_t>(sk_a_rows(M)) * 128u + kSkBBytes;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, p.status, kErrWaitProducer)) break;
                const uint32_t fb = full_bar(stage);
                const uint32_t sb = sB + static_cast<uint32_t>(stage) * kSkBBytes;
                mbar_arrive_expect_tx(fb, tx);
                tma_load_2d(base + static_cast<uint32_t>(stage) * a_bytes, &tmA, fb, kb * kBK, 0);
                if constexpr (kWt) {
                    // one box: 256 weight rows x 64 k (128 bytes each)
                    tma_load_2d(sb, &tmB, fb, kb * kBK, n0);
                } else {
#pragma unroll
                    for (int c = 0; c < kBN / static_cast<int>(kBChunkCols); ++c)
                        tma_load_2d(sb + c * kBChunkBytes, &tmB, fb, n0 + c * static_cast<int>(kBChunkCols),
                                    kb * kBK);
                }
                issued_mask |= 1u << stage;
                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            // Every load of this CTA is issued: the next kernel in the stream
            // may be scheduled now and warm L2 with its weights while these
            // loads land and the split sum runs.  (Allowed earlier -- at the
            // dependency wait -- its warm-up took HBM bandwidth from this
            // kernel's loads: 10.6 against 8.9 us per M = 1 product.)
            grid_launch_dependents();
            // no copy may still be in flight when the CTA exits
            for (int s = 0; s < stages; ++s)
                if (issued_mask & (1u << s))
                    wait_bounded(full_bar(s), (issued_parity >> s) & 1u, abort_flag, p.status,
                                 kErrWaitDrain, /*honour_abort=*/false);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------- MMA issuer --
            // The wide kernel's instructions: A K-major (the batch rows), B
            // N-major from B [K, N] or K-major from W [N, K]; k ascending.
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!wait_bounded(full_bar(stage), phase, abort_flag, p.status, kErrWaitMma)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a0 = base + static_cast<uint32_t>(stage) * a_bytes;
                const uint32_t b0 = sB + static_cast<uint32_t>(stage) * kSkBBytes;
#pragma unroll
                for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
                    const uint64_t ad = smem_desc_sw128(a0 + kk * kUmmaK * 2, 16, 1024);
                    uint64_t bd;
                    if constexpr (kWt) bd = smem_desc_sw128(b0 + kk * kUmmaK * 2, 16, 1024);
                    else bd = smem_desc_sw128(b0 + kk * kUmmaK * 128, kBChunkBytes, 1024);
                    mma_bf16(tmem_base, ad, bd, kWt ? kIdescWt : kIdescBN, (kb > kb0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(empty_bar(stage));
                if (++stage == stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (ok) mma_commit(done_bar);
            // every instruction completes before TMEM is released
            mma_commit(drain_bar);
            wait_bounded(drain_bar, 0, abort_flag, p.status, kErrWaitDrain, /*honour_abort=*/false);
        }
    } else {
        // ------------------------------------------------------ epilogue --
        // Warp w reads TMEM lanes 32 (w % 4) .. + 31, i.e. batch rows; the rows
        // below M go to shared memory (the ring, idle once the last
        // instruction has completed) as P[i][j], row i at i * 1 KiB, its
        // 16-byte chunk c at c ^ (i % 8), so that the lanes' stores and the
        // cluster's reads spread over all banks.
        const int q = warp & 3;
        // (warp-uniform: the TMEM loads below are collective)
        const bool done = __all_sync(0xffffffffu, wait_bounded(done_bar, 0, abort_flag, p.status, kErrWaitEpilogue));
        if (done && q * 32 < M) {
            tc_fence_after();
            fence_proxy_async_smem();  // the tensor core's reads of the ring are complete
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
            const int i = q * 32 + lane;
            const uint32_t row = base + static_cast<uint32_t>(i) * 1024u;
            // two halves of 128 columns, each two 64-column loads and one wait
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                uint32_t r[128];
                tmem_ld_32x32b_x64(taddr + static_cast<uint32_t>(h * 128), r);
                tmem_ld_32x32b_x64(taddr + static_cast<uint32_t>(h * 128 + 64), r + 64);
                tmem_ld_wait();
                if (i < M) {
#pragma unroll
                    for (int v = 0; v < 32; ++v) {
                        const uint32_t c = static_cast<uint32_t>(h * 32 + v);
                        st_shared_v4(row + ((c ^ (static_cast<uint32_t>(i) & 7u)) << 4), r[4 * v],
                                     r[4 * v + 1], r[4 * v + 2], r[4 * v + 3]);
                    }
                }
            }
        }
    }

    // ---- The split sum.  Every thread of every CTA of the cluster passes both
    // cluster barriers on every path.  The tile's 64 four-column groups are
    // dealt to the ranks in contiguous shares (rank r takes groups
    // ceil(64 r / S) .. ceil(64 (r + 1) / S) - 1, so that each rank's stores to
    // C are contiguous); for each (row, group) of its share a rank reads the S
    // partials from the S CTAs' shared memory and adds them in the order
    // 0..S-1 (sk_finish).
    tc_fence_before();
    if (clustered) {
        cluster_arrive_release();
        cluster_wait_acquire();
    } else {
        __syncthreads();
    }
    {
        // every thread of the CTA takes part, kSkPullItems items per round
        // with all their loads issued before any addition (a round trip to
        // another CTA's shared memory takes most of a microsecond here)
        const int g0 = (seg * 64 + S - 1) / S;
        const int groups = ((seg + 1) * 64 + S - 1) / S - g0;
        const int items = M * groups;
        uint32_t src[kSkMaxCluster];
#pragma unroll
        for (int r = 0; r < kSkMaxCluster; ++r)
            src[r] = (clustered && r < S) ? map_shared_rank(base, static_cast<uint32_t>(r)) : base;
        for (int v0 = static_cast<int>(threadIdx.x); v0 < items; v0 += kSkPullItems * kSkThreads) {
            float4 w[kSkPullItems][kSkMaxCluster];
            int row[kSkPullItems], col[kSkPullItems];
            bool act[kSkPullItems];
#pragma unroll
            for (int u = 0; u < kSkPullItems; ++u) {
                const int v = v0 + u * kSkThreads;
                row[u] = v / groups;
                col[u] = n0 + (g0 + (v - row[u] * groups)) * 4;
                act[u] = v < items && col[u] < p.N;
                if (!act[u]) continue;
                const uint32_t c = static_cast<uint32_t>((col[u] - n0) >> 2);
                const uint32_t off = static_cast<uint32_t>(row[u]) * 1024u +
                                     ((c ^ (static_cast<uint32_t>(row[u]) & 7u)) << 4);
#pragma unroll
                for (int s = 0; s < kSkMaxCluster; ++s)
                    if (s < S) w[u][s] = clustered ? ld_dsmem_f32x4(src[s] + off)
                                                   : *reinterpret_cast<const float4*>(smem_raw + off);
            }
#pragma unroll
            for (int u = 0; u < kSkPullItems; ++u)
                if (act[u]) sk_finish<kOut>(p, w[u], S, row[u], col[u]);
        }
    }
    // keep every CTA's shared memory alive until the whole cluster has read it
    // (a relaxed arrival: the stores to C need not be visible to the cluster)
    if (clustered) {
        cluster_arrive_relaxed();
        cluster_wait_acquire();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem_base, static_cast<uint32_t>(kBN));
    }
}

}  // namespace bigemm
