// pair.cuh -- the 2-SM product: one 256 x 256 output tile per CTA pair,
// computed by tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16 for bf16,
// 32 for 8-bit floats): unsplit and folded split-K products, and the Ozaki
// scheme's slice-pair products.
//
// The two CTAs of a thread-block cluster of 2 form the pair.  CTA r (r = 0,
// 1) loads rows 128 r .. 128 r + 127 of the tile's A panel and columns
// 128 r .. 128 r + 127 of its B panel into its own shared memory, with plain
// TMA loads; one thread of CTA 0 issues the pair instructions, which read
// both CTAs' halves and leave rows 128 r .. of the FP32 sum in CTA r's TMEM.
// Each CTA's stage therefore holds 16 KiB of A and 16 KiB of B instead of
// 16 + 32 KiB: a third less shared-memory traffic per instruction's worth of
// work, and six stages instead of four.
//
// Every output element is still one FP32 accumulation chain over the K
// blocks in ascending order, 16 (or 32) k per instruction, as in the 1-SM
// kernel;
// the GPU tests check that both give the same bits (rows of a 2-SM product
// against the same rows from the 1-SM kernel and from one-row products).
// (Tencent AI-infra article "腾讯エンジニア：大規模モデルの出力を確定させるため
// の AI インフラ手法", "Tiling" and "Batch Invariance の由来": the tile shape
// may change, the reduction order of an element may not.)
//
// Synchronisation (all waits bounded, see wait_bounded):
//   full[s]   CTA 0 only: its producer's arrival expecting both CTAs' bytes
//             of stage s; the TMA loads of both CTAs complete on it.
//   empty[s]  in both CTAs: one tensor-core commit from CTA 0's MMA thread.
//   tfull[a]  in both CTAs: one commit per finished accumulator.
//   tempty[a] CTA 0 only: every epilogue thread of both CTAs (count 512).
// A kernel-wide cluster barrier after the set-up (the peer's barriers are
// initialised before any remote arrival) and another before the TMEM is
// released (CTA 0's instructions, which read CTA 1's shared memory and
// write CTA 1's TMEM, have completed before CTA 1 frees either).
#pragma once

#include "kernels.cuh"

namespace bigemm {

constexpr int kPairBM = 2 * kBM;                                  // 256 rows per pair tile
constexpr uint32_t kPairBBytes = kBK * (kBN / 2) * 2;             // 16 KiB: this CTA's half of B
constexpr uint32_t kPairStageBytes = kABytes + kPairBBytes;       // 32 KiB
constexpr int kPairStages = 6;
constexpr int kPairAccStages = 2;                                 // 256-column accumulators
constexpr int kPairTmemCols = kPairAccStages * kBN;
constexpr int kPairBars = 2 * kPairStages + 2 * kPairAccStages + 1;
constexpr uint32_t kPairSmemBytes =
    kPairStages * kPairStageBytes + kStagingBytes + kPairBars * 8 + 16;
static_assert(kPairSmemBytes <= 232448, "shared memory budget of one sm_103 CTA");
static_assert(kPairAccStages >= 1 && kPairAccStages <= 2, "TMEM holds two 256-column accumulators");
constexpr uint32_t kPairIdescBN = idesc_bf16_f32(kPairBM, kBN, /*A MN-major*/ false, /*B MN-major*/ true);
constexpr uint32_t kPairIdescWt = idesc_bf16_f32(kPairBM, kBN, false, false);

// GemmParams as the 1-SM kernel reads them, with m_tiles counting 256-row
// pair tiles, no cluster or Ozaki fields, and either splits == 1 or a folded
// split (p.fold: the unit is a whole tile whose K segments fill one
// accumulator each, summed by the epilogue in the order 0..splits-1 with the
// reduction kernel's FP32 additions, as in the 1-SM kernel).  kWt: W [N, K]
// (K-major, boxes of 64 k x 128 rows); otherwise B [K, N] (N-major, boxes of
// 64 columns x 64 k-rows).  kFp8: 8-bit float operands, both K-major (kWt): a
// K block is 128 elements, still 128 bytes per row, consumed by four
// instructions of K = 32 (kind::f8f6f4) -- shared-memory layout and
// descriptors byte for byte those of BF16.
template <int kOut, bool kWt, bool kFp8 = false>
__global__ void __launch_bounds__(kNumThreads, 1)
    bigemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmC, const GemmParams p) {
    static_assert(kOut == kOutF32 || kOut == kOutBF16 || kOut == kOutOzaki,
                  "the 2-SM kernel writes C directly or adds Ozaki slice pairs");
    static_assert(!kFp8 || kWt, "8-bit operands are read K-major only");
    static_assert(kOut != kOutOzaki || (!kWt && !kFp8), "Ozaki slices: bf16, B [K, N]");
    constexpr int kKB = kFp8 ? 128 : kBK;  // elements per K block (128 bytes per row)
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // Both CTAs of a pair have the same layout, so both stop here or neither
    // does (before any barrier, allocation or remote access).
    const uint32_t base = smem_addr(smem_raw);
    if (base & 1023u) {
        if (threadIdx.x == 0) atomicOr(p.status, kErrSmemAlign);
        return;
    }
    const uint32_t sA = base;                                    // stage s: sA + s * kABytes
    const uint32_t sB = base + kPairStages * kABytes;            // stage s: sB + s * kPairBBytes
    const uint32_t sOut = base + kPairStages * kPairStageBytes;  // epilogue staging boxes
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw + kPairStages * kPairStageBytes + kStagingBytes);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kPairBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const uint32_t bar0 = smem_addr(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kPairStages + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * kPairStages + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * kPairStages + kPairAccStages + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * kPairStages + 2 * kPairAccStages);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank() & 1u;  // 0: issues the pair's instructions
    const int pair_id = static_cast<int>(blockIdx.x >> 1);
    const int n_pairs = static_cast<int>(gridDim.x >> 1);

    if (warp == 2 && lane == 0) {
        for (int s = 0; s < kPairStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < kPairAccStages; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), 2 * kEpilogueThreads);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();  // release.cluster: visible to the peer's arrivals
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmC);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_addr(tmem_slot), kPairTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_arrive_release();
    cluster_wait_acquire();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    // global memory is touched only after the previous kernel has completed
    grid_dependency_wait();

    // Ozaki scheme: the slice pairs p + q < oz_d this product enumerates (with
    // Fast Mode's automatic d, the largest per-element d, that of the least
    // row mass and the least column mass -- as in the 1-SM kernel).
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
    // work items: tiles, or (slice pair, tile) items pair-major for Ozaki
    const int n_work = (kOut == kOutOzaki) ? p.units * oz_pairs : p.units;

    if (warp < kEpilogueWarp0) {
        regs_release_to<kFrontRegs>();
        if (warp == 0 && lane == 0) {
            // ------------------------------------------------ TMA producer --
            // (both CTAs: this CTA's rows of A and columns of B)
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued_mask = 0, issued_parity = 0;
            bool ok = true;
            int pa = 0, pb = 0, pk = 0;  // Ozaki: slice pair pk is (pa, pb)
            for (int L = pair_id; ok && L < n_work; L += n_pairs) {
                int u = L, a_off = 0, b_off = 0;
                if constexpr (kOut == kOutOzaki) {
                    // rows pa * M + m0 of the A slices, rows pb * oz_kpad + k of the B slices
                    const int pair = L / p.units;
                    u = L - pair * p.units;
                    for (; pk < pair; ++pk) ozaki_next_pair(p, oz_d, pa, pb);
                    a_off = pa * p.M;
                    b_off = pb * p.oz_kpad;
                }
                int mt, nt, seg;
                unit_coords(p, u, mt, nt, seg);
                const int m0 = mt * kPairBM + static_cast<int>(rank) * kBM + a_off;
                const int nb0 = nt * kBN + static_cast<int>(rank) * (kBN / 2);
                for (int kb = 0; kb < p.kb_total; ++kb) {
                    if (!wait_bounded<true>(empty_bar(stage), phase ^ 1u, abort_flag, p.status,
                                            kErrWaitProducer)) {
                        ok = false;
                        break;
                    }
                    // CTA 0's barrier counts both CTAs' bytes of the stage
                    const uint32_t fb = map_shared_rank(full_bar(stage), 0u);
                    if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), 2 * kPairStageBytes);
                    tma_load_2d_pair(sA + stage * kABytes, &tmA, fb, kb * kKB, m0);
                    if constexpr (kWt) {
                        tma_load_2d_pair(sB + stage * kPairBBytes, &tmB, fb, kb * kKB, nb0);
                    } else {
#pragma unroll
                        for (int c = 0; c < 2; ++c)
                            tma_load_2d_pair(sB + stage * kPairBBytes + c * kBChunkBytes, &tmB, fb,
                                             nb0 + c * static_cast<int>(kBChunkCols), b_off + kb * kBK);
                    }
                    issued_mask |= 1u << stage;
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == kPairStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            grid_launch_dependents();
            // No copy of this CTA may be in flight when it exits.  CTA 0 waits
            // for the last phase it armed on every stage (those phases count
            // CTA 1's bytes too); CTA 1 cannot see its loads complete, so it
            // waits until CTA 0's instructions have consumed its last load of
            // every stage -- in a run that gave up early, until the bounded wait
            // expires, long after any load has landed.
            // (after one wait has run out, every load has had its 2 s to land)
            bool waited_out = false;
            for (int s = 0; s < kPairStages; ++s)
                if (!waited_out && (issued_mask & (1u << s)))
                    waited_out = !wait_bounded<true>(rank == 0 ? full_bar(s) : empty_bar(s),
                                                     (issued_parity >> s) & 1u, abort_flag, p.status,
                                                     kErrWaitDrain, /*honour_abort=*/false);
        } else if (warp == 1 && lane == 0 && rank == 0) {
            // ------------------------------------------------- MMA issuer --
            const uint32_t idesc = kFp8 ? p.idesc_fp8 : (kWt ? kPairIdescWt : kPairIdescBN);
            int stage = 0;
            uint32_t phase = 0;
            int t = 0;
            bool ok = true;
            const int nseg = p.fold ? p.splits : 1;
            for (int u = pair_id; ok && u < n_work; u += n_pairs) {
              for (int sg = 0; ok && sg < nseg; ++sg, ++t) {
                // one accumulator per K segment (the whole of K when unsplit)
                const int kb0 = p.fold ? sg * p.kb_per_split : 0;
                const int kb1 = p.fold ? min(kb0 + p.kb_per_split, p.kb_total) : p.kb_total;
                const int acc = t % kPairAccStages;
                const uint32_t acc_phase = static_cast<uint32_t>(t / kPairAccStages) & 1u;
                if (!wait_bounded<true>(tempty_bar(acc), acc_phase ^ 1u, abort_flag, p.status,
                                        kErrWaitMma)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_bounded<true>(full_bar(stage), phase, abort_flag, p.status, kErrWaitMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = sA + stage * kABytes;
                    const uint32_t b0 = sB + stage * kPairBBytes;
#pragma unroll
                    for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
                        const uint64_t ad = smem_desc_sw128(a0 + kk * kUmmaK * 2, 16, 1024);
                        // W half: 128 rows of 128 bytes (K-major, like A); B half:
                        // two 64-column chunks, 16 k-rows = 2 KiB per step.
                        const uint64_t bd = kWt ? smem_desc_sw128(b0 + kk * kUmmaK * 2, 16, 1024)
                                                : smem_desc_sw128(b0 + kk * kUmmaK * 128, kBChunkBytes, 1024);
                        if constexpr (kFp8)
                            mma_fp8_pair(d_tmem, ad, bd, idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
                        else
                            mma_bf16_pair(d_tmem, ad, bd, idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
                    }
                    // stage s is free again in both CTAs once these have read it
                    mma_commit_pair(empty_bar(stage));
                    mma_commit_pair(map_shared_rank(empty_bar(stage), 1u));
                    if (++stage == kPairStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit_pair(tfull_bar(acc));
                mma_commit_pair(map_shared_rank(tfull_bar(acc), 1u));
              }
            }
            // every instruction completes before the TMEM and the stages are released
            mma_commit_pair(drain_bar);
            wait_bounded(drain_bar, 0, abort_flag, p.status, kErrWaitDrain, /*honour_abort=*/false);
        }
    } else {
        regs_grow_to<kEpilogueRegs>();
        // ------------------------------------------------------ epilogue --
        // As in the 1-SM kernel: warp w reads TMEM lanes 32 (w % 4) .. +31 (this
        // CTA's tile rows) and the 128 columns of half (w - 4) / 4, in blocks
        // of 32 x 32 staged for TMA stores.
        const int q = warp & 3;
        const int h = (warp - kEpilogueWarp0) >> 2;
        const int per_warp = p.epi_boxes;
        const int batch = p.epi_batch;
        const int slots = per_warp / batch;
        constexpr uint32_t kBox = (kOut == kOutBF16) ? kStageBufBytes / 2 : kStageBufBytes;
        const uint32_t my_boxes = sOut + static_cast<uint32_t>((q * 2 + h) * per_warp) * kBox;
        uint32_t nbat = 0;
        int t = 0;
        const auto release_acc = [&](int acc) {
            tc_fence_before();
            if (rank == 0) mbar_arrive(tempty_bar(acc));
            else mbar_arrive_remote(map_shared_rank(tempty_bar(acc), 0u));
        };
        if constexpr (kOut == kOutOzaki) {
            // ---- Ozaki scheme, as in the 1-SM kernel: for the item's slice
            // pair (pa, pb), C[row][col] += 2^e * P (P the exact FP32 slice-pair
            // product, e = c_a^(pa)[row] + c_b^(pb)[col]), the first pair
            // starting the sum at +0.0.  This CTA's half of a pair tile is a
            // 128 x 256 tile of C with its own count: a warp adds pair k into
            // its 32 rows once the count shows that the 8 warps of that half
            // (whichever pair of CTAs ran it) have added pair k - 1, then
            // raises it.  A half with no rows neither waits nor counts.
            double* C = static_cast<double*>(p.out);
            const int step = p.oz_beta + 1;
            const int tiles128 = ((p.M + kBM - 1) / kBM) * p.n_tiles;
            int* const grid_abort = p.oz_count + tiles128;  // the launch's abort word
            int pa = 0, pb = 0, pk = 0;
            for (int L = pair_id; L < n_work; L += n_pairs, ++t) {
                const int pair = L / p.units, u = L - pair * p.units;
                for (; pk < pair; ++pk) ozaki_next_pair(p, oz_d, pa, pb);
                int mt, nt, seg;
                unit_coords(p, u, mt, nt, seg);
                const int half = 2 * mt + static_cast<int>(rank);
                const bool has_rows = half * kBM < p.M;
                int* const count = p.oz_count + half * p.n_tiles + nt;
                const int m0 = half * kBM + q * 32, n0 = nt * kBN;
                const int row = m0 + lane;
                const bool row_ok = row < p.M;
                const int acc = t % kPairAccStages;
                const uint32_t acc_phase = static_cast<uint32_t>(t / kPairAccStages) & 1u;
                if (!wait_bounded<true>(tfull_bar(acc), acc_phase, abort_flag, p.status, kErrWaitEpilogue))
                    break;
                tc_fence_after();
                if (pair > 0 && has_rows) {
                    bool in_order = true;
                    if (lane == 0)
                        in_order = wait_count_bounded(count, pair * kEpilogueWarps, abort_flag, grid_abort,
                                                      p.status);
                    in_order = __shfl_sync(0xffffffffu, in_order ? 1 : 0, 0) != 0;
                    if (!in_order) {
                        release_acc(acc);
                        break;
                    }
                    // every lane acquires the count itself (its loads of C come
                    // after the stores of the previous pair)
                    (void)ld_acquire_gpu(count);
                }
                if (m0 < p.M) {
                    const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                           static_cast<uint32_t>(acc * kBN);
                    const int e_pair = row_ok ? (p.oz_ca[row] - pa * step) - pb * step : 0;
                    OzakiFastRow fast = ozaki_fast_row(p.oz_fast ? p.oz_tb : nullptr,
                                                       (p.oz_fast && row_ok) ? p.oz_ta[row] : 0ull,
                                                       (pa + pb) * step, p.oz_need0);
#pragma unroll 1
                    for (int i = 0; i < 4; ++i) {
                        uint32_t r[32];
                        tmem_ld_32x32b_x32(tbase + (h * 4 + i) * 32, r);
                        tmem_ld_wait();
                        if (i == 3) release_acc(acc);  // the accumulator is no longer needed
                        const int col0 = n0 + (h * 4 + i) * 32;
                        if (p.oz_fast) fast.tb = p.oz_tb + col0;  // 256-byte aligned: col0 % 32 == 0
                        if (col0 + 32 <= p.N && p.ld_out >= kOzStagedMinLd)
                            ozaki_accumulate_block_staged(
                                C + static_cast<int64_t>(m0) * p.ld_out + col0, p.ld_out, min(32, p.M - m0),
                                p.oz_cb + col0, e_pair, r, pair == 0, fast,
                                reinterpret_cast<double*>(smem_raw + (sOut - base)) + (q * 2 + h) * 512, lane);
                        else if (row_ok && col0 < p.N)
                            ozaki_accumulate_block(C + static_cast<int64_t>(row) * p.ld_out + col0, p.oz_cb + col0,
                                                   min(32, p.N - col0), e_pair, r, pair == 0, fast, p.oz_c32 != 0);
                    }
                } else {
                    release_acc(acc);
                }
                if (has_rows) {
                    // this warp's part of the pair is in C: count it
                    __threadfence();
                    __syncwarp();
                    if (lane == 0) atomicAdd(count, 1);
                }
            }
        } else if (p.fold) {
            // ---- folded tiles: sum = w_0, then sum = sum + w_s for s = 1 ..
            // splits-1 (FP32, round to nearest even) in 128 registers, then the
            // scale, the bias and the stores -- the 1-SM fold's arithmetic in its
            // order.  The host folds only when every warp with rows stores one
            // block per batch (p.epi_batch == 1).
            for (int u = pair_id; u < p.units; u += n_pairs) {
                int mt, nt, seg;
                unit_coords(p, u, mt, nt, seg);
                const int m0 = mt * kPairBM + static_cast<int>(rank) * kBM + q * 32, n0 = nt * kBN;
                const int nchunks = min(h * 4 + 4, min(kBN / 32, (p.N - n0 + 31) / 32));
                uint32_t sum[128];
                bool ok = true;
#pragma unroll 1
                for (int sg = 0; sg < p.splits; ++sg, ++t) {
                    const int acc = t % kPairAccStages;
                    const uint32_t acc_phase = static_cast<uint32_t>(t / kPairAccStages) & 1u;
                    if (!wait_bounded<true>(tfull_bar(acc), acc_phase, abort_flag, p.status,
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
                                        sum[32 * i + j] = __float_as_uint(
                                            __fadd_rn(__uint_as_float(sum[32 * i + j]), __uint_as_float(w[j])));
                                }
                            }
                        }
                    }
                    release_acc(acc);
                }
                if (!ok) break;
                if (m0 < p.M) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (h * 4 + i < nchunks)
                            emit_blocks<kOut, 1>(p, &tmC, sum + 32 * i, 1, h * 4 + i, n0, m0, seg, lane,
                                                 my_boxes, 1, slots, nbat);
                }
            }
        }
        if constexpr (kOut != kOutOzaki) {
          for (int u = pair_id; !p.fold && u < p.units; u += n_pairs, ++t) {
              int mt, nt, seg;
              unit_coords(p, u, mt, nt, seg);
              const int m0 = mt * kPairBM + static_cast<int>(rank) * kBM + q * 32, n0 = nt * kBN;
              const int nchunks = min(h * 4 + 4, min(kBN / 32, (p.N - n0 + 31) / 32));
              const int acc = t % kPairAccStages;
              const uint32_t acc_phase = static_cast<uint32_t>(t / kPairAccStages) & 1u;
              if (!wait_bounded<true>(tfull_bar(acc), acc_phase, abort_flag, p.status, kErrWaitEpilogue))
                  break;
              tc_fence_after();
              bool released = false;
              if (m0 < p.M) {
                  const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                         static_cast<uint32_t>(acc * kBN);
#pragma unroll 1
                  for (int c0 = h * 4; c0 < nchunks; c0 += batch) {
                      const int nb = min(batch, nchunks - c0);
                      uint32_t r[kMaxBatch * 32];
                      if (batch == 4) tmem_ld_32x32b_x128(tbase + c0 * 32, r);
                      else if (batch == 2) tmem_ld_32x32b_x64(tbase + c0 * 32, r);
                      else tmem_ld_32x32b_x32(tbase + c0 * 32, *reinterpret_cast<uint32_t(*)[32]>(r));
                      tmem_ld_wait();
                      if (c0 + nb >= nchunks) {
                          release_acc(acc);
                          released = true;
                      }
                      emit_blocks<kOut, kMaxBatch>(p, &tmC, r, nb, c0, n0, m0, seg, lane, my_boxes, batch,
                                                   slots, nbat);
                  }
              }
              if (!released) release_acc(acc);
          }
        }
        if (lane == 0) bulk_wait_group<0>();
        __syncwarp();
    }

    // CTA 0's instructions are complete (its MMA thread passed the drain
    // wait) before either CTA releases its TMEM or leaves.
    tc_fence_before();
    cluster_arrive_release();
    cluster_wait_acquire();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kPairTmemCols);
    }
}

}  // namespace bigemm
