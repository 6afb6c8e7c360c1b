// bigemm.cu -- host side of libbigemm.so: argument checks, tensor-map
// encoding, launches, and the C ABI declared in include/bigemm.h.
//
// The library allocates no device memory and never synchronises (except in
// bigemm_device_status, which exists to read the device error word).

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/bigemm.h"
#include "kernels.cuh"
#include "ozaki.cuh"
#include "pair.cuh"
#include "skinny.cuh"

namespace bigemm {

// Device-side error word: bits set by a kernel whose bounded wait expired.
__device__ unsigned g_device_status = 0;

static_assert(kBK == BIGEMM_BLOCK_K, "header and kernel disagree on BLOCK_K");
static_assert(kBM == BIGEMM_TILE_M && kBN == BIGEMM_TILE_N, "header and kernel disagree on tiles");

namespace {

thread_local int g_last_launches = 0;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

struct DeviceInfo {
    bool ready = false;
    bool supported = false;
    int sm_count = 0;
    unsigned* status = nullptr;
    // clusters of S GEMM CTAs that can be resident at once, S = 0..8 (0: none)
    int max_clusters[9] = {0, 0, 0, 0, 0, 0, 0, 0, 0};
    // CTA pairs of the 2-SM kernel that can be resident at once (0: never used)
    int pair_clusters = 0;
};

constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
DeviceInfo g_dev[kMaxDevices];

// Per-device set-up with that device current: capability check, the shared
// memory opt-in of every kernel, and the address of the device error word.
bigemm_status device_info(const DeviceInfo** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return BIGEMM_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return BIGEMM_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return BIGEMM_ERR_CUDA;
        d.supported = (major == 10 && minor == 3);
        d.sm_count = sms;
        if (d.supported) {
            // Besides the shared-memory opt-in: a GEMM kernel whose warpgroups
            // re-divide their registers (setmaxnreg: the direct-output and Ozaki
            // epilogues) must have been compiled with kLaunchRegs registers per
            // thread, the allocation that re-division assumes; with fewer, the
            // epilogue's register increase could never be granted.
            const auto opt_in = [](const void* fn, bool split_regs, uint32_t smem) {
                cudaFuncAttributes fa;
                if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess) return BIGEMM_ERR_CUDA;
                if ((split_regs && fa.numRegs < kLaunchRegs) || fa.maxThreadsPerBlock < kNumThreads)
                    return BIGEMM_ERR_UNSUPPORTED;
                return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            static_cast<int>(smem)) == cudaSuccess
                           ? BIGEMM_OK
                           : BIGEMM_ERR_CUDA;
            };
            const struct {
                const void* fn;
                bool split_regs;
                uint32_t smem;
            } kernels[] = {
                {(const void*)bigemm_tc_kernel<kOutF32, false, false>, true, kSmemBytes},
                {(const void*)bigemm_tc_kernel<kOutBF16, false, false>, true, kSmemBytes},
                {(const void*)bigemm_tc_kernel<kOutSlices, false, false>, false, kSmemBytes},
                {(const void*)bigemm_tc_kernel<kOutAtomic, false, false>, false, kSmemBytes},
                {(const void*)bigemm_tc_kernel<kOutF32, true, false>, true, kSmemBytes},
                {(const void*)bigemm_tc_kernel<kOutBF16, true, false>, true, kSmemBytes},
                {(const void*)bigemm_tc_kernel<kOutSlices, true, false>, false, kSmemBytes},
                {(const void*)bigemm_tc_kernel<kOutF32, true, true>, true, kSmemBytes},
                {(const void*)bigemm_tc_kernel<kOutBF16, true, true>, true, kSmemBytes},
                {(const void*)bigemm_tc_kernel<kOutSlices, true, true>, false, kSmemBytes},
                {(const void*)bigemm_tc_kernel<kOutOzaki, false, false>, true, kSmemBytes},
                {(const void*)bigemm_pair_kernel<kOutF32, false>, true, kPairSmemBytes},
                {(const void*)bigemm_pair_kernel<kOutBF16, false>, true, kPairSmemBytes},
                {(const void*)bigemm_pair_kernel<kOutF32, true>, true, kPairSmemBytes},
                {(const void*)bigemm_pair_kernel<kOutBF16, true>, true, kPairSmemBytes},
                {(const void*)bigemm_pair_kernel<kOutF32, true, true>, true, kPairSmemBytes},
                {(const void*)bigemm_pair_kernel<kOutBF16, true, true>, true, kPairSmemBytes},
                {(const void*)bigemm_pair_kernel<kOutOzaki, false>, true, kPairSmemBytes},
#define BIGEMM_NARROW_KERNELS(TN)                                                                  \
    {(const void*)bigemm_tc_kernel<kOutF32, false, false, TN>, true, Tile<TN>::kSmemBytes},        \
        {(const void*)bigemm_tc_kernel<kOutBF16, false, false, TN>, true, Tile<TN>::kSmemBytes},   \
        {(const void*)bigemm_tc_kernel<kOutSlices, false, false, TN>, false, Tile<TN>::kSmemBytes}, \
        {(const void*)bigemm_tc_kernel<kOutAtomic, false, false, TN>, false, Tile<TN>::kSmemBytes}, \
        {(const void*)bigemm_tc_kernel<kOutF32, true, false, TN>, true, Tile<TN>::kSmemBytes},     \
        {(const void*)bigemm_tc_kernel<kOutBF16, true, false, TN>, true, Tile<TN>::kSmemBytes},    \
        {(const void*)bigemm_tc_kernel<kOutSlices, true, false, TN>, false, Tile<TN>::kSmemBytes}
                BIGEMM_NARROW_KERNELS(128),
                BIGEMM_NARROW_KERNELS(64),
#undef BIGEMM_NARROW_KERNELS
            };
            for (const auto& k : kernels) {
                const bigemm_status st = opt_in(k.fn, k.split_regs, k.smem);
                if (st != BIGEMM_OK) return st;
            }
            // the few-row kernels: up to the wide kernel's shared memory
            const void* skinny[] = {(const void*)bigemm_skinny_kernel<kOutF32, false>,
                                    (const void*)bigemm_skinny_kernel<kOutBF16, false>,
                                    (const void*)bigemm_skinny_kernel<kOutF32, true>,
                                    (const void*)bigemm_skinny_kernel<kOutBF16, true>};
            for (const void* fn : skinny)
                if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes)) != cudaSuccess)
                    return BIGEMM_ERR_CUDA;
            void* sym = nullptr;
            if (cudaGetSymbolAddress(&sym, g_device_status) != cudaSuccess) return BIGEMM_ERR_CUDA;
            d.status = static_cast<unsigned*>(sym);
            // How many clusters of S one-CTA-per-SM GEMM blocks fit at once (all
            // instantiations have the same block size, registers and shared
            // memory).  A failed query leaves 0: that split never clusters.
            for (int S = 2; S <= 8; ++S) {
                cudaLaunchConfig_t cfg = {};
                cfg.gridDim = dim3(static_cast<unsigned>(S));
                cfg.blockDim = dim3(kNumThreads);
                cfg.dynamicSmemBytes = kSmemBytes;
                cudaLaunchAttribute attr[1];
                attr[0].id = cudaLaunchAttributeClusterDimension;
                attr[0].val.clusterDim.x = static_cast<unsigned>(S);
                attr[0].val.clusterDim.y = 1;
                attr[0].val.clusterDim.z = 1;
                cfg.attrs = attr;
                cfg.numAttrs = 1;
                int n = 0;
                if (cudaOccupancyMaxActiveClusters(
                        &n, (const void*)bigemm_tc_kernel<kOutF32, false, false>, &cfg) != cudaSuccess) {
                    (void)cudaGetLastError();
                    n = 0;
                }
                d.max_clusters[S] = n;
            }
            {
                cudaLaunchConfig_t cfg = {};
                cfg.gridDim = dim3(2);
                cfg.blockDim = dim3(kNumThreads);
                cfg.dynamicSmemBytes = kPairSmemBytes;
                cudaLaunchAttribute attr[1];
                attr[0].id = cudaLaunchAttributeClusterDimension;
                attr[0].val.clusterDim.x = 2;
                attr[0].val.clusterDim.y = 1;
                attr[0].val.clusterDim.z = 1;
                cfg.attrs = attr;
                cfg.numAttrs = 1;
                int n = 0;
                if (cudaOccupancyMaxActiveClusters(&n, (const void*)bigemm_pair_kernel<kOutF32, false>,
                                                   &cfg) != cudaSuccess) {
                    (void)cudaGetLastError();
                    n = 0;
                }
                d.pair_clusters = n;
            }
        }
        d.ready = true;
    }
    if (!d.supported) return BIGEMM_ERR_UNSUPPORTED;
    *out = &d;
    return BIGEMM_OK;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// A split product that fills the GPU with whole tiles sums its K segments in
// the CTA that owns the tile (GemmParams::fold): no workspace, no second
// kernel, and the same additions in the same order as the reduction kernel.
// A rule on the shape alone; the folded epilogue assumes one 32-column block
// per store batch, which every M >= BIGEMM_FOLD_MIN_ROWS has.
static_assert(epi_batch_for(BIGEMM_FOLD_MIN_ROWS) == 1 && epi_boxes_for(BIGEMM_FOLD_MIN_ROWS) == 1,
              "folded epilogue layout");
bool folds(int64_t M, int64_t N, int splits) {
    if (splits <= 1 || M < BIGEMM_FOLD_MIN_ROWS || N <= 0) return false;
    return ceil_div(M, kBM) * ceil_div(N, kBN) >= BIGEMM_FOLD_MIN_TILES;
}

// A product of at most kSkMaxM rows with bf16 operands and at most
// kSkMaxCluster K segments runs bigemm_skinny_kernel, which forms
// its split sum inside the launch: no workspace, one kernel.  A rule on the
// shape alone (a cluster of up to 8 CTAs always fits); the same bits as the
// other paths.
static_assert(kSkMaxM == BIGEMM_SKINNY_MAX_ROWS && kSkMaxCluster == BIGEMM_SKINNY_MAX_SPLIT,
              "header and kernel disagree on the few-row rule");
bool skinny(int64_t M, int splits, bool fp8) {
    return !fp8 && M >= 1 && M <= kSkMaxM && splits >= 1 && splits <= kSkMaxCluster;
}

// Tile width of a product (kBN = 256, or 128 / 64).  The wide tile unless
// its units (tiles x K segments) would occupy fewer than half of the SMs and
// each unit streams at least kNarrowMinBlocks K blocks: then each unit's K
// loop, not HBM, sets the pace -- an SM takes in at most about 140 GB/s, and
// a unit's dependent MMAs run one after another -- and narrower tiles put
// more SMs to work with fewer bytes each, down to the MMA chain's floor: the
// widest width whose units reach half the SMs, else 64.  Short segments keep
// the wide tile: their time is launch and pipeline latency, which narrower
// tiles do not shorten.  Folded and 8-bit products are always wide.  Speed
// only: every width forms every sum the same way.
constexpr int kNarrowMinBlocks = 32;

int tile_width(int64_t M, int64_t N, int splits, int kb_per_split, bool fold, bool fp8,
               int sm_count) {
    if (fp8 || fold || M <= 0 || N <= 0 || kb_per_split < kNarrowMinBlocks) return kBN;
    const int64_t m_tiles = ceil_div(M, kBM);
    const int64_t half = sm_count / 2;
    if (m_tiles * ceil_div(N, kBN) * splits >= half) return kBN;
    if (m_tiles * ceil_div(N, 128) * splits >= half) return 128;
    return 64;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// An unsplit (or folded) product of at least 256 rows with wide tiles, bf16
// or 8-bit floats, can run on CTA pairs (bigemm_pair_kernel): 256 x 256
// tiles, each CTA loading half of the A and B panels.  A pair instruction takes about as long per SM as a
// 1-SM one, so the gain is the lighter loads of the main loop (measured 3 to
// 15 %), while a pair's start and finish cost more: the rule takes the
// 2-SM kernel once the pair tiles fill at least two waves of the device's
// pairs.  Every output element is the same accumulation chain either way.
// bigemm_set_pair_mode: 0 never, 1 by this rule, 2 for every eligible shape
// (comparisons and tests).
std::atomic<int> g_pair_mode{1};

// A split product qualifies when it folds (folds(): then every 128-row tile
// of it would also sum its segments in the CTA).
bool pairs_tiles(int64_t M, int64_t N, int splits, int tile_n, int pair_clusters) {
    const int mode = g_pair_mode.load(std::memory_order_relaxed);
    if (mode == 0 || M < kPairBM || tile_n != kBN || pair_clusters <= 0) return false;
    if (splits != 1 && !folds(M, N, splits)) return false;
    return mode == 2 || ceil_div(M, kPairBM) * ceil_div(N, kBN) >= 2 * static_cast<int64_t>(pair_clusters);
}

// kb_elems: elements per K block -- 64 for BF16, 128 for 8-bit floats (both
// 128 bytes per row).
int max_split(int64_t K, int kb_elems = kBK) {
    if (K <= 0) return 1;
    const int64_t kb = ceil_div(K, kb_elems);
    return kb > INT_MAX ? INT_MAX : static_cast<int>(kb);
}

int default_split(int64_t K) {
    int64_t cap = K / 512;
    if (cap > 16) cap = 16;
    int s = 1;
    while (2 * s <= cap) s *= 2;
    return s;
}

// Effective split and blocks per segment; 0 when split_k is invalid.
int effective_split(int64_t K, int split_k, int* blocks_per_split, int kb_elems = kBK) {
    if (K < 0) return 0;
    if (split_k == 0) split_k = default_split(K);
    if (split_k < 1 || split_k > max_split(K, kb_elems)) return 0;
    if (K == 0) {
        if (blocks_per_split) *blocks_per_split = 0;
        return 1;
    }
    const int64_t kb = ceil_div(K, kb_elems);
    const int64_t L = ceil_div(kb, split_k);
    if (blocks_per_split) *blocks_per_split = static_cast<int>(L);
    return static_cast<int>(ceil_div(kb, L));
}

int64_t ws_ld_of(int64_t N) { return ceil_div(N, 4) * 4; }

// Bytes of `slices` workspace slices, or SIZE_MAX on overflow.
size_t slice_bytes(int64_t M, int64_t N, int slices) {
    const unsigned __int128 b = static_cast<unsigned __int128>(slices) *
                                static_cast<unsigned __int128>(M) *
                                static_cast<unsigned __int128>(ws_ld_of(N)) * 4u;
    if (b > static_cast<unsigned __int128>(SIZE_MAX)) return SIZE_MAX;
    return static_cast<size_t>(b);
}

// A general strided view: rank dimensions, innermost first (dims[0] elements
// contiguous), strides[i] = bytes between consecutive indices of dimension
// i + 1, boxes of box[0..rank-1].
bool encode_view(CUtensorMap* map, CUtensorMapDataType dtype, const void* ptr, int rank,
                 const int64_t* dims, const int64_t* strides, const uint32_t* box,
                 CUtensorMapSwizzle swizzle) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr || rank < 1 || rank > 5) return false;
    cuuint64_t gdims[5], gstr[4];
    cuuint32_t gbox[5], estr[5];
    for (int i = 0; i < rank; ++i) {
        gdims[i] = static_cast<cuuint64_t>(dims[i]);
        gbox[i] = box[i];
        estr[i] = 1;
        if (i + 1 < rank) gstr[i] = static_cast<cuuint64_t>(strides[i]);
    }
    return fn(map, dtype, static_cast<cuuint32_t>(rank), const_cast<void*>(ptr), gdims, gstr, gbox, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Grouped output views for one TMA store per epilogue batch (N a multiple of
// 32): {32 columns, M rows, N/32 column groups [, slices]} -- the staging
// boxes of a batch sit group after group in shared memory.  Returns false if
// N is not a multiple of 32 or the driver refuses the view; the caller then
// uses the plain 2-D / 3-D maps with one store per 32 x 32 block.
bool encode_out_grouped(CUtensorMap* m, CUtensorMapDataType dtype, uint32_t esize, void* ptr,
                        int64_t M, int64_t N, int64_t ld, int splits, int64_t slice, int batch) {
    if (N % 32 != 0) return false;
    const CUtensorMapSwizzle sw = esize == 4 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    const int64_t dims[4] = {32, M, N / 32, splits};
    const int64_t strides[3] = {ld * static_cast<int64_t>(esize), 32 * static_cast<int64_t>(esize),
                                slice * static_cast<int64_t>(esize)};
    const uint32_t box[4] = {32, 32, static_cast<uint32_t>(batch), 1};
    return encode_view(m, dtype, ptr, splits > 0 ? 4 : 3, dims, strides, box, sw);
}

// A row-major tensor of `rank` (2 or 3) dimensions, innermost first: dims[0]
// contiguous elements, dims[1] rows `ld` elements apart, dims[2] slices
// `slice` elements apart.  Boxes of box[0] x box[1] (x 1).
bool encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t esize, const void* ptr,
                  int rank, const int64_t* dims, int64_t ld, int64_t slice, const uint32_t* box,
                  CUtensorMapSwizzle swizzle) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t gdims[3] = {static_cast<cuuint64_t>(dims[0]), static_cast<cuuint64_t>(dims[1]),
                           static_cast<cuuint64_t>(rank > 2 ? dims[2] : 1)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * esize,
                             static_cast<cuuint64_t>(slice) * esize};
    cuuint32_t gbox[3] = {box[0], box[1], 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, dtype, static_cast<cuuint32_t>(rank), const_cast<void*>(ptr), gdims, strides, gbox,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Operand maps: A [M, K] in boxes of 64 k x 128 rows; B [K, N] in boxes of 64
// columns x 64 k-rows, or a weight matrix W [N, K] (wt) in boxes of 64 k x
// tile_n rows; all with the 128-byte swizzle the MMA descriptors use.  The
// second operand again in tile_n x 256 boxes without swizzle, used only to
// warm L2.
// Rows of A a stage loads: the batch rounded up to 32, 64 or 128 (a function of
// M that changes no sum -- the other rows of the 128-row MMA operand are zero).
int a_box_rows(int64_t M) { return M <= 32 ? 32 : (M <= 64 ? 64 : kBM); }

bool encode_operands(CUtensorMap* tmA, CUtensorMap* tmB, CUtensorMap* tmBp, const void* A,
                     const void* B, int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                     bool wt, bool fp8, int tile_n = kBN) {
    // 8-bit operands: a K block of 128 elements is still 128 bytes per row
    const uint32_t kb = fp8 ? 128u : static_cast<uint32_t>(kBK);
    const CUtensorMapDataType dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const uint32_t es = fp8 ? 1u : 2u;
    const int64_t da[2] = {K, M};
    const int64_t db[2] = {wt ? K : N, wt ? N : K};
    const uint32_t ba[2] = {kb, static_cast<uint32_t>(a_box_rows(M))};
    const uint32_t tn = static_cast<uint32_t>(tile_n);
    const uint32_t bb[2] = {wt ? kb : kBChunkCols, wt ? tn : kb};
    const uint32_t bp[2] = {wt ? static_cast<uint32_t>(kPrefetchRows) : tn,
                            wt ? tn : static_cast<uint32_t>(kPrefetchRows)};
    return encode_tiled(tmA, dt, es, A, 2, da, lda, 0, ba, CU_TENSOR_MAP_SWIZZLE_128B) &&
           encode_tiled(tmB, dt, es, B, 2, db, ldb, 0, bb, CU_TENSOR_MAP_SWIZZLE_128B) &&
           encode_tiled(tmBp, dt, es, B, 2, db, ldb, 0, bp, CU_TENSOR_MAP_SWIZZLE_NONE);
}

// Output maps for the epilogue's 32 x 32 TMA stores: fp32 C (128-byte
// swizzle), bf16 C (64-byte swizzle), or the fp32 workspace as a 3-D tensor
// [splits][M][ws_ld] (128-byte swizzle).
bool encode_out_f32(CUtensorMap* m, void* C, int64_t M, int64_t N, int64_t ldc) {
    const int64_t d[2] = {N, M};
    const uint32_t box[2] = {32, 32};
    return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, C, 2, d, ldc, 0, box,
                        CU_TENSOR_MAP_SWIZZLE_128B);
}

bool encode_out_bf16(CUtensorMap* m, void* C, int64_t M, int64_t N, int64_t ldc) {
    const int64_t d[2] = {N, M};
    const uint32_t box[2] = {32, 32};
    return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, C, 2, d, ldc, 0, box,
                        CU_TENSOR_MAP_SWIZZLE_64B);
}

bool encode_out_slices(CUtensorMap* m, void* ws, int64_t M, int64_t N, int splits) {
    const int64_t ld = ws_ld_of(N);
    const int64_t d[3] = {N, M, splits};
    const uint32_t box[2] = {32, 32};
    return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, ws, 3, d, ld, M * ld, box,
                        CU_TENSOR_MAP_SWIZZLE_128B);
}

// A launch with programmatic stream serialisation, and with thread-block
// clusters of `cluster_x` CTAs along x when cluster_x > 1.
template <typename Kernel, typename... Args>
cudaError_t launch_pdl_cluster(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                               unsigned cluster_x, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cluster_x > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = cluster_x;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <typename Kernel, typename... Args>
cudaError_t launch_pdl(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args) {
    return launch_pdl_cluster(kernel, grid, block, smem, stream, 1u, args...);
}

// A bf16 product with narrow tiles (128 or 64 columns; never clustered).
template <int kOut, int kTN>
cudaError_t launch_narrow(bool wt, dim3 g, dim3 blk, cudaStream_t stream, const CUtensorMap& tmA,
                          const CUtensorMap& tmB, const CUtensorMap& tmBp, const CUtensorMap& tmC,
                          const GemmParams& p) {
    constexpr uint32_t smem = Tile<kTN>::kSmemBytes;
    if constexpr (kOut == kOutAtomic) {
        if (wt) return cudaErrorInvalidValue;
        return launch_pdl(bigemm_tc_kernel<kOut, false, false, kTN>, g, blk, smem, stream, tmA, tmB,
                          tmBp, tmC, p);
    } else {
        if (wt)
            return launch_pdl(bigemm_tc_kernel<kOut, true, false, kTN>, g, blk, smem, stream, tmA, tmB,
                              tmBp, tmC, p);
        return launch_pdl(bigemm_tc_kernel<kOut, false, false, kTN>, g, blk, smem, stream, tmA, tmB,
                          tmBp, tmC, p);
    }
}

template <int kOut>
cudaError_t launch_gemm(bool wt, bool fp8, dim3 g, dim3 blk, cudaStream_t stream,
                        const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmBp,
                        const CUtensorMap& tmC, const GemmParams& p, unsigned cluster_x = 1,
                        int tile_n = kBN) {
    if constexpr (kOut != kOutOzaki) {
        if (tile_n != kBN) {
            if (fp8 || cluster_x > 1 || p.fold) return cudaErrorInvalidValue;
            if (tile_n == 128) return launch_narrow<kOut, 128>(wt, g, blk, stream, tmA, tmB, tmBp, tmC, p);
            if (tile_n == 64) return launch_narrow<kOut, 64>(wt, g, blk, stream, tmA, tmB, tmBp, tmC, p);
            return cudaErrorInvalidValue;
        }
    }
    if constexpr (kOut == kOutOzaki) {
        if (wt || fp8) return cudaErrorInvalidValue;  // bfloat16 slices of B [K, N] only
        // A cooperative launch: the CTAs of an Ozaki product wait on one
        // another (a tile's pairs run on different CTAs, in order), so CUDA
        // must start the grid only when all of its CTAs can be resident at
        // once -- also while other kernels, another Ozaki product among
        // them, hold SMs.  (No programmatic serialisation here: the kernel's
        // dependency wait is then a no-op and it starts after its predecessor.)
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = g;
        cfg.blockDim = blk;
        cfg.dynamicSmemBytes = kSmemBytes;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, bigemm_tc_kernel<kOut, false, false>, tmA, tmB, tmBp, tmC, p);
    } else if constexpr (kOut == kOutAtomic) {
        if (wt || fp8) return cudaErrorInvalidValue;  // the contrast exists for bf16 B [K, N] only
        return launch_pdl(bigemm_tc_kernel<kOut, false, false>, g, blk, kSmemBytes, stream, tmA, tmB,
                          tmBp, tmC, p);
    } else {
        if (fp8) {
            if (!wt) return cudaErrorInvalidValue;
            return launch_pdl_cluster(bigemm_tc_kernel<kOut, true, true>, g, blk, kSmemBytes, stream,
                                      cluster_x, tmA, tmB, tmBp, tmC, p);
        }
        if (wt)
            return launch_pdl_cluster(bigemm_tc_kernel<kOut, true, false>, g, blk, kSmemBytes, stream,
                                      cluster_x, tmA, tmB, tmBp, tmC, p);
        return launch_pdl_cluster(bigemm_tc_kernel<kOut, false, false>, g, blk, kSmemBytes, stream,
                                  cluster_x, tmA, tmB, tmBp, tmC, p);
    }
}

enum Mode { kModeF32, kModeBF16, kModePartial, kModeAtomic };

bigemm_status launch_reduce(const DeviceInfo& d, const float* ws, int splits, int64_t M, int64_t N,
                            void* C, int64_t ldc, bool bf16, cudaStream_t stream,
                            const void* bias = nullptr, float scale = 1.0f) {
    const __nv_bfloat16* b = static_cast<const __nv_bfloat16*>(bias);
    const int64_t ws_ld = ws_ld_of(N);
    const int64_t items = M * (ws_ld / 4);
    // One thread per four-column group, all groups in flight at once up to
    // the SMs' thread capacity (16 blocks of 128 per SM); beyond that the
    // threads loop.  A decode-sized sum is bound by the latency of its L2
    // reads, so every read should be issued in the first round: capping the
    // grid at one block per SM made each thread of an M = 64 sum wait for
    // four rounds of reads.
    int64_t blocks = ceil_div(items, kReduceThreads);
    if (blocks > 16LL * d.sm_count) blocks = 16LL * d.sm_count;
    if (blocks < 1) blocks = 1;
    cudaError_t e;
    const dim3 g(static_cast<unsigned>(blocks)), blk(kReduceThreads);
    const int m = static_cast<int>(M), n = static_cast<int>(N);
    if (bf16)
        e = b ? launch_pdl(splitk_reduce_kernel<true, true>, g, blk, 0, stream, ws, C, m, n, ldc, ws_ld, splits, b, scale)
              : launch_pdl(splitk_reduce_kernel<true, false>, g, blk, 0, stream, ws, C, m, n, ldc, ws_ld, splits, b, scale);
    else
        e = b ? launch_pdl(splitk_reduce_kernel<false, true>, g, blk, 0, stream, ws, C, m, n, ldc, ws_ld, splits, b, scale)
              : launch_pdl(splitk_reduce_kernel<false, false>, g, blk, 0, stream, ws, C, m, n, ldc, ws_ld, splits, b, scale);
    return e == cudaSuccess ? BIGEMM_OK : BIGEMM_ERR_CUDA;
}

// A product of at most kSkMaxM rows with at most kSkMaxCluster K segments
// (skinny()): one launch of bigemm_skinny_kernel, a cluster of S CTAs per
// 128 x 256 output tile.
bigemm_status run_skinny(const DeviceInfo& d, bool bf16, const void* A, const void* B, void* C, int64_t M,
                         int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc, int splits,
                         int kb_per_split, bool wt, const void* bias, cudaStream_t stream) {
    const int64_t tiles = ceil_div(N, kBN);
    if (tiles * splits > INT_MAX) return BIGEMM_ERR_ARG;
    CUtensorMap tmA, tmB;
    const int64_t da[2] = {K, M};
    const uint32_t ba[2] = {static_cast<uint32_t>(kBK), static_cast<uint32_t>(sk_a_rows(static_cast<int>(M)))};
    const int64_t db[2] = {wt ? K : N, wt ? N : K};
    const uint32_t bb[2] = {wt ? static_cast<uint32_t>(kBK) : kBChunkCols,
                            wt ? static_cast<uint32_t>(kBN) : static_cast<uint32_t>(kBK)};
    if (!encode_tiled(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, 2, da, lda, 0, ba,
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tiled(&tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, 2, db, ldb, 0, bb,
                      CU_TENSOR_MAP_SWIZZLE_128B))
        return BIGEMM_ERR_CUDA;
    SkinnyParams p;
    std::memset(&p, 0, sizeof(p));
    p.out = C;
    p.ldc = ldc;
    p.w = static_cast<const __nv_bfloat16*>(B);
    p.ldw = ldb;
    p.status = d.status;
    p.bias = static_cast<const __nv_bfloat16*>(bias);
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.splits = splits;
    p.kb_total = static_cast<int>(ceil_div(K, kBK));
    p.kb_per_split = kb_per_split;
    // ring depth: as deep as fits in half an SM's shared memory, so that the
    // next product's CTAs can be resident beside this product's; the ring
    // also holds the partials once the last instruction is done
    const uint32_t stage = sk_stage_bytes(p.M);
    int stages = static_cast<int>(kSkHalfSmBytes / stage);
    if (stages > kSkMaxStages) stages = kSkMaxStages;
    p.stages = stages;
    const dim3 g(static_cast<unsigned>(tiles * splits)), blk(kSkThreads);
    const uint32_t smem = sk_smem_bytes(p.M, stages);
    const unsigned cx = static_cast<unsigned>(splits);
    cudaError_t e;
    if (wt)
        e = bf16 ? launch_pdl_cluster(bigemm_skinny_kernel<kOutBF16, true>, g, blk, smem, stream, cx, tmA, tmB, p)
                 : launch_pdl_cluster(bigemm_skinny_kernel<kOutF32, true>, g, blk, smem, stream, cx, tmA, tmB, p);
    else
        e = bf16 ? launch_pdl_cluster(bigemm_skinny_kernel<kOutBF16, false>, g, blk, smem, stream, cx, tmA, tmB, p)
                 : launch_pdl_cluster(bigemm_skinny_kernel<kOutF32, false>, g, blk, smem, stream, cx, tmA, tmB, p);
    return e == cudaSuccess ? BIGEMM_OK : BIGEMM_ERR_CUDA;
}

// wt: the second operand is a weight matrix W [N, K] (ldb is its row stride);
// otherwise B [K, N].  bias: bf16 [N] added to every row (linear layers), or
// nullptr.
// The 2-SM product (pairs_tiles): A [M, K] in boxes of 64 k x 128 rows, B
// [K, N] in boxes of 64 columns x 64 k-rows or W [N, K] in boxes of 64 k x
// 128 rows (a CTA's half of a 256-column tile), C in 32 x 32 boxes.
bigemm_status run_pair(const DeviceInfo& d, bool bf16, const void* A, const void* B, void* C, int64_t M,
                       int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc, int splits,
                       int kb_per_split, bool wt, const void* bias, float scale, int fp8_fmt_a,
                       int fp8_fmt_b, cudaStream_t stream) {
    const bool fp8 = fp8_fmt_a >= 0;  // 8-bit float operands, W layout
    if (fp8 && !wt) return BIGEMM_ERR_ARG;
    CUtensorMap tmA, tmB, tmBp, tmC;
    std::memset(&tmC, 0, sizeof(tmC));
    if (!encode_operands(&tmA, &tmB, &tmBp, A, B, M, N, K, lda, ldb, wt, fp8, kBN / 2))
        return BIGEMM_ERR_CUDA;
    const int64_t m_tiles = ceil_div(M, kPairBM), n_tiles = ceil_div(N, kBN);
    const int64_t units = m_tiles * n_tiles;
    if (units > INT_MAX) return BIGEMM_ERR_ARG;
    GemmParams p;
    std::memset(&p, 0, sizeof(p));
    p.status = d.status;
    p.out = C;
    p.ld_out = ldc;
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.m_tiles = static_cast<int>(m_tiles);
    p.n_tiles = static_cast<int>(n_tiles);
    p.splits = splits;
    p.kb_total = static_cast<int>(ceil_div(K, fp8 ? 128 : kBK));
    p.kb_per_split = splits > 1 ? kb_per_split : p.kb_total;
    p.fold = splits > 1 ? 1 : 0;
    p.idesc_fp8 = fp8 ? idesc_fp8_f32(kPairBM, kBN, static_cast<uint32_t>(fp8_fmt_a),
                                      static_cast<uint32_t>(fp8_fmt_b))
                      : 0u;
    p.units = static_cast<int>(units);
    p.epi_boxes = epi_boxes_for(static_cast<int>(M));
    p.epi_batch = epi_batch_for(static_cast<int>(M));
    // GROUP_M swizzle over 256-row tiles: the same rows per group as the
    // 1-SM rule (8 pair tile rows once there are four waves, else 4)
    p.group_m = (units >= 4 * static_cast<int64_t>(d.pair_clusters)) ? 8 : 4;
    p.a_rows = kBM;
    p.bias = static_cast<const __nv_bfloat16*>(bias);
    p.scale = scale;
    const CUtensorMapDataType dt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    if (encode_out_grouped(&tmC, dt, bf16 ? 2u : 4u, C, M, N, ldc, 0, 0, p.epi_batch))
        p.grouped = 1;
    else if (!(bf16 ? encode_out_bf16(&tmC, C, M, N, ldc) : encode_out_f32(&tmC, C, M, N, ldc)))
        return BIGEMM_ERR_CUDA;
    // persistent: at most one pair per two SMs, as many as fit at once
    const int64_t pairs = units < d.pair_clusters ? units : d.pair_clusters;
    const dim3 g(static_cast<unsigned>(2 * pairs)), blk(kNumThreads);
    cudaError_t e;
    if (fp8)
        e = bf16 ? launch_pdl_cluster(bigemm_pair_kernel<kOutBF16, true, true>, g, blk, kPairSmemBytes, stream,
                                      2u, tmA, tmB, tmC, p)
                 : launch_pdl_cluster(bigemm_pair_kernel<kOutF32, true, true>, g, blk, kPairSmemBytes, stream,
                                      2u, tmA, tmB, tmC, p);
    else if (bf16)
        e = wt ? launch_pdl_cluster(bigemm_pair_kernel<kOutBF16, true>, g, blk, kPairSmemBytes, stream, 2u,
                                    tmA, tmB, tmC, p)
               : launch_pdl_cluster(bigemm_pair_kernel<kOutBF16, false>, g, blk, kPairSmemBytes, stream, 2u,
                                    tmA, tmB, tmC, p);
    else
        e = wt ? launch_pdl_cluster(bigemm_pair_kernel<kOutF32, true>, g, blk, kPairSmemBytes, stream, 2u,
                                    tmA, tmB, tmC, p)
               : launch_pdl_cluster(bigemm_pair_kernel<kOutF32, false>, g, blk, kPairSmemBytes, stream, 2u,
                                    tmA, tmB, tmC, p);
    return e == cudaSuccess ? BIGEMM_OK : BIGEMM_ERR_CUDA;
}

bigemm_status run_impl(Mode mode, const void* A, const void* B, void* C, int64_t M, int64_t N,
                       int64_t K, int64_t lda, int64_t ldb, int64_t ldc, int split_k, void* ws,
                       size_t ws_bytes, cudaStream_t stream, bool wt = false,
                       const void* bias = nullptr, int fp8_fmt_a = -1, int fp8_fmt_b = -1,
                       float scale = 1.0f, bool selftest_stall = false) {
    // fp8_fmt_a / fp8_fmt_b >= 0: 8-bit float operands (0 = E4M3, 1 = E5M2), W layout
    const bool fp8 = fp8_fmt_a >= 0;
    const int kb_elems = fp8 ? 128 : kBK;
    const int ld_align = fp8 ? 16 : 8;  // elements per 16 bytes
    g_last_launches = 0;
    // ---- sizes and the split
    if (M < 0 || N < 0 || K < 0) return BIGEMM_ERR_ARG;
    if (M > INT_MAX || N > INT_MAX || K > INT_MAX) return BIGEMM_ERR_ARG;
    int kb_per_split = 0;
    const int splits = effective_split(K, split_k, &kb_per_split, kb_elems);
    if (splits == 0) return BIGEMM_ERR_ARG;
    const bool want_c = (mode != kModePartial);
    // ---- pointers and strides (checked even for empty products)
    if (K > 0 && (A == nullptr || B == nullptr)) return BIGEMM_ERR_ARG;
    if (K > 0 && (lda < K || ldb < (wt ? K : N))) return BIGEMM_ERR_ARG;
    if (want_c && (C == nullptr || ldc < N)) return BIGEMM_ERR_ARG;
    if (K > 0 && (!aligned16(A) || !aligned16(B) || lda % ld_align != 0 || ldb % ld_align != 0))
        return BIGEMM_ERR_ALIGN;
    if (want_c) {
        if (!aligned16(C)) return BIGEMM_ERR_ALIGN;
        if (ldc % (mode == kModeBF16 ? 8 : 4) != 0) return BIGEMM_ERR_ALIGN;
    }
    if (bias != nullptr && !aligned16(bias)) return BIGEMM_ERR_ALIGN;
    // ---- workspace
    const bool direct = (mode == kModeF32 || mode == kModeBF16);
    const bool fold = direct && folds(M, N, splits);
    const bool few_rows = direct && skinny(M, splits, fp8);
    const bool need_ws = (mode == kModePartial) || (direct && splits > 1 && !fold && !few_rows);
    if (need_ws) {
        const size_t need = slice_bytes(M, N, splits);
        if (need == SIZE_MAX) return BIGEMM_ERR_ARG;
        if (need > 0 && (ws == nullptr || !aligned16(ws) || ws_bytes < need))
            return BIGEMM_ERR_WORKSPACE;
    }
    if (M == 0 || N == 0) return BIGEMM_OK;

    const DeviceInfo* d = nullptr;
    bigemm_status st = device_info(&d);
    if (st != BIGEMM_OK) return st;
    const int tile_n = tile_width(M, N, splits, kb_per_split, fold, fp8, d->sm_count);
    const int64_t m_tiles = ceil_div(M, kBM);
    const int64_t n_tiles = ceil_div(N, tile_n);
    const int64_t units = m_tiles * n_tiles * (fold ? 1 : splits);
    if (units > INT_MAX) return BIGEMM_ERR_ARG;
    // A split product that is not folded sums its segments inside clusters of
    // `splits` CTAs when all of its clusters can be resident at once (one
    // wave) and its tiles are wide; otherwise through the workspace and the
    // reduction kernel.  Same bits either way; the workspace is required in
    // both cases.
    const bool cluster = direct && !fold && tile_n == kBN && splits >= 2 && splits <= 8 && K > 0 &&
                         m_tiles * n_tiles <= d->max_clusters[splits];
    const bool pair = direct && K > 0 && pairs_tiles(M, N, splits, tile_n, d->pair_clusters);

    // ---- K == 0: the empty sum is +0.0 everywhere (plus the bias, if any)
    if (K == 0 && bias != nullptr) {
        st = launch_reduce(*d, nullptr, 0, M, N, C, ldc, mode == kModeBF16, stream, bias, scale);
        if (st == BIGEMM_OK) g_last_launches = 1;
        return st;
    }
    if (K == 0) {
        cudaError_t e;
        if (mode == kModePartial) {
            e = cudaMemsetAsync(ws, 0, slice_bytes(M, N, 1), stream);
        } else {
            const size_t es = (mode == kModeBF16) ? 2 : 4;
            e = cudaMemset2DAsync(C, static_cast<size_t>(ldc) * es, 0, static_cast<size_t>(N) * es,
                                  static_cast<size_t>(M), stream);
        }
        return e == cudaSuccess ? BIGEMM_OK : BIGEMM_ERR_CUDA;
    }

    if (few_rows) {
        st = run_skinny(*d, mode == kModeBF16, A, B, C, M, N, K, lda, ldb, ldc, splits, kb_per_split, wt,
                        bias, stream);
        if (st == BIGEMM_OK) g_last_launches = 1;
        return st;
    }
    if (pair) {
        st = run_pair(*d, mode == kModeBF16, A, B, C, M, N, K, lda, ldb, ldc, splits, kb_per_split, wt, bias,
                      scale, fp8_fmt_a, fp8_fmt_b, stream);
        if (st == BIGEMM_OK) g_last_launches = 1;
        return st;
    }

    CUtensorMap tmA, tmB, tmBp, tmC;
    std::memset(&tmC, 0, sizeof(tmC));
    if (!encode_operands(&tmA, &tmB, &tmBp, A, B, M, N, K, lda, ldb, wt, fp8, tile_n))
        return BIGEMM_ERR_CUDA;

    GemmParams p;
    std::memset(&p, 0, sizeof(p));
    p.status = d->status;
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.m_tiles = static_cast<int>(m_tiles);
    p.n_tiles = static_cast<int>(n_tiles);
    p.splits = splits;
    p.kb_total = static_cast<int>(ceil_div(K, kb_elems));
    p.kb_per_split = kb_per_split;
    p.units = static_cast<int>(units);
    p.epi_boxes = epi_boxes_for(static_cast<int>(M));
    // a batch of 32-column blocks never spans past the warp's half of a tile
    p.epi_batch = epi_batch_for(static_cast<int>(M));
    if (p.epi_batch > tile_n / 64) p.epi_batch = tile_n / 64;
    p.grouped = 0;
    // what the ring holds: its first 4 (wide), 6 or 8 (narrow) K blocks
    p.prefetch_rows = (tile_n == 128 ? Tile<128>::kStages : (tile_n == 64 ? Tile<64>::kStages : kStages)) *
                      kb_elems;
    // GROUP_M swizzle: 16 tile rows per group once there are four or more waves
    // of tiles (the concurrent tiles then span about 16 x 9 tiles, whose A and
    // B panels stay in L2), else 8.  It orders tiles only; no sum changes.
    p.group_m = (m_tiles * n_tiles >= 4 * static_cast<int64_t>(d->sm_count)) ? 16 : 8;
    p.fold = fold ? 1 : 0;
    p.cluster = cluster ? 1 : 0;
    p.selftest_stall = selftest_stall ? 1 : 0;
    p.a_rows = a_box_rows(M);
    // the scale and the bias follow the full sum: in this kernel unless a
    // reduction kernel forms that sum
    const bool sum_here = (splits == 1) || fold || cluster;
    p.bias = sum_here ? static_cast<const __nv_bfloat16*>(bias) : nullptr;
    p.scale = sum_here ? scale : 1.0f;
    p.idesc_fp8 = fp8 ? idesc_fp8_f32(kBM, kBN, static_cast<uint32_t>(fp8_fmt_a),
                                      static_cast<uint32_t>(fp8_fmt_b))
                      : 0u;

    // persistent (at most one CTA per SM), except with clusters: one unit per CTA
    const int grid = cluster ? static_cast<int>(units)
                             : static_cast<int>(units < d->sm_count ? units : d->sm_count);
    const dim3 g(static_cast<unsigned>(grid)), blk(kNumThreads);
    cudaError_t e = cudaSuccess;
    int launches = 0;

    if (mode == kModeAtomic) {
        e = cudaMemset2DAsync(C, static_cast<size_t>(ldc) * 4, 0, static_cast<size_t>(N) * 4,
                              static_cast<size_t>(M), stream);
        if (e != cudaSuccess) return BIGEMM_ERR_CUDA;
        p.out = C;
        p.ld_out = ldc;
        e = launch_gemm<kOutAtomic>(wt, fp8, g, blk, stream, tmA, tmB, tmBp, tmC, p, 1u, tile_n);
        launches = 1;
    } else if (mode == kModePartial || (splits > 1 && !fold && !cluster)) {
        p.out = ws;
        p.ld_out = ws_ld_of(N);
        p.slice_stride = M * p.ld_out;
        if (encode_out_grouped(&tmC, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, ws, M, N, p.ld_out, splits,
                               p.slice_stride, p.epi_batch))
            p.grouped = 1;
        else if (!encode_out_slices(&tmC, ws, M, N, splits))
            return BIGEMM_ERR_CUDA;
        e = launch_gemm<kOutSlices>(wt, fp8, g, blk, stream, tmA, tmB, tmBp, tmC, p, 1u, tile_n);
        launches = 1;
        if (e == cudaSuccess && mode != kModePartial) {
            st = launch_reduce(*d, static_cast<const float*>(ws), splits, M, N, C, ldc,
                               mode == kModeBF16, stream, bias, scale);
            if (st != BIGEMM_OK) return st;
            launches = 2;
        }
    } else {
        p.out = C;
        p.ld_out = ldc;
        if (mode == kModeBF16) {
            if (encode_out_grouped(&tmC, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, C, M, N, ldc, 0, 0,
                                   p.epi_batch))
                p.grouped = 1;
            else if (!encode_out_bf16(&tmC, C, M, N, ldc))
                return BIGEMM_ERR_CUDA;
            e = launch_gemm<kOutBF16>(wt, fp8, g, blk, stream, tmA, tmB, tmBp, tmC, p,
                                      cluster ? static_cast<unsigned>(splits) : 1u, tile_n);
        } else {
            if (encode_out_grouped(&tmC, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, C, M, N, ldc, 0, 0,
                                   p.epi_batch))
                p.grouped = 1;
            else if (!encode_out_f32(&tmC, C, M, N, ldc))
                return BIGEMM_ERR_CUDA;
            e = launch_gemm<kOutF32>(wt, fp8, g, blk, stream, tmA, tmB, tmBp, tmC, p,
                                     cluster ? static_cast<unsigned>(splits) : 1u, tile_n);
        }
        launches = 1;
    }
    if (e != cudaSuccess) return BIGEMM_ERR_CUDA;
    g_last_launches = launches;
    return BIGEMM_OK;
}

// ---------------------------------------------------------------- Ozaki --
// The Ozaki scheme's binary64 product (cuTile article, "倍精度行列積エミュレー
// ション"): rho = max(ceil(53 - (24 - log2 K) / 2), 53 - 8), in integers:
// ceil(41 + log2(K) / 2) = 41 + t with t the least integer such that 4^t >= K.
constexpr int64_t kOzakiMaxK = int64_t(1) << 22;   // rho <= 52: at least one bit per slice
constexpr int kOzakiMaxSlices = 32;

int ozaki_rho(int64_t K) {
    int t = 0;
    for (int64_t q = 1; q < K; q *= 4) ++t;
    const int gamma = 41 + t;
    return gamma > 45 ? gamma : 45;
}

// Slices whose bits reach 2^-53 below each vector's maximum: beta bits in the
// first slice and beta + 1 in each later one, s (beta + 1) - 1 >= 53.
int ozaki_default_slices(int rho) {
    const int beta = 53 - rho;
    return (54 + beta) / (beta + 1);
}

int64_t ozaki_pair_count(int slices, int d) {
    int64_t n = 0;
    for (int a = 0; a < slices; ++a)
        for (int b = 0; b < slices; ++b)
            if (a + b < d) ++n;
    return n;
}

int64_t round_up(int64_t x, int64_t m) { return ceil_div(x, m) * m; }

// Workspace of bigemm_ozaki_dgemm, in this order, each part 256-byte aligned:
// A slices [s][M][lda_s] bf16, B slices [s][kpad][ldb_s] bf16, c^(1) of the
// rows of A [M] int32, c^(1) of the columns of B [N] int32, one int32 count
// per 128 x 256 output tile (the slice pairs added so far) and one int32
// abort word for the launch.
struct OzakiLayout {
    int64_t lda_s, ldb_s, kpad, tiles;
    size_t off_b, off_ca, off_cb, off_cnt, off_ta, off_tb, total;
};

OzakiLayout ozaki_layout(int64_t M, int64_t N, int64_t K, int slices) {
    OzakiLayout L;
    L.lda_s = round_up(K > 0 ? K : 1, 8);
    L.ldb_s = round_up(N > 0 ? N : 1, 8);
    L.kpad = round_up(K > 0 ? K : 1, kBK);
    const auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    const size_t a = up(static_cast<size_t>(slices) * M * L.lda_s * 2);
    const size_t b = up(static_cast<size_t>(slices) * L.kpad * L.ldb_s * 2);
    const size_t ca = up(static_cast<size_t>(M) * 4);
    const size_t cb = up(static_cast<size_t>(N) * 4);
    L.tiles = ceil_div(M, kBM) * ceil_div(N, kBN);
    const size_t cnt = up(static_cast<size_t>(L.tiles + 1) * 4);
    const size_t ta = up(static_cast<size_t>(M) * 8);
    const size_t tb = up(static_cast<size_t>(N) * 8);
    L.off_b = a;
    L.off_ca = a + b;
    L.off_cb = a + b + ca;
    L.off_cnt = a + b + ca + cb;
    L.off_ta = L.off_cnt + cnt;
    L.off_tb = L.off_ta + ta;
    L.total = L.off_tb + tb;
    return L;
}

int ceil_log2_int(int64_t v) {
    int l = 0;
    while ((int64_t(1) << l) < v) ++l;
    return l;
}

bool aligned_to(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

// The split kernels specialised for the slice width 54 - rho and count that
// the default slice counts pair with it (1..5), else 0: the general kernels.
int ozaki_split_shape(int rho, int slices) {
    const int w = 54 - rho;
    if (w == 9 && slices == 6) return 1;
    if (w == 8 && slices == 7) return 2;
    if (w == 7 && slices == 8) return 3;
    if (w == 6 && slices == 9) return 4;
    if (w == 5 && slices == 11) return 5;
    return 0;
}

// mass: Fast Mode's vector masses (zeroed here for the columns), or nullptr.
cudaError_t launch_ozaki_split(const DeviceInfo& d, const double* X, int64_t rows, int64_t cols,
                               int64_t ld, int axis, int rho, int slices, __nv_bfloat16* out,
                               int64_t out_ld, int64_t out_rows, int* exps, cudaStream_t stream,
                               unsigned long long* mass = nullptr) {
    if (axis == 0) {
        // one block per row, at most 16 resident blocks' worth per SM at a time
        int64_t blocks = rows;
        if (blocks > 16 * static_cast<int64_t>(d.sm_count)) blocks = 16 * static_cast<int64_t>(d.sm_count);
        const dim3 g(static_cast<unsigned>(blocks)), blk(kOzakiRowThreads);
        const int64_t plane = rows * out_ld;
        switch (ozaki_split_shape(rho, slices)) {
        case 1: ozaki_split_rows_kernel<9, 6><<<g, blk, 0, stream>>>(X, rows, cols, ld, rho, slices, out, out_ld, plane, exps, mass); break;
        case 2: ozaki_split_rows_kernel<8, 7><<<g, blk, 0, stream>>>(X, rows, cols, ld, rho, slices, out, out_ld, plane, exps, mass); break;
        case 3: ozaki_split_rows_kernel<7, 8><<<g, blk, 0, stream>>>(X, rows, cols, ld, rho, slices, out, out_ld, plane, exps, mass); break;
        case 4: ozaki_split_rows_kernel<6, 9><<<g, blk, 0, stream>>>(X, rows, cols, ld, rho, slices, out, out_ld, plane, exps, mass); break;
        case 5: ozaki_split_rows_kernel<5, 11><<<g, blk, 0, stream>>>(X, rows, cols, ld, rho, slices, out, out_ld, plane, exps, mass); break;
        default: ozaki_split_rows_kernel<><<<g, blk, 0, stream>>>(X, rows, cols, ld, rho, slices, out, out_ld, plane, exps, mass);
        }
        return cudaGetLastError();
    }
    // column maxima: every exponent starts below any c^(1), then chunks of
    // rows merge theirs with an integer atomicMax
    cudaError_t e = cudaMemsetAsync(exps, 0x80, static_cast<size_t>(cols) * sizeof(int), stream);
    if (e != cudaSuccess) return e;
    if (mass != nullptr) {
        e = cudaMemsetAsync(mass, 0, static_cast<size_t>(cols) * sizeof(unsigned long long), stream);
        if (e != cudaSuccess) return e;
    }
    // chunks of at least kOzakiColChunk rows, at most 65535 of them
    int64_t chunk = ceil_div(ceil_div(rows, 65535), 8) * 8;
    if (chunk < kOzakiColChunk) chunk = kOzakiColChunk;
    const int64_t chunks = ceil_div(rows, chunk);
    ozaki_col_exps_kernel<<<dim3(static_cast<unsigned>(ceil_div(cols, 32)), static_cast<unsigned>(chunks)), 256,
                            0, stream>>>(X, rows, cols, ld, chunk, exps);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // column pairs across threads, rows across blockIdx.y: about 16 blocks per SM
    const int64_t bx = ceil_div(ceil_div(cols, 2), 256);
    int64_t by = ceil_div(16 * static_cast<int64_t>(d.sm_count), bx);
    if (by > out_rows) by = out_rows;
    if (by > 65535) by = 65535;
    if (by < 1) by = 1;
    const dim3 g(static_cast<unsigned>(bx), static_cast<unsigned>(by));
    const int64_t plane = out_rows * out_ld;
    switch (ozaki_split_shape(rho, slices)) {
    case 1: ozaki_split_cols_kernel<9, 6><<<g, 256, 0, stream>>>(X, rows, cols, ld, out_rows, rho, slices, out, out_ld, plane, exps, mass); break;
    case 2: ozaki_split_cols_kernel<8, 7><<<g, 256, 0, stream>>>(X, rows, cols, ld, out_rows, rho, slices, out, out_ld, plane, exps, mass); break;
    case 3: ozaki_split_cols_kernel<7, 8><<<g, 256, 0, stream>>>(X, rows, cols, ld, out_rows, rho, slices, out, out_ld, plane, exps, mass); break;
    case 4: ozaki_split_cols_kernel<6, 9><<<g, 256, 0, stream>>>(X, rows, cols, ld, out_rows, rho, slices, out, out_ld, plane, exps, mass); break;
    case 5: ozaki_split_cols_kernel<5, 11><<<g, 256, 0, stream>>>(X, rows, cols, ld, out_rows, rho, slices, out, out_ld, plane, exps, mass); break;
    default: ozaki_split_cols_kernel<><<<g, 256, 0, stream>>>(X, rows, cols, ld, out_rows, rho, slices, out, out_ld, plane, exps, mass);
    }
    return cudaGetLastError();
}

}  // namespace

// Split-K scratch for bigemm_run_splitk_static, for callers that cannot
// allocate: a fixed array in every loaded device image.  Host code sees only a
// host-side stand-in under this name, so the device address is looked up per
// device with cudaGetSymbolAddress and passed to the kernels.
static __device__ __align__(256) unsigned char g_static_scratch[BIGEMM_STATIC_SCRATCH_BYTES];

namespace {

std::mutex g_static_mu;
void* g_static_addr[kMaxDevices];

// Device address of g_static_scratch on the current device, looked up on the
// first call for that device.
bigemm_status static_scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return BIGEMM_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return BIGEMM_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_static_mu);
    if (g_static_addr[dev] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress((void**)&ptr, g_static_scratch) != cudaSuccess || ptr == nullptr)
            return BIGEMM_ERR_CUDA;
        g_static_addr[dev] = ptr;
    }
    *out = g_static_addr[dev];
    return BIGEMM_OK;
}

}  // namespace
}  // namespace bigemm

using namespace bigemm;

extern "C" {

int bigemm_version(void) { return (0 << 16) | 1; }

const char* bigemm_status_string(bigemm_status s) {
    switch (s) {
        case BIGEMM_OK: return "BIGEMM_OK";
        case BIGEMM_ERR_ARG: return "BIGEMM_ERR_ARG: invalid size, pointer, leading dimension or split_k";
        case BIGEMM_ERR_ALIGN: return "BIGEMM_ERR_ALIGN: pointer or leading dimension not aligned";
        case BIGEMM_ERR_WORKSPACE: return "BIGEMM_ERR_WORKSPACE: workspace missing, misaligned or too small";
        case BIGEMM_ERR_UNSUPPORTED: return "BIGEMM_ERR_UNSUPPORTED: current device is not sm_103";
        case BIGEMM_ERR_CUDA: return "BIGEMM_ERR_CUDA: a CUDA call failed";
        case BIGEMM_ERR_TIMEOUT: return "BIGEMM_ERR_TIMEOUT: a kernel's bounded wait expired";
        case BIGEMM_ERR_STATIC_LIMIT:
            return "BIGEMM_ERR_STATIC_LIMIT: the product needs more split-K scratch than the "
                   "library's built-in 16 MiB array; pass a workspace to bigemm_run or use a "
                   "smaller split_k";
    }
    return "BIGEMM_ERR_UNKNOWN";
}

int bigemm_max_split_k(int64_t K) { return K < 0 ? 0 : max_split(K); }

int bigemm_default_split_k(int64_t K) { return K < 0 ? 0 : default_split(K); }

int bigemm_effective_split_k(int64_t K, int split_k) { return effective_split(K, split_k, nullptr); }

int64_t bigemm_workspace_ld(int64_t N) { return N < 0 ? 0 : ws_ld_of(N); }

int bigemm_split_is_folded(int64_t M, int64_t N, int64_t K, int split_k) {
    if (M < 0 || N < 0) return 0;
    return folds(M, N, effective_split(K, split_k, nullptr)) ? 1 : 0;
}

int bigemm_cluster_capacity(int splits) {
    if (splits < 2 || splits > 8) return 0;
    const DeviceInfo* d = nullptr;
    if (device_info(&d) != BIGEMM_OK) return -1;
    return d->max_clusters[splits];
}

int bigemm_split_path(int64_t M, int64_t N, int64_t K, int split_k, int fp8) {
    if (M < 0 || N < 0 || K < 0) return -1;
    int L = 0;
    const int s = effective_split(K, split_k, &L, fp8 ? 128 : kBK);
    if (s == 0) return -1;
    if (s == 1 || K == 0) return BIGEMM_PATH_UNSPLIT;
    if (skinny(M, s, fp8 != 0)) return BIGEMM_PATH_SKINNY;
    if (folds(M, N, s)) return BIGEMM_PATH_FOLDED;
    const DeviceInfo* d = nullptr;
    if (device_info(&d) != BIGEMM_OK) return -1;
    if (tile_width(M, N, s, L, false, fp8 != 0, d->sm_count) != kBN) return BIGEMM_PATH_WORKSPACE;
    if (s <= 8 && ceil_div(M, kBM) * ceil_div(N, kBN) <= d->max_clusters[s]) return BIGEMM_PATH_CLUSTER;
    return BIGEMM_PATH_WORKSPACE;
}

int bigemm_tile_n(int64_t M, int64_t N, int64_t K, int split_k, int fp8) {
    if (M < 0 || N < 0 || K < 0) return -1;
    int L = 0;
    const int s = effective_split(K, split_k, &L, fp8 ? 128 : kBK);
    if (s == 0) return -1;
    if (M == 0 || N == 0 || K == 0) return kBN;
    if (skinny(M, s, fp8 != 0)) return kBN;
    const DeviceInfo* d = nullptr;
    if (device_info(&d) != BIGEMM_OK) return -1;
    return tile_width(M, N, s, L, folds(M, N, s), fp8 != 0, d->sm_count);
}

int bigemm_uses_pair(int64_t M, int64_t N, int64_t K, int split_k, int fp8) {
    if (M < 0 || N < 0 || K < 0) return -1;
    int L = 0;
    const int s = effective_split(K, split_k, &L, fp8 ? 128 : kBK);
    if (s == 0) return -1;
    if (M == 0 || N == 0 || K == 0 || skinny(M, s, fp8 != 0)) return 0;
    const DeviceInfo* d = nullptr;
    if (device_info(&d) != BIGEMM_OK) return -1;
    const int tn = tile_width(M, N, s, L, folds(M, N, s), fp8 != 0, d->sm_count);
    return pairs_tiles(M, N, s, tn, d->pair_clusters) ? 1 : 0;
}

int bigemm_set_pair_mode(int mode) {
    if (mode < 0 || mode > 2) return -1;
    return g_pair_mode.exchange(mode);
}

int bigemm_pair_capacity(void) {
    const DeviceInfo* d = nullptr;
    if (device_info(&d) != BIGEMM_OK) return -1;
    return d->pair_clusters;
}

size_t bigemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int split_k) {
    if (M < 0 || N < 0) return 0;
    const int s = effective_split(K, split_k, nullptr);
    if (s <= 1 || folds(M, N, s) || skinny(M, s, false)) return 0;
    return slice_bytes(M, N, s);
}

size_t bigemm_partial_workspace_bytes(int64_t M, int64_t N, int64_t K, int split_k) {
    if (M < 0 || N < 0) return 0;
    const int s = effective_split(K, split_k, nullptr);
    if (s < 1) return 0;
    return slice_bytes(M, N, s);
}

bigemm_status bigemm_run(const void* A, const void* B, float* C, int64_t M, int64_t N, int64_t K,
                         int64_t lda, int64_t ldb, int64_t ldc, int split_k, void* workspace,
                         size_t workspace_bytes, bigemm_stream stream) {
    return run_impl(kModeF32, A, B, C, M, N, K, lda, ldb, ldc, split_k, workspace, workspace_bytes,
                    static_cast<cudaStream_t>(stream));
}

bigemm_status bigemm_run_bf16out(const void* A, const void* B, void* C, int64_t M, int64_t N,
                                 int64_t K, int64_t lda, int64_t ldb, int64_t ldc, int split_k,
                                 void* workspace, size_t workspace_bytes, bigemm_stream stream) {
    return run_impl(kModeBF16, A, B, C, M, N, K, lda, ldb, ldc, split_k, workspace, workspace_bytes,
                    static_cast<cudaStream_t>(stream));
}

bigemm_status bigemm_run_partial(const void* A, const void* B, int64_t M, int64_t N, int64_t K,
                                 int64_t lda, int64_t ldb, int split_k, void* workspace,
                                 size_t workspace_bytes, bigemm_stream stream) {
    return run_impl(kModePartial, A, B, nullptr, M, N, K, lda, ldb, 0, split_k, workspace,
                    workspace_bytes, static_cast<cudaStream_t>(stream));
}

bigemm_status bigemm_splitk_reduce(const float* workspace, int splits, int64_t M, int64_t N, void* C,
                                   int64_t ldc, int c_is_bf16, bigemm_stream stream) {
    g_last_launches = 0;
    if (M < 0 || N < 0 || M > INT_MAX || N > INT_MAX || splits < 1) return BIGEMM_ERR_ARG;
    if (M == 0 || N == 0) return BIGEMM_OK;
    if (workspace == nullptr || C == nullptr || ldc < N) return BIGEMM_ERR_ARG;
    if (!aligned16(workspace) || !aligned16(C)) return BIGEMM_ERR_ALIGN;
    if (ldc % (c_is_bf16 ? 8 : 4) != 0) return BIGEMM_ERR_ALIGN;
    if (slice_bytes(M, N, splits) == SIZE_MAX) return BIGEMM_ERR_ARG;
    const DeviceInfo* d = nullptr;
    bigemm_status st = device_info(&d);
    if (st != BIGEMM_OK) return st;
    st = launch_reduce(*d, workspace, splits, M, N, C, ldc, c_is_bf16 != 0,
                       static_cast<cudaStream_t>(stream));
    if (st == BIGEMM_OK) g_last_launches = 1;
    return st;
}

bigemm_status bigemm_linear(const void* A, const void* W, const void* bias, void* C, int64_t M,
                            int64_t N, int64_t K, int64_t lda, int64_t ldw, int64_t ldc, int split_k,
                            int c_is_bf16, void* workspace, size_t workspace_bytes,
                            bigemm_stream stream) {
    return run_impl(c_is_bf16 ? kModeBF16 : kModeF32, A, W, C, M, N, K, lda, ldw, ldc, split_k,
                    workspace, workspace_bytes, static_cast<cudaStream_t>(stream), /*wt=*/true, bias);
}

int bigemm_fp8_effective_split_k(int64_t K, int split_k) {
    return effective_split(K, split_k, nullptr, 128);
}

size_t bigemm_fp8_workspace_bytes(int64_t M, int64_t N, int64_t K, int split_k) {
    if (M < 0 || N < 0) return 0;
    const int s = effective_split(K, split_k, nullptr, 128);
    if (s <= 1 || folds(M, N, s)) return 0;
    return slice_bytes(M, N, s);
}

bigemm_status bigemm_linear_fp8(const void* A, const void* W, int fmt_a, int fmt_w, float scale,
                                const void* bias, void* C, int64_t M, int64_t N, int64_t K,
                                int64_t lda, int64_t ldw, int64_t ldc, int split_k, int c_is_bf16,
                                void* workspace, size_t workspace_bytes, bigemm_stream stream) {
    g_last_launches = 0;
    if ((fmt_a != BIGEMM_FP8_E4M3 && fmt_a != BIGEMM_FP8_E5M2) ||
        (fmt_w != BIGEMM_FP8_E4M3 && fmt_w != BIGEMM_FP8_E5M2) || !(scale == scale))
        return BIGEMM_ERR_ARG;
    return run_impl(c_is_bf16 ? kModeBF16 : kModeF32, A, W, C, M, N, K, lda, ldw, ldc, split_k,
                    workspace, workspace_bytes, static_cast<cudaStream_t>(stream), /*wt=*/true, bias,
                    fmt_a, fmt_w, scale);
}

size_t bigemm_fp8_kn_workspace_bytes(int64_t M, int64_t N, int64_t K, int split_k) {
    if (M < 0 || N < 0 || K < 0 || effective_split(K, split_k, nullptr, 128) == 0) return 0;
    const size_t bt = static_cast<size_t>(N) * static_cast<size_t>(round_up(K > 0 ? K : 1, 16));
    return (bt + 255) / 256 * 256 + bigemm_fp8_workspace_bytes(M, N, K, split_k);
}

bigemm_status bigemm_run_fp8(const void* A, const void* B, int fmt_a, int fmt_b, float scale, const void* bias,
                             void* C, int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                             int split_k, int c_is_bf16, void* workspace, size_t workspace_bytes,
                             bigemm_stream stream) {
    g_last_launches = 0;
    if ((fmt_a != BIGEMM_FP8_E4M3 && fmt_a != BIGEMM_FP8_E5M2) ||
        (fmt_b != BIGEMM_FP8_E4M3 && fmt_b != BIGEMM_FP8_E5M2) || !(scale == scale))
        return BIGEMM_ERR_ARG;
    if (M < 0 || N < 0 || K < 0 || M > INT_MAX || N > INT_MAX || K > INT_MAX) return BIGEMM_ERR_ARG;
    if (effective_split(K, split_k, nullptr, 128) == 0) return BIGEMM_ERR_ARG;
    if (K > 0 && (B == nullptr || ldb < N)) return BIGEMM_ERR_ARG;
    if (K > 0 && (!aligned16(B) || ldb % 16 != 0)) return BIGEMM_ERR_ALIGN;
    const int64_t ldt = round_up(K > 0 ? K : 1, 16);
    const size_t bt = (static_cast<size_t>(N) * static_cast<size_t>(ldt) + 255) / 256 * 256;
    const size_t need = bigemm_fp8_kn_workspace_bytes(M, N, K, split_k);
    if (K > 0 && M > 0 && N > 0 &&
        (workspace == nullptr || !aligned_to(workspace, 256) || workspace_bytes < need))
        return BIGEMM_ERR_WORKSPACE;
    const cudaStream_t strm = static_cast<cudaStream_t>(stream);
    uint8_t* Bt = static_cast<uint8_t*>(workspace);
    if (K > 0 && M > 0 && N > 0) {
        const dim3 g(static_cast<unsigned>(ceil_div(N, kTrTile)), static_cast<unsigned>(ceil_div(ldt, kTrTile)));
        fp8_transpose_kernel<<<g, kTrThreads, 0, strm>>>(static_cast<const uint8_t*>(B), ldb, Bt, ldt,
                                                          static_cast<int>(K), static_cast<int>(N));
        if (cudaGetLastError() != cudaSuccess) return BIGEMM_ERR_CUDA;
    }
    unsigned char* ws2 = workspace != nullptr ? static_cast<unsigned char*>(workspace) + bt : nullptr;
    const size_t ws2_bytes = workspace_bytes > bt ? workspace_bytes - bt : 0;
    const bigemm_status st = run_impl(c_is_bf16 ? kModeBF16 : kModeF32, A, (K > 0 && M > 0 && N > 0) ? Bt : B, C,
                                      M, N, K, lda, ldt, ldc, split_k, ws2, ws2_bytes, strm, /*wt=*/true, bias,
                                      fmt_a, fmt_b, scale);
    if (st == BIGEMM_OK && K > 0 && M > 0 && N > 0) g_last_launches += 1;
    return st;
}

bigemm_status bigemm_run_atomic_splitk(const void* A, const void* B, float* C, int64_t M, int64_t N,
                                       int64_t K, int64_t lda, int64_t ldb, int64_t ldc, int split_k,
                                       bigemm_stream stream) {
    return run_impl(kModeAtomic, A, B, C, M, N, K, lda, ldb, ldc, split_k, nullptr, 0,
                    static_cast<cudaStream_t>(stream));
}

bigemm_status bigemm_run_splitk_static(const void* A, const void* B, float* C, int64_t M, int64_t N,
                                       int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                                       int split_k, bigemm_stream stream) {
    g_last_launches = 0;
    const size_t need = bigemm_workspace_bytes(M, N, K, split_k);
    if (need > BIGEMM_STATIC_SCRATCH_BYTES) return BIGEMM_ERR_STATIC_LIMIT;
    void* scratch = nullptr;
    if (need > 0) {
        const bigemm_status st = static_scratch_address(&scratch);
        if (st != BIGEMM_OK) return st;
    }
    return run_impl(kModeF32, A, B, C, M, N, K, lda, ldb, ldc, split_k, scratch,
                    scratch ? static_cast<size_t>(BIGEMM_STATIC_SCRATCH_BYTES) : 0,
                    static_cast<cudaStream_t>(stream));
}

bigemm_status bigemm_selftest_timeout(bigemm_stream stream) {
    g_last_launches = 0;
    void* scratch = nullptr;
    const bigemm_status st = static_scratch_address(&scratch);
    if (st != BIGEMM_OK) return st;
    // a 16 x 256 x 512 split-K partial product whose operands and workspace
    // sit in the built-in array; nothing is ever loaded or stored
    unsigned char* base = static_cast<unsigned char*>(scratch);
    return run_impl(kModePartial, base, base + (64 << 10), nullptr, 16, 256, 512, 512, 256, 0, 1,
                    base + (1 << 20), 16 * 256 * 4, static_cast<cudaStream_t>(stream), false, nullptr,
                    -1, -1, 1.0f, /*selftest_stall=*/true);
}

static bigemm_status ozaki_dgemm_impl(const double* A, const double* B, double* C, int64_t M, int64_t N,
                                      int64_t K, int64_t lda, int64_t ldb, int64_t ldc, int slices, int d,
                                      void* workspace, size_t workspace_bytes, bigemm_stream stream,
                                      bool stall_order);

bigemm_status bigemm_selftest_ozaki_order_timeout(bigemm_stream stream) {
    g_last_launches = 0;
    void* scratch = nullptr;
    const bigemm_status st = static_scratch_address(&scratch);
    if (st != BIGEMM_OK) return st;
    // a 256 x 256 x 128 product of zero matrices in the built-in array:
    // A and B (256 KiB each), C (512 KiB), then the workspace
    constexpr int64_t M = 256, N = 256, K = 128;
    unsigned char* base = static_cast<unsigned char*>(scratch);
    double* A = reinterpret_cast<double*>(base);
    double* B = reinterpret_cast<double*>(base + (256 << 10));
    double* C = reinterpret_cast<double*>(base + (512 << 10));
    unsigned char* ws = base + (1 << 20);
    const size_t need = ozaki_layout(M, N, K, ozaki_default_slices(ozaki_rho(K))).total;
    if (need + (1u << 20) > BIGEMM_STATIC_SCRATCH_BYTES) return BIGEMM_ERR_STATIC_LIMIT;
    if (cudaMemsetAsync(base, 0, 512 << 10, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return BIGEMM_ERR_CUDA;
    return ozaki_dgemm_impl(A, B, C, M, N, K, K, N, N, 0, 0, ws, need, stream, /*stall_order=*/true);
}

int bigemm_ozaki_rho(int64_t K) { return (K < 1 || K > kOzakiMaxK) ? -1 : ozaki_rho(K); }

int bigemm_ozaki_default_slices(int64_t K) {
    return (K < 1 || K > kOzakiMaxK) ? -1 : ozaki_default_slices(ozaki_rho(K));
}

int64_t bigemm_ozaki_pairs(int slices, int d) {
    return (slices < 1 || d < 0) ? -1 : ozaki_pair_count(slices, d);
}

size_t bigemm_ozaki_workspace_bytes(int64_t M, int64_t N, int64_t K, int slices) {
    if (M < 0 || N < 0 || K < 0 || K > kOzakiMaxK) return 0;
    if (slices == 0) slices = K > 0 ? ozaki_default_slices(ozaki_rho(K)) : 1;
    if (slices < 1 || slices > kOzakiMaxSlices) return 0;
    return ozaki_layout(M, N, K, slices).total;
}

bigemm_status bigemm_ozaki_split(const double* X, int64_t rows, int64_t cols, int64_t ld, int axis,
                                 int rho, int slices, void* out, int64_t out_ld, int64_t out_rows,
                                 int* exps, bigemm_stream stream) {
    g_last_launches = 0;
    if (rows < 0 || cols < 0 || (axis != 0 && axis != 1)) return BIGEMM_ERR_ARG;
    if (rho < 45 || rho > 52 || slices < 1 || slices > kOzakiMaxSlices) return BIGEMM_ERR_ARG;
    if (rows == 0 || cols == 0) return BIGEMM_OK;
    if (X == nullptr || out == nullptr || exps == nullptr || ld < cols || out_ld < cols) return BIGEMM_ERR_ARG;
    if (axis == 1 && out_rows < rows) return BIGEMM_ERR_ARG;
    if (!aligned_to(X, 8) || !aligned_to(out, 2) || !aligned_to(exps, 4)) return BIGEMM_ERR_ALIGN;
    const DeviceInfo* d = nullptr;
    bigemm_status st = device_info(&d);
    if (st != BIGEMM_OK) return st;
    const cudaError_t e = launch_ozaki_split(*d, X, rows, cols, ld, axis, rho, slices,
                                             static_cast<__nv_bfloat16*>(out), out_ld,
                                             axis == 1 ? out_rows : rows, exps,
                                             static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return BIGEMM_ERR_CUDA;
    g_last_launches = axis == 0 ? 1 : 2;
    return BIGEMM_OK;
}

// stall_order (the failure self-test only): every tile's count starts far
// below zero, so no epilogue wait for a previous slice pair is ever met.
static bigemm_status ozaki_dgemm_impl(const double* A, const double* B, double* C, int64_t M, int64_t N,
                                      int64_t K, int64_t lda, int64_t ldb, int64_t ldc, int slices, int d,
                                      void* workspace, size_t workspace_bytes, bigemm_stream stream,
                                      bool stall_order) {
    g_last_launches = 0;
    const cudaStream_t strm = static_cast<cudaStream_t>(stream);
    if (M < 0 || N < 0 || K < 0 || K > kOzakiMaxK || M > INT_MAX || N > INT_MAX) return BIGEMM_ERR_ARG;
    const int rho = K > 0 ? ozaki_rho(K) : 52;
    if (slices == 0) slices = ozaki_default_slices(rho);
    if (slices < 1 || slices > kOzakiMaxSlices || d < -1) return BIGEMM_ERR_ARG;
    const bool fast = (d == -1);  // Fast Mode's automatic d, per element
    if (d == 0 || fast) d = slices;
    if (K > 0 && (A == nullptr || B == nullptr || lda < K || ldb < N)) return BIGEMM_ERR_ARG;
    if (C == nullptr || ldc < N) return BIGEMM_ERR_ARG;
    if (K > 0 && (!aligned_to(A, 8) || !aligned_to(B, 8))) return BIGEMM_ERR_ALIGN;
    if (!aligned16(C) || ldc % 2 != 0) return BIGEMM_ERR_ALIGN;
    const OzakiLayout L = ozaki_layout(M, N, K, slices);
    if (K > 0 && (workspace == nullptr || !aligned_to(workspace, 256) || workspace_bytes < L.total))
        return BIGEMM_ERR_WORKSPACE;
    if (static_cast<int64_t>(slices) * M > INT_MAX || static_cast<int64_t>(slices) * L.kpad > INT_MAX)
        return BIGEMM_ERR_ARG;
    if (M == 0 || N == 0) return BIGEMM_OK;
    const DeviceInfo* dev = nullptr;
    bigemm_status st = device_info(&dev);
    if (st != BIGEMM_OK) return st;
    if (K == 0) {  // the empty sum
        const cudaError_t e = cudaMemset2DAsync(C, static_cast<size_t>(ldc) * 8, 0,
                                                static_cast<size_t>(N) * 8, static_cast<size_t>(M), strm);
        return e == cudaSuccess ? BIGEMM_OK : BIGEMM_ERR_CUDA;
    }
    const int64_t pairs = ozaki_pair_count(slices, d);
    if (pairs == 0) {  // every pair skipped: the sum of no terms
        const cudaError_t e = cudaMemset2DAsync(C, static_cast<size_t>(ldc) * 8, 0,
                                                static_cast<size_t>(N) * 8, static_cast<size_t>(M), strm);
        return e == cudaSuccess ? BIGEMM_OK : BIGEMM_ERR_CUDA;
    }
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    __nv_bfloat16* As = reinterpret_cast<__nv_bfloat16*>(ws);
    __nv_bfloat16* Bs = reinterpret_cast<__nv_bfloat16*>(ws + L.off_b);
    int* ca = reinterpret_cast<int*>(ws + L.off_ca);
    int* cb = reinterpret_cast<int*>(ws + L.off_cb);
    int* cnt = reinterpret_cast<int*>(ws + L.off_cnt);
    unsigned long long* ta = fast ? reinterpret_cast<unsigned long long*>(ws + L.off_ta) : nullptr;
    unsigned long long* tb = fast ? reinterpret_cast<unsigned long long*>(ws + L.off_tb) : nullptr;
    // 1-3: split A by rows and B by columns (plain launches: they read the
    // caller's A and B, so they wait for everything before them); with Fast
    // Mode's automatic d also the vectors' masses
    if (launch_ozaki_split(*dev, A, M, K, lda, 0, rho, slices, As, L.lda_s, M, ca, strm, ta) != cudaSuccess ||
        launch_ozaki_split(*dev, B, K, N, ldb, 1, rho, slices, Bs, L.ldb_s, L.kpad, cb, strm, tb) != cudaSuccess)
        return BIGEMM_ERR_CUDA;
    // 4: every slice pair's product on the tensor cores, summed in binary64
    CUtensorMap tmA, tmB, tmBp;
    {
        const int64_t da[2] = {K, slices * M};
        const int64_t db[2] = {N, slices * L.kpad};
        const uint32_t ba[2] = {static_cast<uint32_t>(kBK), static_cast<uint32_t>(kBM)};
        const uint32_t bb[2] = {kBChunkCols, static_cast<uint32_t>(kBK)};
        const uint32_t bp[2] = {static_cast<uint32_t>(kBN), static_cast<uint32_t>(kPrefetchRows)};
        if (!encode_tiled(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, As, 2, da, L.lda_s, 0, ba,
                          CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_tiled(&tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Bs, 2, db, L.ldb_s, 0, bb,
                          CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_tiled(&tmBp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Bs, 2, db, L.ldb_s, 0, bp,
                          CU_TENSOR_MAP_SWIZZLE_NONE))
            return BIGEMM_ERR_CUDA;
    }
    const int64_t m_tiles = ceil_div(M, kBM), n_tiles = ceil_div(N, kBN);
    if (m_tiles * n_tiles * pairs > INT_MAX) return BIGEMM_ERR_ARG;
    // every tile's count of added slice pairs starts at zero, and so does the
    // launch's abort word after them
    if (cudaMemsetAsync(cnt, 0, static_cast<size_t>(L.tiles + 1) * sizeof(int), strm) != cudaSuccess)
        return BIGEMM_ERR_CUDA;
    if (stall_order &&
        cudaMemsetAsync(cnt, 0x80, static_cast<size_t>(L.tiles) * sizeof(int), strm) != cudaSuccess)
        return BIGEMM_ERR_CUDA;
    GemmParams p;
    std::memset(&p, 0, sizeof(p));
    p.out = C;
    p.ld_out = ldc;
    p.status = dev->status;
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.m_tiles = static_cast<int>(m_tiles);
    p.n_tiles = static_cast<int>(n_tiles);
    p.splits = 1;
    p.kb_total = static_cast<int>(ceil_div(K, kBK));
    p.kb_per_split = p.kb_total;
    p.units = static_cast<int>(m_tiles * n_tiles);
    p.epi_boxes = epi_boxes_for(static_cast<int>(M));
    p.epi_batch = epi_batch_for(static_cast<int>(M));
    p.prefetch_rows = kStages * kBK;
    p.group_m = (m_tiles * n_tiles >= 4 * static_cast<int64_t>(dev->sm_count)) ? 16 : 8;
    p.scale = 1.0f;
    p.oz_ca = ca;
    p.oz_cb = cb;
    p.oz_count = cnt;
    p.oz_slices = slices;
    p.oz_d = d;
    p.oz_beta = 53 - rho;
    p.oz_pairs = static_cast<int>(pairs);
    p.oz_kpad = static_cast<int>(L.kpad);
    p.oz_fast = fast ? 1 : 0;
    p.oz_ta = ta;
    p.oz_tb = tb;
    p.oz_need0 = 134 + ceil_log2_int(slices) + ceil_log2_int(K);
    p.oz_c32 = (aligned_to(C, 32) && ldc % 4 == 0) ? 1 : 0;
    p.a_rows = kBM;
    // On CTA pairs: the same items over 256-row tiles, each CTA adding its 128
    // rows under the count of its 128 x 256 tile; a cooperative launch of
    // clusters of two.  The rule (pair mode 1): the (slice pair, tile) items
    // fill two waves of pairs and K is below 4096.  Measured with 32-byte C
    // accesses in the epilogue: pairs 2-3 % faster at 2048^3 and 3072^3, 6 %
    // slower at 4096^3, 13 % at 6144^3 and 3 % at 8192^3 -- with the shorter
    // products the loads pace an item, with the longer ones the binary64
    // read-add-write of C, and a pair waits for the slower of its two CTAs.
    {
        const int mode = g_pair_mode.load(std::memory_order_relaxed);
        const int64_t pm_tiles = ceil_div(M, kPairBM);
        const int64_t pitems = pm_tiles * n_tiles * pairs;
        if (mode != 0 && M >= kPairBM && dev->pair_clusters > 0 &&
            (mode == 2 || (pitems >= 2 * static_cast<int64_t>(dev->pair_clusters) && K < 4096))) {
            GemmParams q = p;
            q.m_tiles = static_cast<int>(pm_tiles);
            q.units = static_cast<int>(pm_tiles * n_tiles);
            q.group_m = (q.units >= 4 * static_cast<int64_t>(dev->pair_clusters)) ? 8 : 4;
            const int64_t gp = pitems < dev->pair_clusters ? pitems : dev->pair_clusters;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(static_cast<unsigned>(2 * gp));
            cfg.blockDim = dim3(kNumThreads);
            cfg.dynamicSmemBytes = kPairSmemBytes;
            cfg.stream = strm;
            cudaLaunchAttribute attr[2];
            attr[0].id = cudaLaunchAttributeCooperative;
            attr[0].val.cooperative = 1;
            attr[1].id = cudaLaunchAttributeClusterDimension;
            attr[1].val.clusterDim.x = 2;
            attr[1].val.clusterDim.y = 1;
            attr[1].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 2;
            if (cudaLaunchKernelEx(&cfg, bigemm_pair_kernel<kOutOzaki, false>, tmA, tmB, tmA, q) != cudaSuccess)
                return BIGEMM_ERR_CUDA;
            g_last_launches = 4;
            return BIGEMM_OK;
        }
    }
    // one CTA per SM at most, over all (slice pair, tile) items: a tile's pairs
    // may run on different CTAs at once, their additions ordered by the counts
    const int64_t items = static_cast<int64_t>(p.units) * pairs;
    const int grid = static_cast<int>(items < dev->sm_count ? items : dev->sm_count);
    if (launch_gemm<kOutOzaki>(false, false, dim3(static_cast<unsigned>(grid)), dim3(kNumThreads), strm,
                               tmA, tmB, tmBp, tmA, p) != cudaSuccess)
        return BIGEMM_ERR_CUDA;
    g_last_launches = 4;
    return BIGEMM_OK;
}

bigemm_status bigemm_ozaki_dgemm(const double* A, const double* B, double* C, int64_t M, int64_t N,
                                 int64_t K, int64_t lda, int64_t ldb, int64_t ldc, int slices, int d,
                                 void* workspace, size_t workspace_bytes, bigemm_stream stream) {
    return ozaki_dgemm_impl(A, B, C, M, N, K, lda, ldb, ldc, slices, d, workspace, workspace_bytes, stream,
                            false);
}

bigemm_status bigemm_device_status(int reset) {
    const DeviceInfo* d = nullptr;
    bigemm_status st = device_info(&d);
    if (st != BIGEMM_OK) return st;
    if (cudaDeviceSynchronize() != cudaSuccess) return BIGEMM_ERR_CUDA;
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof(v)) != cudaSuccess) return BIGEMM_ERR_CUDA;
    if (reset && v != 0) {
        const unsigned zero = 0;
        if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof(zero)) != cudaSuccess)
            return BIGEMM_ERR_CUDA;
    }
    return v ? BIGEMM_ERR_TIMEOUT : BIGEMM_OK;
}

int bigemm_last_launch_count(void) { return g_last_launches; }

}  // extern "C"
