// Host side of the C ABI declared in include/tpgemm.h: argument checks, kernel
// selection, TMA tensor-map encoding and launch. Nothing here allocates or
// synchronises on the gemm_run path; the only device allocation is the 8-byte
// status word made by gemm_create.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include "tpgemm.h"

#include "aux_kernels.cuh"
#include "launch.cuh"
#include "schedule.cuh"

namespace {

constexpr int64_t kMaxDim = 2147483647; // 2^31 - 1
constexpr int kGroupM = 16;             // grouped-raster band height, in tiles (1-CTA mode)
constexpr int kGroupMPair = 8;          // band height in 256-row pair tiles
constexpr int kStreamMaxM = 64;

// The tiled kernels' schedule for an mt x nt tile grid on at most `cap`
// workers. A 1-CTA tile loads 128 A rows and 256 B columns per k-block (A is a
// third of the bytes) and may be cut into 2 or 4 column pieces; a pair tile
// loads 128 A rows and 128 B columns per CTA (A is half) and is cut in halves
// at most, so that each CTA of the pair keeps a 64-column B box.
tpg::Schedule tiled_schedule(int64_t mt, int64_t nt, int64_t cap, bool pair, bool allow_split) {
    const int max_split = allow_split ? (pair ? 2 : 4) : 1;
    return tpg::make_schedule(mt, nt, pair ? kGroupMPair : kGroupM, cap, max_split, pair ? 0.5 : 1.0 / 3.0);
}

struct Plan {
    int variant = TPGEMM_VARIANT_AUTO;
    int ksplit = 1; // tiled 1-CTA mode: CTAs of a cluster that share one tile's K range
    int tile_m = 0, tile_n = 0;
    int64_t num_tiles = 0;
    int grid = 0;
    int cluster = 1;
    int smem = 0;
    int launches = 0;
    int mt_pad = 0, stages = 0, split = 1;
    int ktail = 0; // CTA-pair mode: the last partial round's tiles split over K (workspace)
    tpg::Schedule sched{};
};

// Workspace bytes of the K split tail for `tail_tiles` tiles: the flags, then
// four 64 KB partial-sum slots per tile (two CTAs of each of two pairs).
int64_t tail_ws_bytes(int64_t tail_tiles) {
    return tpg::tiled::kTailFlagBytes + tail_tiles * 4 * static_cast<int64_t>(tpg::tiled::kTailSlotBytes);
}

// Fewest K blocks for which the K split tail is used. On square 4096^3 the
// exchange of partial sums costs about 4.5 us more than a column half's plain
// epilogue, and a K half saves 0.168 us per K block of the tile (half of a
// 256 x 256 K block's 0.336 us): the split pays from about 27 K blocks.
constexpr int64_t kTailMinKb = 32;

// Whether the last partial round of a CTA-pair schedule is split over K: its
// tiles are cut into column halves (split == 2), K has at least kTailMinKb
// blocks, and the workspace holds the tail's flags and partial sums.
bool tail_ksplit_choice(int split, int64_t kb, int64_t tail_tiles, int64_t ws_bytes) {
    return split == 2 && kb >= kTailMinKb && tail_tiles > 0 && tail_ws_bytes(tail_tiles) <= ws_bytes;
}

} // namespace

struct tpgemm_handle {
    int device = -1;
    int num_sms = 0;
    uint32_t *status = nullptr;
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    int forced = TPGEMM_VARIANT_AUTO;
    uint64_t timeout_ns = 2000000000ull;
    // Occupancy caches, filled on first use. Calls from several host threads
    // may fill one at the same time; they store the same value, and the
    // atomics make that well defined.
    // co-resident clusters of the streaming kernel, per [out f32][K split - 2][mt/16 - 1]
    std::atomic<int> stream_clusters[2][3][4] = {};
    // co-resident CTA pairs of the tiled kernel in pair mode, per [out f32]
    std::atomic<int> pair_clusters[2] = {};
    // co-resident clusters of 2 and 4 CTAs of the tiled kernel in 1-CTA mode (K
    // split), per [out f32][0: two, 1: four]
    std::atomic<int> ks_clusters[2][2] = {};
    // co-resident CTA pairs of the MX kernel's pair mode, per [out f32]
    std::atomic<int> mx_pairs[2] = {};
    // the same for its FP4 forms, per [format][out f32]
    std::atomic<int> fp4_pairs[2][2] = {};
    // Caller-owned workspace (gemm_set_workspace), or null, and the tag of the
    // latest call that may use it.
    void *ws = nullptr;
    int64_t ws_bytes = 0;
    std::atomic<uint32_t> epoch{0};
};

namespace {

// Makes `dev` the calling thread's device for the scope of a call, and binds
// its primary context to the thread. The binding matters: the tensor-map
// encoder is a driver call that needs a current context, and a fresh host
// thread has none until some runtime call creates the binding (cudaGetDevice
// does not), so it is made here on every call, not only on a device switch.
struct DeviceGuard {
    int prev = -1;
    bool switched = false;
    explicit DeviceGuard(int dev) {
        const bool other = cudaGetDevice(&prev) == cudaSuccess && prev != dev;
        const bool set = cudaSetDevice(dev) == cudaSuccess;
        switched = other && set;
    }
    ~DeviceGuard() {
        if (switched) cudaSetDevice(prev);
    }
};

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Byte range [lo, hi) touched by a row-major rows x cols matrix with row stride ld.
struct Range {
    uintptr_t lo, hi;
};
Range byte_range(const void *p, int64_t rows, int64_t cols, int64_t ld, int64_t elt) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    if (rows <= 0 || cols <= 0) return {lo, lo};
    return {lo, lo + static_cast<uintptr_t>(((rows - 1) * ld + cols) * elt)};
}
bool overlaps(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi && a.lo != a.hi && b.lo != b.hi; }

// Row stride in bytes given to the tensor map: the caller's, except for a
// single-row matrix whose stride is never used (any 16-byte multiple works).
uint64_t tma_stride(int64_t rows, int64_t cols, int64_t ld, int64_t elt) {
    if (rows <= 1) return static_cast<uint64_t>(((cols * elt) + 15) / 16 * 16);
    return static_cast<uint64_t>(ld * elt);
}

int encode_2d(tpgemm_handle *h, CUtensorMap *map, CUtensorMapDataType dt, const void *ptr,
              uint64_t inner, uint64_t outer, uint64_t stride_bytes, uint32_t box_inner,
              uint32_t box_outer) {
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {stride_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = h->encode(map, dt, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? TPGEMM_OK : TPGEMM_ERR_CUDA;
}

// Rank-3 tensor map of a row-major matrix stack: `slices` matrices of rows x
// inner elements with row stride ld and slice stride slice_ld (elements). One
// slice when slices == 1 (its slice stride is never used).
int encode_3d(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap *map, CUtensorMapDataType dt, const void *ptr,
              uint64_t inner, uint64_t rows, uint64_t row_stride_bytes, uint64_t slices, int64_t slice_ld, int64_t elt,
              uint32_t box_inner, uint32_t box_outer) {
    cuuint64_t dims[3] = {inner, rows, slices};
    uint64_t s2 = slices > 1 ? static_cast<uint64_t>(slice_ld * elt) : row_stride_bytes * (rows > 0 ? rows : 1);
    s2 = (s2 + 15) / 16 * 16;
    if (s2 >= (1ull << 40)) s2 = (1ull << 40) - 16;
    cuuint64_t strides[2] = {row_stride_bytes, s2};
    cuuint32_t box[3] = {box_inner, box_outer, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = encode(map, dt, 3, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? TPGEMM_OK : TPGEMM_ERR_CUDA;
}

// B (bf16, [slices][K][N] with row stride ldb) viewed as [slices][N/64][K][64]:
// a box of {64 columns, 64 K rows, 2 groups} is two 64 x 64 boxes of the 3-D
// view, side by side in shared memory. N must be a multiple of 64, so that no
// group runs past the end of a row.
int encode_b_grouped(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap *map, const void *ptr, int64_t N,
                     int64_t K, int64_t ldb, int64_t slices, int64_t slice_ld) {
    cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(N / 64),
                          static_cast<cuuint64_t>(slices)};
    uint64_t s3 = slices > 1 ? static_cast<uint64_t>(slice_ld * 2) : static_cast<uint64_t>(ldb * 2 * K);
    s3 = (s3 + 15) / 16 * 16;
    if (s3 >= (1ull << 40)) s3 = (1ull << 40) - 16;
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(ldb * 2), 128, s3};
    cuuint32_t box[4] = {64, 64, 2, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? TPGEMM_OK : TPGEMM_ERR_CUDA;
}

// One tiled launch, in the general form: `batch` slices of A, C, D (rows rows
// each, or one stack of rows rows for a grouped GEMM) and `bslices` slices of
// B. A stride of 0 shares one slice between all batches.
struct TiledCall {
    int64_t rows, N, K, batch, bslices;
    const void *A;
    int64_t lda, sA;
    const void *B;
    int64_t ldb, sB;
    const void *C;
    int64_t ldc, sC;
    void *D;
    int64_t ldd, sD;
    float alpha, beta;
    bool f32;
};

int build_tiled(PFN_cuTensorMapEncodeTiled_v12000 encode, const TiledCall &c, CUtensorMap *tmA, CUtensorMap *tmB,
                CUtensorMap *tmB1, CUtensorMap *tmC, CUtensorMap *tmD, tpg::TiledParams *p) {
    const int64_t elt = c.f32 ? 4 : 2;
    const bool use_c = c.beta != 0.0f;
    const CUtensorMapDataType out_dt = c.f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const uint32_t chunk = c.f32 ? 32u : 64u;
    // C and D maps stop at the last whole 16-byte cell of a row (see TiledParams::n_tma);
    // with no whole cell the maps are placeholders and every column takes the plain path.
    const int64_t cell = 16 / elt;
    const int64_t n_tma = c.N / cell * cell;
    const uint64_t map_n = static_cast<uint64_t>(n_tma > 0 ? n_tma : c.N);
    const int64_t aslices = c.sA ? c.batch : 1, bslices = c.sB ? c.bslices : 1;
    const int64_t cslices = (use_c && c.sC) ? c.batch : 1;
    const bool b_grouped = c.N % 64 == 0;
    if (encode_3d(encode, tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c.A, c.K, c.rows, tma_stride(c.rows, c.K, c.lda, 2),
                  aslices, c.sA, 2, 64, tpg::tiled::BM) ||
        encode_3d(encode, tmB1, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c.B, c.N, c.K, tma_stride(c.K, c.N, c.ldb, 2),
                  bslices, c.sB, 2, 64, 64) ||
        (b_grouped ? encode_b_grouped(encode, tmB, c.B, c.N, c.K, c.ldb, bslices, c.sB) : (*tmB = *tmB1, 0)) ||
        encode_3d(encode, tmD, out_dt, c.D, map_n, c.rows, tma_stride(c.rows, c.N, c.ldd, elt), c.batch, c.sD, elt,
                  chunk, tpg::tiled::BM) ||
        encode_3d(encode, tmC, out_dt, use_c ? c.C : c.D, map_n, c.rows,
                  use_c ? tma_stride(c.rows, c.N, c.ldc, elt) : tma_stride(c.rows, c.N, c.ldd, elt), cslices,
                  use_c ? c.sC : c.sD, elt, chunk, tpg::tiled::BM))
        return TPGEMM_ERR_CUDA;
    *p = tpg::TiledParams{};
    p->M = static_cast<int32_t>(c.rows);
    p->N = static_cast<int32_t>(c.N);
    p->K = static_cast<int32_t>(c.K);
    p->kb = static_cast<int32_t>((c.K + tpg::tiled::BK - 1) / tpg::tiled::BK);
    p->a_bcast = c.sA ? 0 : 1;
    p->b_bcast = c.sB ? 0 : 1;
    p->c_bcast = c.sC ? 0 : 1;
    p->sC = c.sC;
    p->sD = c.sD;
    p->n_tma = static_cast<int32_t>(n_tma);
    p->b_grouped = b_grouped ? 1 : 0;
    p->ksplit = 1;
    p->alpha = c.alpha;
    p->beta = c.beta;
    p->C = use_c ? c.C : nullptr;
    p->ldc = c.ldc;
    p->D = c.D;
    p->ldd = c.ldd;
    return TPGEMM_OK;
}

// K split of the streaming variant: each panel's K range over s CTAs of a
// cluster, s from 1 to 4, so that narrow outputs (few panels) still stream B on
// every SM. Each CTA needs at least one K block and a ring of at least 4
// stages beside the reduction slots. A panel takes one time unit on one CTA,
// so s costs rounds(s) / s, rounds(s) being the panels over the co-resident
// clusters of s CTAs, plus 2% per extra CTA for the reduction. clusters[s - 2]
// is the number of clusters of s CTAs that fit at once (0: s not possible).
// Returns s and the cluster count it runs on.
int stream_split_choice(int64_t nt, int64_t kb, int mt_pad, int num_sms, const int *clusters, int *clusters_used) {
    int best_s = 1, best_clusters = num_sms;
    double best_cost = 1e300;
    for (int sp = 1; sp <= tpg::stream::MAX_SPLIT && sp <= kb; ++sp) {
        if (tpg::stream::max_stages(mt_pad, sp) < 4) continue;
        const int c = sp == 1 ? num_sms : clusters[sp - 2];
        if (c < 1) continue;
        const int64_t rounds = (nt + c - 1) / c;
        const double cost = static_cast<double>(rounds) / sp * (1.0 + 0.02 * (sp - 1));
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            best_s = sp;
            best_clusters = c;
        }
    }
    if (clusters_used) *clusters_used = best_clusters;
    return best_s;
}

int stream_clusters_for(tpgemm_handle *h, bool f32, int mt, int stages, int split) {
    std::atomic<int> &slot = h->stream_clusters[f32 ? 1 : 0][split - 2][mt / 16 - 1];
    const int cached = slot.load(std::memory_order_relaxed);
    if (cached > 0) return cached;
    const int n = tpg::stream_split_clusters(f32, h->num_sms,
                                             static_cast<int>(tpg::stream::smem_bytes(mt, stages, split)), split);
    const int v = n > 0 ? n : h->num_sms / split;
    slot.store(v, std::memory_order_relaxed);
    return v;
}

int pair_clusters_for(tpgemm_handle *h, bool f32) {
    std::atomic<int> &slot = h->pair_clusters[f32 ? 1 : 0];
    const int cached = slot.load(std::memory_order_relaxed);
    if (cached > 0) return cached;
    const int n = tpg::tiled_clusters(true, f32, h->num_sms, 2);
    const int v = n > 0 ? n : h->num_sms / 2;
    slot.store(v, std::memory_order_relaxed);
    return v;
}

// K split of the tiled kernel's 1-CTA mode for `tiles` 128 x 256 tiles of kb K
// blocks: 4 when every tile gets a cluster of four CTAs at once (cap4 such
// clusters fit) and kb >= 4, else 2 under the same conditions, else 1 (the
// persistent schedule). Few tiles for many SMs is a short M with a narrow N;
// there, rather than cut tiles into narrow column pieces, whose small MMAs run
// far below the tensor pipe's rate, the CTAs of a cluster share each tile's K
// range and exchange partial sums through distributed shared memory.
int tiled_ksplit_choice(int64_t tiles, int64_t kb, int cap2, int cap4) {
    if (kb >= 4 && tiles <= cap4) return 4;
    if (kb >= 2 && tiles <= cap2) return 2;
    return 1;
}

int ks_clusters_for(tpgemm_handle *h, bool f32, int split) {
    std::atomic<int> &slot = h->ks_clusters[f32 ? 1 : 0][split == 4 ? 1 : 0];
    const int cached = slot.load(std::memory_order_relaxed);
    if (cached > 0) return cached;
    const int n = tpg::tiled_clusters(false, f32, h->num_sms, split);
    const int v = n > 0 ? n : h->num_sms / split;
    slot.store(v, std::memory_order_relaxed);
    return v;
}

Plan make_plan(tpgemm_handle *h, int64_t M, int64_t N, int64_t K, int out_dtype) {
    Plan pl;
    if (M == 0 || N == 0) return pl;
    if (K == 0) {
        pl.variant = TPGEMM_VARIANT_EPILOGUE_ONLY;
        const int64_t total = M * N;
        int64_t blocks = (total + 1023) / 1024;
        if (blocks > 8LL * h->num_sms) blocks = 8LL * h->num_sms;
        pl.grid = static_cast<int>(blocks < 1 ? 1 : blocks);
        pl.launches = 1;
        return pl;
    }
    int variant = h->forced;
    if (variant == TPGEMM_VARIANT_AUTO)
        variant = M <= kStreamMaxM ? TPGEMM_VARIANT_STREAM
                  : M <= tpg::tiled::BM ? TPGEMM_VARIANT_TILED
                                        : TPGEMM_VARIANT_TILED_PAIR;
    if (variant == TPGEMM_VARIANT_STREAM && M > kStreamMaxM) variant = TPGEMM_VARIANT_TILED;
    pl.variant = variant;
    pl.launches = 1;
    if (variant == TPGEMM_VARIANT_TILED || variant == TPGEMM_VARIANT_TILED_PAIR) {
        const bool f32 = out_dtype == TPGEMM_OUT_F32;
        // K split of 1-CTA tiles (tiled_ksplit_choice); the automatic choice only.
        if (h->forced == TPGEMM_VARIANT_AUTO) {
            const int64_t kbt = (K + tpg::tiled::BK - 1) / tpg::tiled::BK;
            const int64_t tiles1 = ((M + tpg::tiled::BM - 1) / tpg::tiled::BM) * ((N + tpg::tiled::BN - 1) / tpg::tiled::BN);
            const int ks = tiled_ksplit_choice(tiles1, kbt, ks_clusters_for(h, f32, 2), ks_clusters_for(h, f32, 4));
            if (ks > 1) {
                pl.variant = TPGEMM_VARIANT_TILED;
                pl.ksplit = ks;
                pl.tile_m = tpg::tiled::BM;
                pl.tile_n = tpg::tiled::BN;
                pl.num_tiles = tiles1;
                pl.cluster = ks;
                pl.sched = tiled_schedule((M + tpg::tiled::BM - 1) / tpg::tiled::BM,
                                          (N + tpg::tiled::BN - 1) / tpg::tiled::BN, tiles1, false, false);
                pl.grid = static_cast<int>(pl.sched.workers * ks);
                pl.split = 1;
                pl.smem = static_cast<int>(tpg::tiled::Layout<false>::SMEM_BYTES);
                return pl;
            }
        }
        const bool pair = variant == TPGEMM_VARIANT_TILED_PAIR;
        const int64_t rows = tpg::tiled::BM * (pair ? 2 : 1);
        const int64_t mt = (M + rows - 1) / rows;
        const int64_t nt = (N + tpg::tiled::BN - 1) / tpg::tiled::BN;
        pl.tile_m = static_cast<int>(rows);
        pl.tile_n = tpg::tiled::BN;
        pl.num_tiles = mt * nt;
        const int64_t cap = pair ? pair_clusters_for(h, out_dtype == TPGEMM_OUT_F32) : h->num_sms;
        pl.cluster = pair ? 2 : 1;
        pl.sched = tiled_schedule(mt, nt, cap, pair, true);
        pl.grid = static_cast<int>(pl.sched.workers * pl.cluster);
        pl.split = pl.sched.split;
        pl.smem = static_cast<int>(pair ? tpg::tiled::Layout<true>::SMEM_BYTES : tpg::tiled::Layout<false>::SMEM_BYTES);
        // With a workspace, the halves of the last partial round become K halves
        // over the whole tile width (tiled::item_krange): a piece then takes half
        // of a tile's K blocks, where a column half takes all of them. Only for
        // K of at least kTailMinKb blocks, where that outweighs the exchange.
        const int64_t kbt = (K + tpg::tiled::BK - 1) / tpg::tiled::BK;
        if (pair && h->ws && tail_ksplit_choice(pl.sched.split, kbt, pl.sched.pieces / 2, h->ws_bytes))
            pl.ktail = 1;
        return pl;
    }
    // weight-streaming variant
    const int mt_pad = static_cast<int>((M + 15) / 16 * 16);
    const int64_t kb = (K + tpg::stream::BK - 1) / tpg::stream::BK;
    const int64_t nt = (N + tpg::stream::BN - 1) / tpg::stream::BN;
    pl.tile_m = static_cast<int>(M);
    pl.tile_n = tpg::stream::BN;
    pl.num_tiles = nt;
    pl.mt_pad = mt_pad;
    const bool f32 = out_dtype == TPGEMM_OUT_F32;
    int clusters[tpg::stream::MAX_SPLIT - 1];
    for (int sp = 2; sp <= tpg::stream::MAX_SPLIT; ++sp) {
        const int st = tpg::stream::max_stages(mt_pad, sp);
        clusters[sp - 2] = st >= 4 && sp <= kb ? stream_clusters_for(h, f32, mt_pad, st, sp) : 0;
    }
    int best_clusters = h->num_sms;
    const int best_s = stream_split_choice(nt, kb, mt_pad, h->num_sms, clusters, &best_clusters);
    pl.split = best_s;
    pl.stages = tpg::stream::max_stages(mt_pad, pl.split);
    pl.smem = static_cast<int>(tpg::stream::smem_bytes(mt_pad, pl.stages, pl.split));
    const int64_t c = nt < best_clusters ? nt : best_clusters;
    pl.grid = static_cast<int>(pl.split * c);
    pl.cluster = pl.split;
    return pl;
}

// Launches one of the small kernels of this file (no PDL, no cluster).
template <typename Kernel, typename... Args>
int launch(Kernel kernel, int grid, int block, int smem, int cluster, cudaStream_t stream, Args... args) {
    return tpg::launch_ex(kernel, grid, block, smem, cluster, false, stream, args...) == cudaSuccess
               ? TPGEMM_OK
               : TPGEMM_ERR_CUDA;
}

// Opts every GEMM instantiation into its dynamic shared-memory size (current device).
bool set_smem_limits() {
    bool ok = tpg::tiled_set_limits_e0();
    ok = tpg::tiled_set_limits_g0() && ok;
    ok = tpg::tiled_set_limits_e1() && ok;
    ok = tpg::tiled_set_limits_e2() && ok;
    ok = tpg::tiled_set_limits_e3() && ok;
    ok = tpg::tiled_set_limits_e4() && ok;
    ok = tpg::tiled_set_limits_e5() && ok;
    ok = tpg::stream_set_limits() && ok;
    ok = tpg::mx_set_limits() && ok;
    ok = tpg::fp4_set_limits_nv() && ok;
    ok = tpg::fp4_set_limits_mx() && ok;
    return ok;
}

// Argument checks of the fused epilogue (see tpgemm_epilogue).
int check_epilogue(int64_t M, int64_t N, const void *D, int64_t ldd, int out_dtype, const tpgemm_epilogue *e) {
    if (!e) return TPGEMM_OK;
    if (e->activation < TPGEMM_ACT_NONE || e->activation > TPGEMM_ACT_TANH) return TPGEMM_ERR_INVALID_ARG;
    const int64_t elt = out_dtype == TPGEMM_OUT_F32 ? 4 : 2;
    const Range rd = byte_range(D, M, N, ldd, elt);
    if (e->bias) {
        if (e->bias_dtype != TPGEMM_OUT_BF16 && e->bias_dtype != TPGEMM_OUT_F32) return TPGEMM_ERR_INVALID_ARG;
        if (!aligned16(e->bias)) return TPGEMM_ERR_ALIGNMENT;
        if (overlaps(rd, byte_range(e->bias, 1, N, N, e->bias_dtype == TPGEMM_OUT_F32 ? 4 : 2)))
            return TPGEMM_ERR_OVERLAP;
    }
    if (e->aux) {
        if (e->ldaux < N) return TPGEMM_ERR_INVALID_ARG;
        if (!aligned16(e->aux) || (M > 1 && (e->ldaux * elt) % 16 != 0)) return TPGEMM_ERR_ALIGNMENT;
        if (!(e->aux == D && e->ldaux == ldd) && overlaps(rd, byte_range(e->aux, M, N, e->ldaux, elt)))
            return TPGEMM_ERR_OVERLAP;
    }
    return TPGEMM_OK;
}

tpg::EpiParams epi_params(const tpgemm_epilogue *e) {
    tpg::EpiParams p{};
    if (e) {
        p.bias = e->bias;
        p.bias_f32 = e->bias_dtype == TPGEMM_OUT_F32 ? 1 : 0;
        p.act = e->activation;
        p.aux = e->aux;
        p.ldaux = e->ldaux;
    }
    return p;
}

// Launches the tiled kernel in fused-epilogue mode `mode` (0 plain, 1 + activation).
int launch_tiled(int mode, const tpg::TiledLaunch &l) {
    cudaError_t e;
    switch (mode) {
    case 1: e = tpg::tiled_launch_e1(l); break;
    case 2: e = tpg::tiled_launch_e2(l); break;
    case 3: e = tpg::tiled_launch_e3(l); break;
    case 4: e = tpg::tiled_launch_e4(l); break;
    case tpg::tiled::kEpiUnitAlpha: e = tpg::tiled_launch_e5(l); break;
    default: e = tpg::tiled_launch_e0(l); break;
    }
    return e == cudaSuccess ? TPGEMM_OK : TPGEMM_ERR_CUDA;
}

int run_impl(tpgemm_handle *h, int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B,
             int64_t ldb, const void *C, int64_t ldc, void *D, int64_t ldd, float alpha, float beta, int out_dtype,
             const tpgemm_epilogue *epi, void *stream_ptr);

} // namespace

extern "C" {

const char *gemm_status_string(int status) {
    switch (status) {
    case TPGEMM_OK: return "TPGEMM_OK";
    case TPGEMM_ERR_INVALID_ARG: return "TPGEMM_ERR_INVALID_ARG";
    case TPGEMM_ERR_ALIGNMENT: return "TPGEMM_ERR_ALIGNMENT";
    case TPGEMM_ERR_OVERLAP: return "TPGEMM_ERR_OVERLAP";
    case TPGEMM_ERR_UNSUPPORTED_DEVICE: return "TPGEMM_ERR_UNSUPPORTED_DEVICE";
    case TPGEMM_ERR_CUDA: return "TPGEMM_ERR_CUDA";
    case TPGEMM_ERR_TIMEOUT: return "TPGEMM_ERR_TIMEOUT";
    case TPGEMM_ERR_TOO_LARGE: return "TPGEMM_ERR_TOO_LARGE";
    default: return "TPGEMM_ERR_UNKNOWN";
    }
}

int gemm_create(tpgemm_handle **out, int device) {
    if (!out) return TPGEMM_ERR_INVALID_ARG;
    *out = nullptr;
    int count = 0;
    if (cudaGetDeviceCount(&count) != cudaSuccess) {
        (void)cudaGetLastError();
        return TPGEMM_ERR_CUDA;
    }
    if (device < 0 || device >= count) return TPGEMM_ERR_INVALID_ARG;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return TPGEMM_ERR_CUDA;
    if (prop.major != 10 || prop.minor != 3) return TPGEMM_ERR_UNSUPPORTED_DEVICE;

    tpgemm_handle *h = new (std::nothrow) tpgemm_handle();
    if (!h) return TPGEMM_ERR_CUDA;
    h->device = device;
    h->num_sms = prop.multiProcessorCount;
    if (const char *env = std::getenv("TPGEMM_WATCHDOG_NS")) {
        const unsigned long long v = std::strtoull(env, nullptr, 10);
        if (v >= 1000ull && v <= 60000000000ull) h->timeout_ns = v;
    }
    DeviceGuard guard(device);
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn) {
        delete h;
        return TPGEMM_ERR_CUDA;
    }
    h->encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    const bool ok = set_smem_limits();
    if (!ok || cudaMalloc(&h->status, sizeof(uint64_t)) != cudaSuccess ||
        cudaMemset(h->status, 0, sizeof(uint64_t)) != cudaSuccess) {
        (void)cudaGetLastError();
        if (h->status) cudaFree(h->status);
        delete h;
        return TPGEMM_ERR_CUDA;
    }
    *out = h;
    return TPGEMM_OK;
}

int gemm_destroy(tpgemm_handle *h) {
    if (!h) return TPGEMM_OK;
    int rc = TPGEMM_OK;
    {
        DeviceGuard guard(h->device);
        if (h->status && cudaFree(h->status) != cudaSuccess) rc = TPGEMM_ERR_CUDA;
    }
    delete h;
    return rc;
}

int gemm_num_sms(tpgemm_handle *h) { return h ? h->num_sms : TPGEMM_ERR_INVALID_ARG; }

int64_t gemm_workspace_size(tpgemm_handle *h) {
    if (!h) return TPGEMM_ERR_INVALID_ARG;
    // at most one tail tile per two CTA pairs
    return tail_ws_bytes(h->num_sms / 4);
}

int gemm_set_workspace(tpgemm_handle *h, void *ws, int64_t bytes, void *stream_ptr) {
    if (!h) return TPGEMM_ERR_INVALID_ARG;
    if (!ws) {
        h->ws = nullptr;
        h->ws_bytes = 0;
        return TPGEMM_OK;
    }
    if (bytes < tail_ws_bytes(1)) return TPGEMM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return TPGEMM_ERR_ALIGNMENT;
    DeviceGuard guard(h->device);
    // every flag starts clear; calls enqueued after this on the same stream see it
    if (cudaMemsetAsync(ws, 0, tpg::tiled::kTailFlagBytes, static_cast<cudaStream_t>(stream_ptr)) != cudaSuccess)
        return TPGEMM_ERR_CUDA;
    h->ws = ws;
    h->ws_bytes = bytes;
    return TPGEMM_OK;
}

int gemm_plan_tail_ksplit(tpgemm_handle *h, int64_t M, int64_t N, int64_t K, int out_dtype) {
    if (!h || M < 0 || N < 0 || K < 0) return TPGEMM_ERR_INVALID_ARG;
    if (out_dtype != TPGEMM_OUT_BF16 && out_dtype != TPGEMM_OUT_F32) return TPGEMM_ERR_INVALID_ARG;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return TPGEMM_ERR_TOO_LARGE;
    DeviceGuard guard(h->device);
    return make_plan(h, M, N, K, out_dtype).ktail;
}

int gemm_force_variant(tpgemm_handle *h, int variant) {
    if (!h) return TPGEMM_ERR_INVALID_ARG;
    if (variant != TPGEMM_VARIANT_AUTO && variant != TPGEMM_VARIANT_TILED && variant != TPGEMM_VARIANT_STREAM &&
        variant != TPGEMM_VARIANT_TILED_PAIR)
        return TPGEMM_ERR_INVALID_ARG;
    h->forced = variant;
    return TPGEMM_OK;
}

int gemm_query_plan(tpgemm_handle *h, int64_t M, int64_t N, int64_t K, int out_dtype, int *variant,
                    int *tile_m, int *tile_n, int64_t *num_tiles, int *grid, int *cluster, int *smem_bytes,
                    int *launches) {
    if (!h || M < 0 || N < 0 || K < 0) return TPGEMM_ERR_INVALID_ARG;
    if (out_dtype != TPGEMM_OUT_BF16 && out_dtype != TPGEMM_OUT_F32) return TPGEMM_ERR_INVALID_ARG;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return TPGEMM_ERR_TOO_LARGE;
    DeviceGuard guard(h->device);
    const Plan pl = make_plan(h, M, N, K, out_dtype);
    if (variant) *variant = pl.variant;
    if (tile_m) *tile_m = pl.tile_m;
    if (tile_n) *tile_n = pl.tile_n;
    if (num_tiles) *num_tiles = pl.num_tiles;
    if (grid) *grid = pl.grid;
    if (cluster) *cluster = pl.cluster;
    if (smem_bytes) *smem_bytes = pl.smem;
    if (launches) *launches = pl.launches;
    return TPGEMM_OK;
}

int gemm_stream_split(int64_t nt, int64_t kb, int mt_pad, int num_sms, const int *clusters) {
    if (nt < 1 || kb < 1 || mt_pad < 16 || mt_pad > 64 || mt_pad % 16 != 0 || num_sms < 1 || !clusters)
        return TPGEMM_ERR_INVALID_ARG;
    return stream_split_choice(nt, kb, mt_pad, num_sms, clusters, nullptr);
}

int gemm_tail_ksplit(int split, int64_t kb, int64_t tail_tiles, int64_t ws_bytes) {
    if (split < 1 || kb < 1 || tail_tiles < 0 || ws_bytes < 0) return TPGEMM_ERR_INVALID_ARG;
    return tail_ksplit_choice(split, kb, tail_tiles, ws_bytes) ? 1 : 0;
}

int64_t gemm_tail_workspace_bytes(int64_t tail_tiles) {
    if (tail_tiles < 0) return TPGEMM_ERR_INVALID_ARG;
    return tail_ws_bytes(tail_tiles);
}

int gemm_tiled_ksplit(int64_t tiles, int64_t kb, int cap2, int cap4) {
    if (tiles < 1 || kb < 1 || cap2 < 0 || cap4 < 0) return TPGEMM_ERR_INVALID_ARG;
    return tiled_ksplit_choice(tiles, kb, cap2, cap4);
}

int gemm_schedule_workers(int64_t mt, int64_t nt, int cap, int pair, int allow_split) {
    if (mt < 0 || nt < 0 || cap < 1) return TPGEMM_ERR_INVALID_ARG;
    return static_cast<int>(tiled_schedule(mt, nt, cap, pair != 0, allow_split != 0).workers);
}

int64_t gemm_schedule_tiles(int64_t mt, int64_t nt, int group_m, int cap, int pair, int allow_split, int worker,
                            int32_t *out, int64_t cap_items) {
    if (mt < 0 || nt < 0 || group_m < 1 || cap < 1 || worker < 0 || cap_items < 0 || (cap_items > 0 && !out))
        return TPGEMM_ERR_INVALID_ARG;
    tpg::Schedule s = tiled_schedule(mt, nt, cap, pair != 0, allow_split != 0);
    s.group_m = group_m;
    if (worker >= s.workers) return 0;
    int64_t count = 0;
    tpg::WorkItem w;
    for (int64_t t = worker; tpg::work_item(s, t, tpg::tiled::BN, w); t += s.workers, ++count) {
        if (count < cap_items) {
            out[3 * count] = w.m;
            out[3 * count + 1] = w.n;
            out[3 * count + 2] = w.width;
        }
    }
    return count;
}

int gemm_check_args(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B, int64_t ldb,
                    const void *C, int64_t ldc, const void *D, int64_t ldd, float beta, int out_dtype) {
    if (out_dtype != TPGEMM_OUT_BF16 && out_dtype != TPGEMM_OUT_F32) return TPGEMM_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K < 0) return TPGEMM_ERR_INVALID_ARG;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return TPGEMM_ERR_TOO_LARGE;
    if (M == 0 || N == 0) return TPGEMM_OK;
    const int64_t elt = out_dtype == TPGEMM_OUT_F32 ? 4 : 2;
    const bool use_c = beta != 0.0f;
    // shapes and strides
    if (!D || ldd < N) return TPGEMM_ERR_INVALID_ARG;
    if (K > 0 && (!A || !B || lda < K || ldb < N)) return TPGEMM_ERR_INVALID_ARG;
    if (use_c && (!C || ldc < N)) return TPGEMM_ERR_INVALID_ARG;
    if (ldd > kMaxDim * 8 || (K > 0 && (lda > kMaxDim * 8 || ldb > kMaxDim * 8)) || (use_c && ldc > kMaxDim * 8))
        return TPGEMM_ERR_TOO_LARGE;
    // alignment (TMA: 16-byte base addresses and 16-byte multiple row strides)
    if (!aligned16(D) || (M > 1 && (ldd * elt) % 16 != 0)) return TPGEMM_ERR_ALIGNMENT;
    if (K > 0) {
        if (!aligned16(A) || !aligned16(B)) return TPGEMM_ERR_ALIGNMENT;
        if (M > 1 && (lda * 2) % 16 != 0) return TPGEMM_ERR_ALIGNMENT;
        if (K > 1 && (ldb * 2) % 16 != 0) return TPGEMM_ERR_ALIGNMENT;
    }
    if (use_c && (!aligned16(C) || (M > 1 && (ldc * elt) % 16 != 0))) return TPGEMM_ERR_ALIGNMENT;
    // overlap: D is written, so it may not share bytes with an input, except
    // the exact in-place case D == C with the same row stride.
    const Range rd = byte_range(D, M, N, ldd, elt);
    if (K > 0 && (overlaps(rd, byte_range(A, M, K, lda, 2)) || overlaps(rd, byte_range(B, K, N, ldb, 2))))
        return TPGEMM_ERR_OVERLAP;
    if (use_c && !(C == D && ldc == ldd) && overlaps(rd, byte_range(C, M, N, ldc, elt)))
        return TPGEMM_ERR_OVERLAP;
    return TPGEMM_OK;
}

int gemm_run(tpgemm_handle *h, int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B,
             int64_t ldb, const void *C, int64_t ldc, void *D, int64_t ldd, float alpha, float beta,
             int out_dtype, void *stream_ptr) {
    return run_impl(h, M, N, K, A, lda, B, ldb, C, ldc, D, ldd, alpha, beta, out_dtype, nullptr, stream_ptr);
}

int gemm_run_epilogue(tpgemm_handle *h, int64_t M, int64_t N, int64_t K, const void *A, int64_t lda,
                      const void *B, int64_t ldb, const void *C, int64_t ldc, void *D, int64_t ldd, float alpha,
                      float beta, int out_dtype, const tpgemm_epilogue *epi, void *stream_ptr) {
    return run_impl(h, M, N, K, A, lda, B, ldb, C, ldc, D, ldd, alpha, beta, out_dtype, epi, stream_ptr);
}

} // extern "C"

namespace {

int run_impl(tpgemm_handle *h, int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B,
             int64_t ldb, const void *C, int64_t ldc, void *D, int64_t ldd, float alpha, float beta, int out_dtype,
             const tpgemm_epilogue *epi, void *stream_ptr) {
    if (!h) return TPGEMM_ERR_INVALID_ARG;
    int chk = gemm_check_args(M, N, K, A, lda, B, ldb, C, ldc, D, ldd, beta, out_dtype);
    if (chk == TPGEMM_OK && M > 0 && N > 0) chk = check_epilogue(M, N, D, ldd, out_dtype, epi);
    if (chk != TPGEMM_OK || M == 0 || N == 0) return chk;
    const bool fused = epi && (epi->bias || epi->aux || epi->activation != TPGEMM_ACT_NONE);
    const tpg::EpiParams ep = epi_params(epi);
    const int64_t elt = out_dtype == TPGEMM_OUT_F32 ? 4 : 2;
    const bool use_c = beta != 0.0f;

    DeviceGuard guard(h->device);
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    const Plan pl = make_plan(h, M, N, K, out_dtype);
    const bool f32 = out_dtype == TPGEMM_OUT_F32;

    if (pl.variant == TPGEMM_VARIANT_EPILOGUE_ONLY) {
        const int32_t m = static_cast<int32_t>(M), n = static_cast<int32_t>(N);
        const void *c = use_c ? C : nullptr;
        if (fused)
            return f32 ? launch(tpg::epilogue_only_kernel<true, true>, pl.grid, 256, 0, 1, stream, m, n, beta, c, ldc,
                                D, ldd, ep)
                       : launch(tpg::epilogue_only_kernel<false, true>, pl.grid, 256, 0, 1, stream, m, n, beta, c,
                                ldc, D, ldd, ep);
        return f32 ? launch(tpg::epilogue_only_kernel<true, false>, pl.grid, 256, 0, 1, stream, m, n, beta, c, ldc, D,
                            ldd, ep)
                   : launch(tpg::epilogue_only_kernel<false, false>, pl.grid, 256, 0, 1, stream, m, n, beta, c, ldc,
                            D, ldd, ep);
    }

    CUtensorMap tmA, tmB;
    if (pl.variant == TPGEMM_VARIANT_TILED || pl.variant == TPGEMM_VARIANT_TILED_PAIR) {
        CUtensorMap tmB1, tmC, tmD;
        tpg::TiledParams p;
        const TiledCall call{M, N, K, 1, 1, A, lda, 0, B, ldb, 0, C, ldc, 0, D, ldd, 0, alpha, beta, f32};
        if (build_tiled(h->encode, call, &tmA, &tmB, &tmB1, &tmC, &tmD, &p) != TPGEMM_OK) return TPGEMM_ERR_CUDA;
        p.sched = pl.sched;
        p.mt_batch = static_cast<int32_t>(pl.sched.mt);
        p.ksplit = pl.ksplit;
        p.status = h->status;
        p.timeout_ns = h->timeout_ns;
        p.epi = ep;
        if (pl.ktail) {
            // The kernel writes the workspace: it may not share bytes with an operand.
            const Range rw{reinterpret_cast<uintptr_t>(h->ws), reinterpret_cast<uintptr_t>(h->ws) +
                                                                   static_cast<uintptr_t>(tail_ws_bytes(pl.sched.pieces / 2))};
            if (overlaps(rw, byte_range(A, M, K, lda, 2)) || overlaps(rw, byte_range(B, K, N, ldb, 2)) ||
                overlaps(rw, byte_range(D, M, N, ldd, elt)) || (use_c && overlaps(rw, byte_range(C, M, N, ldc, elt))) ||
                (epi && epi->aux && overlaps(rw, byte_range(epi->aux, M, N, epi->ldaux, elt))) ||
                (epi && epi->bias && overlaps(rw, byte_range(epi->bias, 1, N, N, epi->bias_dtype == TPGEMM_OUT_F32 ? 4 : 2))))
                return TPGEMM_ERR_OVERLAP;
            uint32_t e = h->epoch.fetch_add(1u, std::memory_order_relaxed) + 1u;
            if (e == 0u) e = h->epoch.fetch_add(1u, std::memory_order_relaxed) + 1u;
            p.ktail = 1;
            p.epoch = e;
            p.ws = h->ws;
        }
        const tpg::TiledLaunch l{pl.grid, pl.smem, pl.cluster, pl.variant == TPGEMM_VARIANT_TILED_PAIR, f32, stream,
                                 &tmA, &tmB, &tmB1, &tmC, &tmD, &p, nullptr};
        return launch_tiled(fused ? 1 + ep.act : (alpha == 1.0f ? tpg::tiled::kEpiUnitAlpha : 0), l);
    }

    // weight-streaming variant
    if (encode_2d(h, &tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A, K, M, tma_stride(M, K, lda, 2), 64,
                  static_cast<uint32_t>(pl.mt_pad)) ||
        encode_2d(h, &tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, B, N, K, tma_stride(K, N, ldb, 2), 64, 64))
        return TPGEMM_ERR_CUDA;
    tpg::StreamParams p;
    p.M = static_cast<int32_t>(M);
    p.N = static_cast<int32_t>(N);
    p.K = static_cast<int32_t>(K);
    p.nt = static_cast<int32_t>(pl.num_tiles);
    p.kb = static_cast<int32_t>((K + tpg::stream::BK - 1) / tpg::stream::BK);
    p.mt_pad = pl.mt_pad;
    p.stages = pl.stages;
    p.alpha = alpha;
    p.beta = beta;
    p.C = use_c ? C : nullptr;
    p.ldc = ldc;
    p.D = D;
    p.ldd = ldd;
    p.status = h->status;
    p.timeout_ns = h->timeout_ns;
    p.epi = ep;
    const tpg::StreamLaunch l{pl.grid, pl.smem, pl.split, f32, fused, stream, &tmA, &tmB, &p};
    return tpg::stream_launch(l) == cudaSuccess ? TPGEMM_OK : TPGEMM_ERR_CUDA;
}

} // namespace

extern "C" {

int gemm_run_batched(tpgemm_handle *h, int64_t batch, int64_t M, int64_t N, int64_t K, const void *A, int64_t lda,
                     int64_t sA, const void *B, int64_t ldb, int64_t sB, const void *C, int64_t ldc, int64_t sC,
                     void *D, int64_t ldd, int64_t sD, float alpha, float beta, int out_dtype, void *stream_ptr) {
    if (!h) return TPGEMM_ERR_INVALID_ARG;
    if (batch < 0 || sA < 0 || sB < 0 || sC < 0 || sD < 0) return TPGEMM_ERR_INVALID_ARG;
    int chk = gemm_check_args(M, N, K, A, lda, B, ldb, C, ldc, D, ldd, beta, out_dtype);
    if (chk != TPGEMM_OK || batch == 0 || M == 0 || N == 0) return chk;
    if (batch > kMaxDim || batch * ((M + tpg::tiled::BM - 1) / tpg::tiled::BM) > kMaxDim) return TPGEMM_ERR_TOO_LARGE;
    const bool f32 = out_dtype == TPGEMM_OUT_F32;
    const int64_t elt = f32 ? 4 : 2;
    const bool use_c = beta != 0.0f;
    if (batch > 1) {
        if ((sA * 2) % 16 || (sB * 2) % 16 || (use_c && (sC * elt) % 16) || (sD * elt) % 16)
            return TPGEMM_ERR_ALIGNMENT;
        if (sD < (M - 1) * ldd + N) return TPGEMM_ERR_OVERLAP; // D slices must be disjoint
        // every byte any slice of D touches, against every byte any slice of an input touches
        const uintptr_t dlo = reinterpret_cast<uintptr_t>(D);
        const Range rd_all{dlo, dlo + static_cast<uintptr_t>(((batch - 1) * sD + (M - 1) * ldd + N) * elt)};
        auto extent = [&](const void *ptr, int64_t rows, int64_t cols, int64_t ld, int64_t st, int64_t e) {
            const uintptr_t lo = reinterpret_cast<uintptr_t>(ptr);
            return Range{lo, lo + static_cast<uintptr_t>(((batch - 1) * st + (rows - 1) * ld + cols) * e)};
        };
        if (K > 0 && (overlaps(rd_all, extent(A, M, K, lda, sA, 2)) || overlaps(rd_all, extent(B, K, N, ldb, sB, 2))))
            return TPGEMM_ERR_OVERLAP;
        if (use_c && !(C == D && ldc == ldd && sC == sD) && overlaps(rd_all, extent(C, M, N, ldc, sC, elt)))
            return TPGEMM_ERR_OVERLAP;
    }
    DeviceGuard guard(h->device);
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    if (K == 0) {
        // D_b = beta * C_b, one small launch per slice
        int64_t blocks = (M * N + 1023) / 1024;
        if (blocks > 8LL * h->num_sms) blocks = 8LL * h->num_sms;
        const tpg::EpiParams none{};
        for (int64_t b = 0; b < batch; ++b) {
            const void *cb = use_c ? static_cast<const char *>(C) + b * sC * elt : nullptr;
            void *db = static_cast<char *>(D) + b * sD * elt;
            const int32_t m = static_cast<int32_t>(M), n = static_cast<int32_t>(N);
            const int rc = f32 ? launch(tpg::epilogue_only_kernel<true, false>, static_cast<int>(blocks), 256, 0, 1,
                                        stream, m, n, beta, cb, ldc, db, ldd, none)
                               : launch(tpg::epilogue_only_kernel<false, false>, static_cast<int>(blocks), 256, 0, 1,
                                        stream, m, n, beta, cb, ldc, db, ldd, none);
            if (rc != TPGEMM_OK) return rc;
        }
        return TPGEMM_OK;
    }
    const bool pair = M > tpg::tiled::BM;
    const int64_t rows_per_tile = tpg::tiled::BM * (pair ? 2 : 1);
    const int64_t mt = (M + rows_per_tile - 1) / rows_per_tile;
    const int64_t nt = (N + tpg::tiled::BN - 1) / tpg::tiled::BN;
    const int64_t cap = pair ? pair_clusters_for(h, f32) : h->num_sms;
    CUtensorMap tmA, tmB, tmB1, tmC, tmD;
    tpg::TiledParams p;
    const TiledCall call{M, N, K, batch, batch, A, lda, sA, B, ldb, sB, C, ldc, sC, D, ldd, sD, alpha, beta, f32};
    if (build_tiled(h->encode, call, &tmA, &tmB, &tmB1, &tmC, &tmD, &p) != TPGEMM_OK) return TPGEMM_ERR_CUDA;
    p.sched = tiled_schedule(mt * batch, nt, cap, pair, true);
    p.mt_batch = static_cast<int32_t>(mt);
    p.status = h->status;
    p.timeout_ns = h->timeout_ns;
    const int smem = static_cast<int>(pair ? tpg::tiled::Layout<true>::SMEM_BYTES : tpg::tiled::Layout<false>::SMEM_BYTES);
    const tpg::TiledLaunch l{static_cast<int>(p.sched.workers * (pair ? 2 : 1)), smem, pair ? 2 : 1, pair, f32, stream,
                             &tmA, &tmB, &tmB1, &tmC, &tmD, &p, nullptr};
    return launch_tiled(p.alpha == 1.0f ? tpg::tiled::kEpiUnitAlpha : 0, l);
}

int gemm_run_grouped(tpgemm_handle *h, int64_t groups, const int64_t *group_rows, int64_t N, int64_t K,
                     const void *A, int64_t lda, const void *B, int64_t ldb, int64_t sB, const void *C, int64_t ldc,
                     void *D, int64_t ldd, float alpha, float beta, int out_dtype, void *stream_ptr) {
    if (!h || groups < 0 || sB < 0 || (groups > 0 && !group_rows)) return TPGEMM_ERR_INVALID_ARG;
    if (groups > TPGEMM_MAX_GROUPS) return TPGEMM_ERR_TOO_LARGE;
    int64_t total = 0;
    for (int64_t g = 0; g < groups; ++g) {
        if (group_rows[g] < 0) return TPGEMM_ERR_INVALID_ARG;
        total += group_rows[g];
        if (total > kMaxDim) return TPGEMM_ERR_TOO_LARGE;
    }
    int chk = gemm_check_args(total, N, K, A, lda, B, ldb, C, ldc, D, ldd, beta, out_dtype);
    if (chk != TPGEMM_OK || total == 0 || N == 0) return chk;
    const bool f32 = out_dtype == TPGEMM_OUT_F32;
    const int64_t elt = f32 ? 4 : 2;
    if (groups > 1 && K > 0) {
        if ((sB * 2) % 16) return TPGEMM_ERR_ALIGNMENT;
        const uintptr_t lo = reinterpret_cast<uintptr_t>(B);
        const Range rb{lo, lo + static_cast<uintptr_t>(((groups - 1) * sB + (K - 1) * ldb + N) * 2)};
        if (overlaps(byte_range(D, total, N, ldd, elt), rb)) return TPGEMM_ERR_OVERLAP;
    }
    DeviceGuard guard(h->device);
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    const bool use_c = beta != 0.0f;
    if (K == 0) {
        int64_t blocks = (total * N + 1023) / 1024;
        if (blocks > 8LL * h->num_sms) blocks = 8LL * h->num_sms;
        const tpg::EpiParams none{};
        const int32_t m = static_cast<int32_t>(total), n = static_cast<int32_t>(N);
        const void *c = use_c ? C : nullptr;
        return f32 ? launch(tpg::epilogue_only_kernel<true, false>, static_cast<int>(blocks), 256, 0, 1, stream, m, n,
                            beta, c, ldc, D, ldd, none)
                   : launch(tpg::epilogue_only_kernel<false, false>, static_cast<int>(blocks), 256, 0, 1, stream, m,
                            n, beta, c, ldc, D, ldd, none);
    }
    // CTA pairs when groups are large enough on average to fill 256-row tiles
    const bool pair = total > static_cast<int64_t>(tpg::tiled::BM) * groups;
    const int32_t rows_per_tile = tpg::tiled::BM * (pair ? 2 : 1);
    tpg::GroupTable table{};
    table.groups = static_cast<int32_t>(groups);
    int64_t row = 0, tiles = 0;
    for (int64_t g = 0; g < groups; ++g) {
        table.tile_prefix[g] = static_cast<int32_t>(tiles);
        table.row_start[g] = static_cast<int32_t>(row);
        table.rows[g] = static_cast<int32_t>(group_rows[g]);
        row += group_rows[g];
        tiles += (group_rows[g] + rows_per_tile - 1) / rows_per_tile;
    }
    table.tile_prefix[groups] = static_cast<int32_t>(tiles);
    const int64_t nt = (N + tpg::tiled::BN - 1) / tpg::tiled::BN;
    const int64_t cap = pair ? pair_clusters_for(h, f32) : h->num_sms;
    CUtensorMap tmA, tmB, tmB1, tmC, tmD;
    tpg::TiledParams p;
    const TiledCall call{total, N, K, 1, groups, A, lda, 0, B, ldb, groups > 1 ? sB : 0, C, ldc, 0, D, ldd, 0,
                         alpha, beta, f32};
    if (build_tiled(h->encode, call, &tmA, &tmB, &tmB1, &tmC, &tmD, &p) != TPGEMM_OK) return TPGEMM_ERR_CUDA;
    p.sched = tiled_schedule(tiles, nt, cap, pair, true);
    p.mt_batch = 1;
    p.status = h->status;
    p.timeout_ns = h->timeout_ns;
    const int smem = static_cast<int>(pair ? tpg::tiled::Layout<true>::SMEM_BYTES : tpg::tiled::Layout<false>::SMEM_BYTES);
    const tpg::TiledLaunch l{static_cast<int>(p.sched.workers * (pair ? 2 : 1)), smem, pair ? 2 : 1, pair, f32, stream,
                             &tmA, &tmB, &tmB1, &tmC, &tmD, &p, &table};
    return tpg::tiled_launch_g0(l) == cudaSuccess ? TPGEMM_OK : TPGEMM_ERR_CUDA;
}

int gemm_run_chunked(tpgemm_handle *h, int chunks, int64_t M, int64_t N, int64_t K, const void *A, int64_t lda,
                     const void *B, int64_t ldb, const void *C, int64_t ldc, void *D, int64_t ldd, float alpha,
                     float beta, int out_dtype, void *const *events, void *stream_ptr) {
    if (!h || chunks < 1 || chunks > 64 || !events) return TPGEMM_ERR_INVALID_ARG;
    for (int i = 0; i < chunks; ++i)
        if (!events[i]) return TPGEMM_ERR_INVALID_ARG;
    const int chk = gemm_check_args(M, N, K, A, lda, B, ldb, C, ldc, D, ldd, beta, out_dtype);
    if (chk != TPGEMM_OK) return chk;
    const int64_t elt = out_dtype == TPGEMM_OUT_F32 ? 4 : 2;
    const bool use_c = beta != 0.0f;
    DeviceGuard guard(h->device);
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    int64_t r0 = 0;
    for (int i = 0; i < chunks; ++i) {
        const int64_t r1 = (i == chunks - 1) ? M : (static_cast<int64_t>(i + 1) * M / chunks) / 128 * 128;
        const int64_t rows = r1 > r0 ? r1 - r0 : 0;
        if (rows > 0 && N > 0) {
            // row offsets are multiples of 128, so every chunk keeps the 16-byte alignment of the whole
            const void *a = K > 0 ? static_cast<const char *>(A) + r0 * lda * 2 : A;
            const void *c = use_c ? static_cast<const char *>(C) + r0 * ldc * elt : C;
            void *d = static_cast<char *>(D) + r0 * ldd * elt;
            const int rc = run_impl(h, rows, N, K, a, lda, B, ldb, c, ldc, d, ldd, alpha, beta, out_dtype, nullptr,
                                    stream_ptr);
            if (rc != TPGEMM_OK) return rc;
        }
        if (cudaEventRecord(static_cast<cudaEvent_t>(events[i]), stream) != cudaSuccess) return TPGEMM_ERR_CUDA;
        if (r1 > r0) r0 = r1;
    }
    return TPGEMM_OK;
}

int gemm_sync_status(tpgemm_handle *h, void *stream) {
    if (!h) return TPGEMM_ERR_INVALID_ARG;
    DeviceGuard guard(h->device);
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return TPGEMM_ERR_CUDA;
    uint32_t word = 0;
    if (cudaMemcpy(&word, h->status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return TPGEMM_ERR_CUDA;
    if (word != 0) {
        if (cudaMemset(h->status, 0, sizeof(uint64_t)) != cudaSuccess) return TPGEMM_ERR_CUDA;
        return TPGEMM_ERR_TIMEOUT;
    }
    return TPGEMM_OK;
}

int gemm_watchdog_selftest(tpgemm_handle *h, uint64_t timeout_ns, void *stream_ptr) {
    if (!h || timeout_ns < 1000ull || timeout_ns > 1000000000ull) return TPGEMM_ERR_INVALID_ARG;
    DeviceGuard guard(h->device);
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    // Start from a clear word so the result reflects this launch only.
    if (cudaStreamSynchronize(stream) != cudaSuccess) return TPGEMM_ERR_CUDA;
    if (cudaMemset(h->status, 0, sizeof(uint64_t)) != cudaSuccess) return TPGEMM_ERR_CUDA;
    if (launch(tpg::watchdog_selftest_kernel, 1, 32, 0, 1, stream, h->status, timeout_ns) != TPGEMM_OK)
        return TPGEMM_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return TPGEMM_ERR_CUDA;
    uint32_t word = 0;
    if (cudaMemcpy(&word, h->status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return TPGEMM_ERR_CUDA;
    if (cudaMemset(h->status, 0, sizeof(uint64_t)) != cudaSuccess) return TPGEMM_ERR_CUDA;
    return (word & tpg::kStatusSelftest) ? TPGEMM_ERR_TIMEOUT : TPGEMM_OK;
}

} // extern "C"

// ---------------------------------------------------------------------------
// Block-scaled (MX) GEMM (gemm_run_mx).
namespace {

constexpr int64_t kMxBlock = 32;

// Bytes of one operand's scales in the blocked layout: 512-byte chunks of 128
// rows x 4 scale columns, ceil(rows / 128) x ceil(K / 128) of them.
int64_t mx_scale_bytes(int64_t rows, int64_t K) {
    return ((rows + 127) / 128) * ((K + 127) / 128) * 512;
}

// Tile width of the MX kernel: 192 columns (fewer MMAs per output, each long
// enough to hide its issue cost) unless the output is at most 128 wide.
int mx_tile_n(int64_t N) { return N > 128 ? 192 : 128; }

// CTA pairs (256 x 256 tiles) when there are more than 128 rows and columns:
// per SM they stage and read 32 KB of operands per K block for twice the
// work of a 1-CTA 128 x 192 tile's 40 KB, with MMAs wide enough to hide their
// issue cost.
bool mx_pair(int64_t M, int64_t N) { return M > 128 && N > 128; }
constexpr int kMxPairTileN = 256;

int mx_pairs_for(tpgemm_handle *h, bool f32) {
    std::atomic<int> &slot = h->mx_pairs[f32 ? 1 : 0];
    const int cached = slot.load(std::memory_order_relaxed);
    if (cached > 0) return cached;
    const int n = tpg::mx_pair_clusters(f32, h->num_sms);
    const int v = n > 0 ? n : h->num_sms / 2;
    slot.store(v, std::memory_order_relaxed);
    return v;
}

struct MxPlan {
    int tile_m, tile_n;
    bool pair;
    int a_rows; // rows of A's box: 128, or 64 / 32 on 1-CTA 192-wide tiles for M <= 64 / 32 (deeper rings)
    int64_t mt, nt;
    tpg::Schedule sched;
    int grid;
};

MxPlan mx_plan(tpgemm_handle *h, int64_t M, int64_t N, bool f32) {
    MxPlan pl;
    pl.pair = mx_pair(M, N);
    pl.tile_n = pl.pair ? kMxPairTileN : mx_tile_n(N);
    pl.a_rows = (!pl.pair && pl.tile_n == 192 && M <= 32) ? 32 : (!pl.pair && pl.tile_n == 192 && M <= 64) ? 64 : 128;
    pl.tile_m = tpg::mx::BM * (pl.pair ? 2 : 1);
    pl.mt = (M + pl.tile_m - 1) / pl.tile_m;
    pl.nt = (N + pl.tile_n - 1) / pl.tile_n;
    const int64_t cap = pl.pair ? mx_pairs_for(h, f32) : h->num_sms;
    pl.sched = tpg::make_schedule(pl.mt, pl.nt, pl.pair ? kGroupMPair : kGroupM, cap, 1, 0.5);
    pl.grid = static_cast<int>(pl.sched.workers * (pl.pair ? 2 : 1));
    return pl;
}

// The scales of one operand as a tensor of 512-byte chunks (128 x 32-bit
// words each), one chunk per box.
int encode_chunks(tpgemm_handle *h, CUtensorMap *map, const void *ptr, int64_t chunks) {
    cuuint64_t dims[2] = {128, static_cast<cuuint64_t>(chunks)};
    cuuint64_t strides[1] = {512};
    cuuint32_t box[2] = {128, 1};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = h->encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? TPGEMM_OK : TPGEMM_ERR_CUDA;
}

} // namespace

extern "C" {

int64_t gemm_mx_scale_bytes(int64_t rows, int64_t K) {
    if (rows < 0 || K < 0) return TPGEMM_ERR_INVALID_ARG;
    return mx_scale_bytes(rows, K);
}

int gemm_mx_check_args(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, int a_format, const void *SA,
                       const void *B, int64_t ldb, int b_format, const void *SB, const void *C, int64_t ldc,
                       const void *D, int64_t ldd, float beta, int out_dtype) {
    if (out_dtype != TPGEMM_OUT_BF16 && out_dtype != TPGEMM_OUT_F32) return TPGEMM_ERR_INVALID_ARG;
    if ((a_format != TPGEMM_FP8_E4M3 && a_format != TPGEMM_FP8_E5M2) ||
        (b_format != TPGEMM_FP8_E4M3 && b_format != TPGEMM_FP8_E5M2))
        return TPGEMM_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K < 0 || K % kMxBlock != 0) return TPGEMM_ERR_INVALID_ARG;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return TPGEMM_ERR_TOO_LARGE;
    if (M == 0 || N == 0) return TPGEMM_OK;
    // the kernel addresses scale chunks with 32-bit indices
    if (mx_scale_bytes(M, K) / 512 > kMaxDim || mx_scale_bytes(N, K) / 512 > kMaxDim) return TPGEMM_ERR_TOO_LARGE;
    const int64_t elt = out_dtype == TPGEMM_OUT_F32 ? 4 : 2;
    const bool use_c = beta != 0.0f;
    if (!D || ldd < N) return TPGEMM_ERR_INVALID_ARG;
    if (K > 0 && (!A || !B || !SA || !SB || lda < K || ldb < K)) return TPGEMM_ERR_INVALID_ARG;
    if (use_c && (!C || ldc < N)) return TPGEMM_ERR_INVALID_ARG;
    if (ldd > kMaxDim * 8 || (K > 0 && (lda > kMaxDim * 16 || ldb > kMaxDim * 16)) || (use_c && ldc > kMaxDim * 8))
        return TPGEMM_ERR_TOO_LARGE;
    if (!aligned16(D) || (M > 1 && (ldd * elt) % 16 != 0)) return TPGEMM_ERR_ALIGNMENT;
    if (K > 0) {
        if (!aligned16(A) || !aligned16(B) || !aligned16(SA) || !aligned16(SB)) return TPGEMM_ERR_ALIGNMENT;
        if ((M > 1 && lda % 16 != 0) || (N > 1 && ldb % 16 != 0)) return TPGEMM_ERR_ALIGNMENT;
    }
    if (use_c && (!aligned16(C) || (M > 1 && (ldc * elt) % 16 != 0))) return TPGEMM_ERR_ALIGNMENT;
    const Range rd = byte_range(D, M, N, ldd, elt);
    if (K > 0) {
        const Range rsa{reinterpret_cast<uintptr_t>(SA), reinterpret_cast<uintptr_t>(SA) +
                                                             static_cast<uintptr_t>(mx_scale_bytes(M, K))};
        const Range rsb{reinterpret_cast<uintptr_t>(SB), reinterpret_cast<uintptr_t>(SB) +
                                                             static_cast<uintptr_t>(mx_scale_bytes(N, K))};
        if (overlaps(rd, byte_range(A, M, K, lda, 1)) || overlaps(rd, byte_range(B, N, K, ldb, 1)) ||
            overlaps(rd, rsa) || overlaps(rd, rsb))
            return TPGEMM_ERR_OVERLAP;
    }
    if (use_c && !(C == D && ldc == ldd) && overlaps(rd, byte_range(C, M, N, ldc, elt))) return TPGEMM_ERR_OVERLAP;
    return TPGEMM_OK;
}

int gemm_run_mx(tpgemm_handle *h, int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, int a_format,
                const void *SA, const void *B, int64_t ldb, int b_format, const void *SB, const void *C,
                int64_t ldc, void *D, int64_t ldd, float alpha, float beta, int out_dtype, void *stream_ptr) {
    if (!h) return TPGEMM_ERR_INVALID_ARG;
    const int chk = gemm_mx_check_args(M, N, K, A, lda, a_format, SA, B, ldb, b_format, SB, C, ldc, D, ldd, beta,
                                       out_dtype);
    if (chk != TPGEMM_OK || M == 0 || N == 0) return chk;
    const bool f32 = out_dtype == TPGEMM_OUT_F32;
    const int64_t elt = f32 ? 4 : 2;
    const bool use_c = beta != 0.0f;
    DeviceGuard guard(h->device);
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    if (K == 0) {
        int64_t blocks = (M * N + 1023) / 1024;
        if (blocks > 8LL * h->num_sms) blocks = 8LL * h->num_sms;
        const int32_t m = static_cast<int32_t>(M), n = static_cast<int32_t>(N);
        const tpg::EpiParams none{};
        const void *c = use_c ? C : nullptr;
        return f32 ? launch(tpg::epilogue_only_kernel<true, false>, static_cast<int>(blocks), 256, 0, 1, stream, m, n,
                            beta, c, ldc, D, ldd, none)
                   : launch(tpg::epilogue_only_kernel<false, false>, static_cast<int>(blocks), 256, 0, 1, stream, m,
                            n, beta, c, ldc, D, ldd, none);
    }
    const MxPlan pl = mx_plan(h, M, N, f32);
    const int tile_n = pl.tile_n;
    const uint32_t chunk = f32 ? 32u : 64u;
    const int64_t cell = 16 / elt;
    const int64_t n_tma = N / cell * cell;
    const uint64_t map_n = static_cast<uint64_t>(n_tma > 0 ? n_tma : N);
    const CUtensorMapDataType out_dt = f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUtensorMap tmA, tmB, tmSA, tmSB, tmC, tmD;
    if (encode_2d(h, &tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, K, M, tma_stride(M, K, lda, 1), 128,
                  static_cast<uint32_t>(pl.a_rows)) ||
        encode_2d(h, &tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, K, N, tma_stride(N, K, ldb, 1), 128,
                  static_cast<uint32_t>(pl.pair ? tile_n / 2 : tile_n)) ||
        encode_chunks(h, &tmSA, SA, mx_scale_bytes(M, K) / 512) ||
        encode_chunks(h, &tmSB, SB, mx_scale_bytes(N, K) / 512) ||
        encode_2d(h, &tmD, out_dt, D, map_n, M, tma_stride(M, N, ldd, elt), chunk, 128) ||
        encode_2d(h, &tmC, out_dt, use_c ? C : D, map_n, M,
                  use_c ? tma_stride(M, N, ldc, elt) : tma_stride(M, N, ldd, elt), chunk, 128))
        return TPGEMM_ERR_CUDA;
    tpg::MxParams p{};
    p.M = static_cast<int32_t>(M);
    p.N = static_cast<int32_t>(N);
    p.K = static_cast<int32_t>(K);
    p.kb = static_cast<int32_t>((K + tpg::mx::BK - 1) / tpg::mx::BK);
    p.sched = pl.sched;
    p.n_tma = static_cast<int32_t>(n_tma);
    p.sfb_rows = static_cast<int32_t>((N + 127) / 128);
    p.sf_kc = static_cast<int32_t>((K + 127) / 128);
    p.idesc = tpg::make_idesc_mxf8(static_cast<uint32_t>(pl.tile_m), static_cast<uint32_t>(tile_n),
                                   static_cast<uint32_t>(a_format), static_cast<uint32_t>(b_format));
    p.alpha = alpha;
    p.beta = beta;
    p.C = use_c ? C : nullptr;
    p.ldc = ldc;
    p.D = D;
    p.ldd = ldd;
    p.status = h->status;
    p.timeout_ns = h->timeout_ns;
    const tpg::MxLaunch l{pl.grid, tile_n, pl.pair, pl.a_rows, f32, stream, &tmA, &tmB, &tmSA, &tmSB, &tmC, &tmD, &p};
    return tpg::mx_launch(l) == cudaSuccess ? TPGEMM_OK : TPGEMM_ERR_CUDA;
}

int gemm_mx_query_plan(tpgemm_handle *h, int64_t M, int64_t N, int64_t K, int out_dtype, int *tile_m, int *tile_n,
                       int64_t *num_tiles, int *grid, int *cluster, int *smem_bytes) {
    if (!h || M < 0 || N < 0 || K < 0) return TPGEMM_ERR_INVALID_ARG;
    if (out_dtype != TPGEMM_OUT_BF16 && out_dtype != TPGEMM_OUT_F32) return TPGEMM_ERR_INVALID_ARG;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return TPGEMM_ERR_TOO_LARGE;
    DeviceGuard guard(h->device);
    const MxPlan pl = mx_plan(h, M, N, out_dtype == TPGEMM_OUT_F32);
    if (tile_m) *tile_m = pl.tile_m;
    if (tile_n) *tile_n = pl.tile_n;
    if (num_tiles) *num_tiles = pl.mt * pl.nt;
    if (grid) *grid = pl.grid;
    if (cluster) *cluster = pl.pair ? 2 : 1;
    if (smem_bytes) *smem_bytes = tpg::mx_smem_bytes(pl.tile_n, pl.pair, pl.a_rows);
    return TPGEMM_OK;
}

} // extern "C"

// ---------------------------------------------------------------------------
// Block-scaled FP4 GEMM (gemm_run_fp4): the MX kernel with packed E2M1
// operands, NVFP4 or MXFP4 scales.
namespace {

int64_t fp4_block(int format) { return format == TPGEMM_NVFP4 ? 16 : 32; }

// Scale chunks (128 rows x 4 scale columns) per row block: one per 64
// elements of K (NVFP4) or per 128 (MXFP4).
int64_t fp4_chunks_per_row_block(int format, int64_t K) {
    const int64_t span = 4 * fp4_block(format);
    return (K + span - 1) / span;
}

int64_t fp4_scale_bytes(int format, int64_t rows, int64_t K) {
    return ((rows + 127) / 128) * fp4_chunks_per_row_block(format, K) * 512;
}

int fp4_pairs_for(tpgemm_handle *h, int format, bool f32) {
    std::atomic<int> &slot = h->fp4_pairs[format == TPGEMM_NVFP4 ? 0 : 1][f32 ? 1 : 0];
    const int cached = slot.load(std::memory_order_relaxed);
    if (cached > 0) return cached;
    const int n = format == TPGEMM_NVFP4 ? tpg::fp4_pair_clusters_nv(f32, h->num_sms)
                                         : tpg::fp4_pair_clusters_mx(f32, h->num_sms);
    const int v = n > 0 ? n : h->num_sms / 2;
    slot.store(v, std::memory_order_relaxed);
    return v;
}

// As mx_plan. FP4 moves half the bytes of FP8 per MMA, so up to 256 rows the
// GEMM is bound by reading B, and the tiles are chosen to cover the SMs in
// whole waves: 256 x 192 on pairs (256 x 256 above 256 rows, where the MMAs'
// width pays), 128 x 192 on single CTAs (128 x 128 when N <= 128).
MxPlan fp4_plan(tpgemm_handle *h, int format, int64_t M, int64_t N, bool f32) {
    MxPlan pl;
    pl.pair = mx_pair(M, N);
    pl.tile_n = pl.pair ? (M <= 256 ? 192 : kMxPairTileN) : (N > 128 ? 192 : 128);
    pl.a_rows = (!pl.pair && pl.tile_n == 192) ? (M <= 32 ? 32 : (M <= 64 ? 64 : 128)) : 128;
    pl.tile_m = tpg::mx::BM * (pl.pair ? 2 : 1);
    pl.mt = (M + pl.tile_m - 1) / pl.tile_m;
    pl.nt = (N + pl.tile_n - 1) / pl.tile_n;
    const int64_t cap = pl.pair ? fp4_pairs_for(h, format, f32) : h->num_sms;
    pl.sched = tpg::make_schedule(pl.mt, pl.nt, pl.pair ? kGroupMPair : kGroupM, cap, 1, 0.5);
    pl.grid = static_cast<int>(pl.sched.workers * (pl.pair ? 2 : 1));
    return pl;
}

// One operand's FP4 scales as [row block][chunk][128 words]; a box is `chunks`
// chunks of `row_blocks` row blocks, and chunks past either end read as zeros.
int encode_fp4_scales(tpgemm_handle *h, CUtensorMap *map, const void *ptr, int64_t rows, int64_t kc,
                      uint32_t chunks, uint32_t row_blocks) {
    cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(kc), static_cast<cuuint64_t>((rows + 127) / 128)};
    cuuint64_t strides[2] = {512, static_cast<cuuint64_t>(kc * 512)};
    cuuint32_t box[3] = {128, chunks, row_blocks};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = h->encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void *>(ptr), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? TPGEMM_OK : TPGEMM_ERR_CUDA;
}

} // namespace

extern "C" {

int64_t gemm_fp4_scale_bytes(int format, int64_t rows, int64_t K) {
    if ((format != TPGEMM_NVFP4 && format != TPGEMM_MXFP4) || rows < 0 || K < 0) return TPGEMM_ERR_INVALID_ARG;
    return fp4_scale_bytes(format, rows, K);
}

int gemm_fp4_check_args(int64_t M, int64_t N, int64_t K, int format, const void *A, int64_t lda, const void *SA,
                        const void *B, int64_t ldb, const void *SB, const void *C, int64_t ldc, const void *D,
                        int64_t ldd, float beta, int out_dtype) {
    if (out_dtype != TPGEMM_OUT_BF16 && out_dtype != TPGEMM_OUT_F32) return TPGEMM_ERR_INVALID_ARG;
    if (format != TPGEMM_NVFP4 && format != TPGEMM_MXFP4) return TPGEMM_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K < 0 || K % fp4_block(format) != 0) return TPGEMM_ERR_INVALID_ARG;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return TPGEMM_ERR_TOO_LARGE;
    if (M == 0 || N == 0) return TPGEMM_OK;
    // the kernel addresses scale chunks and row blocks with 32-bit coordinates
    if (fp4_scale_bytes(format, M, K) / 512 > kMaxDim || fp4_scale_bytes(format, N, K) / 512 > kMaxDim)
        return TPGEMM_ERR_TOO_LARGE;
    const int64_t elt = out_dtype == TPGEMM_OUT_F32 ? 4 : 2;
    const int64_t row_bytes = K / 2;
    const bool use_c = beta != 0.0f;
    if (!D || ldd < N) return TPGEMM_ERR_INVALID_ARG;
    if (K > 0 && (!A || !B || !SA || !SB || lda < row_bytes || ldb < row_bytes)) return TPGEMM_ERR_INVALID_ARG;
    if (use_c && (!C || ldc < N)) return TPGEMM_ERR_INVALID_ARG;
    if (ldd > kMaxDim * 8 || (K > 0 && (lda > kMaxDim * 16 || ldb > kMaxDim * 16)) || (use_c && ldc > kMaxDim * 8))
        return TPGEMM_ERR_TOO_LARGE;
    if (!aligned16(D) || (M > 1 && (ldd * elt) % 16 != 0)) return TPGEMM_ERR_ALIGNMENT;
    if (K > 0) {
        if (!aligned16(A) || !aligned16(B) || !aligned16(SA) || !aligned16(SB)) return TPGEMM_ERR_ALIGNMENT;
        if ((M > 1 && lda % 16 != 0) || (N > 1 && ldb % 16 != 0)) return TPGEMM_ERR_ALIGNMENT;
    }
    if (use_c && (!aligned16(C) || (M > 1 && (ldc * elt) % 16 != 0))) return TPGEMM_ERR_ALIGNMENT;
    const Range rd = byte_range(D, M, N, ldd, elt);
    if (K > 0) {
        const Range rsa{reinterpret_cast<uintptr_t>(SA), reinterpret_cast<uintptr_t>(SA) +
                                                             static_cast<uintptr_t>(fp4_scale_bytes(format, M, K))};
        const Range rsb{reinterpret_cast<uintptr_t>(SB), reinterpret_cast<uintptr_t>(SB) +
                                                             static_cast<uintptr_t>(fp4_scale_bytes(format, N, K))};
        if (overlaps(rd, byte_range(A, M, row_bytes, lda, 1)) || overlaps(rd, byte_range(B, N, row_bytes, ldb, 1)) ||
            overlaps(rd, rsa) || overlaps(rd, rsb))
            return TPGEMM_ERR_OVERLAP;
    }
    if (use_c && !(C == D && ldc == ldd) && overlaps(rd, byte_range(C, M, N, ldc, elt))) return TPGEMM_ERR_OVERLAP;
    return TPGEMM_OK;
}

int gemm_run_fp4(tpgemm_handle *h, int64_t M, int64_t N, int64_t K, int format, const void *A, int64_t lda,
                 const void *SA, const void *B, int64_t ldb, const void *SB, const void *C, int64_t ldc, void *D,
                 int64_t ldd, float alpha, float beta, int out_dtype, void *stream_ptr) {
    if (!h) return TPGEMM_ERR_INVALID_ARG;
    const int chk =
        gemm_fp4_check_args(M, N, K, format, A, lda, SA, B, ldb, SB, C, ldc, D, ldd, beta, out_dtype);
    if (chk != TPGEMM_OK || M == 0 || N == 0) return chk;
    const bool f32 = out_dtype == TPGEMM_OUT_F32;
    const int64_t elt = f32 ? 4 : 2;
    const bool use_c = beta != 0.0f;
    DeviceGuard guard(h->device);
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    if (K == 0) {
        int64_t blocks = (M * N + 1023) / 1024;
        if (blocks > 8LL * h->num_sms) blocks = 8LL * h->num_sms;
        const int32_t m = static_cast<int32_t>(M), n = static_cast<int32_t>(N);
        const tpg::EpiParams none{};
        const void *c = use_c ? C : nullptr;
        return f32 ? launch(tpg::epilogue_only_kernel<true, false>, static_cast<int>(blocks), 256, 0, 1, stream, m, n,
                            beta, c, ldc, D, ldd, none)
                   : launch(tpg::epilogue_only_kernel<false, false>, static_cast<int>(blocks), 256, 0, 1, stream, m,
                            n, beta, c, ldc, D, ldd, none);
    }
    const MxPlan pl = fp4_plan(h, format, M, N, f32);
    const int tile_n = pl.tile_n;
    const uint32_t chunk = f32 ? 32u : 64u;
    const int64_t cell = 16 / elt;
    const int64_t n_tma = N / cell * cell;
    const uint64_t map_n = static_cast<uint64_t>(n_tma > 0 ? n_tma : N);
    const int64_t row_bytes = K / 2;
    const int64_t kc = fp4_chunks_per_row_block(format, K);
    // chunks per 256-element stage: four of 64 elements (NVFP4), two of 128 (MXFP4)
    const uint32_t cps = format == TPGEMM_NVFP4 ? 4u : 2u;
    const CUtensorMapDataType out_dt = f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUtensorMap tmA, tmB, tmSA, tmSB, tmC, tmD;
    if (encode_2d(h, &tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, row_bytes, M, tma_stride(M, row_bytes, lda, 1), 128,
                  static_cast<uint32_t>(pl.a_rows)) ||
        encode_2d(h, &tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, row_bytes, N, tma_stride(N, row_bytes, ldb, 1), 128,
                  static_cast<uint32_t>(pl.pair ? tile_n / 2 : tile_n)) ||
        encode_fp4_scales(h, &tmSA, SA, M, kc, cps, 1) ||
        encode_fp4_scales(h, &tmSB, SB, N, kc, cps, tile_n == 128 ? 1u : 2u) ||
        encode_2d(h, &tmD, out_dt, D, map_n, M, tma_stride(M, N, ldd, elt), chunk, 128) ||
        encode_2d(h, &tmC, out_dt, use_c ? C : D, map_n, M,
                  use_c ? tma_stride(M, N, ldc, elt) : tma_stride(M, N, ldd, elt), chunk, 128))
        return TPGEMM_ERR_CUDA;
    tpg::MxParams p{};
    p.M = static_cast<int32_t>(M);
    p.N = static_cast<int32_t>(N);
    p.K = static_cast<int32_t>(K);
    // a stage is 128 bytes of a row: 256 elements
    p.kb = static_cast<int32_t>((K + 255) / 256);
    p.sched = pl.sched;
    p.n_tma = static_cast<int32_t>(n_tma);
    p.sfb_rows = static_cast<int32_t>((N + 127) / 128);
    p.sf_kc = static_cast<int32_t>(kc);
    p.idesc = tpg::make_idesc_fp4(static_cast<uint32_t>(pl.tile_m), static_cast<uint32_t>(tile_n),
                                  format == TPGEMM_MXFP4);
    p.alpha = alpha;
    p.beta = beta;
    p.C = use_c ? C : nullptr;
    p.ldc = ldc;
    p.D = D;
    p.ldd = ldd;
    p.status = h->status;
    p.timeout_ns = h->timeout_ns;
    const tpg::MxLaunch l{pl.grid, tile_n, pl.pair, pl.a_rows, f32, stream, &tmA, &tmB, &tmSA, &tmSB, &tmC, &tmD, &p};
    const cudaError_t e = format == TPGEMM_NVFP4 ? tpg::fp4_launch_nv(l) : tpg::fp4_launch_mx(l);
    return e == cudaSuccess ? TPGEMM_OK : TPGEMM_ERR_CUDA;
}

int gemm_fp4_query_plan(tpgemm_handle *h, int format, int64_t M, int64_t N, int64_t K, int out_dtype, int *tile_m,
                        int *tile_n, int64_t *num_tiles, int *grid, int *cluster, int *smem_bytes) {
    if (!h || M < 0 || N < 0 || K < 0) return TPGEMM_ERR_INVALID_ARG;
    if (format != TPGEMM_NVFP4 && format != TPGEMM_MXFP4) return TPGEMM_ERR_INVALID_ARG;
    if (out_dtype != TPGEMM_OUT_BF16 && out_dtype != TPGEMM_OUT_F32) return TPGEMM_ERR_INVALID_ARG;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return TPGEMM_ERR_TOO_LARGE;
    DeviceGuard guard(h->device);
    const MxPlan pl = fp4_plan(h, format, M, N, out_dtype == TPGEMM_OUT_F32);
    if (tile_m) *tile_m = pl.tile_m;
    if (tile_n) *tile_n = pl.tile_n;
    if (num_tiles) *num_tiles = pl.mt * pl.nt;
    if (grid) *grid = pl.grid;
    if (cluster) *cluster = pl.pair ? 2 : 1;
    if (smem_bytes)
        *smem_bytes = format == TPGEMM_NVFP4 ? tpg::fp4_smem_bytes_nv(pl.tile_n, pl.pair, pl.a_rows)
                                             : tpg::fp4_smem_bytes_mx(pl.tile_n, pl.pair, pl.a_rows);
    return TPGEMM_OK;
}

} // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free entry point (gemm_run_noalloc).
//
// Some callers cannot call cudaMalloc: code that runs while a memory pool or
// arena owned by an outer framework is the only legal source of device memory,
// serving loops that forbid allocation after warm-up (an allocation there can
// stall on the driver, fragment the pool or break a stream capture in
// progress), and callers that have no place to keep a handle. gemm_create
// allocates the handle's status word with cudaMalloc, so those callers use this
// entry point instead: it runs the tiled GEMM kernel with its scratch (the
// 4-byte status word the kernel's bounded waits report into) taken from the
// file-scope array below, which every GPU that loads this library holds until
// the process exits.
namespace {

constexpr int kNoallocStatusWords = 4;   // maximum scratch: 16 bytes
constexpr int kNoallocMaxDevices = 64;
static __device__ __align__(256) uint32_t g_noalloc_scratch[kNoallocStatusWords];

struct NoallocDevice {
    bool ready = false;
    uint32_t *status = nullptr; // device address of g_noalloc_scratch on this device
    int num_sms = 0;
    int ks_clusters[2][2] = {}; // as tpgemm_handle::ks_clusters
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
};
NoallocDevice g_noalloc_dev[kNoallocMaxDevices];
std::mutex g_noalloc_mutex;

// One-time set-up for the current device (which must be the device the
// pointers live on). In host code the array's name is only a host-side stand-in,
// so its device address is looked up here, with this device current, and passed
// to the kernel as a pointer.
int noalloc_setup(int dev, NoallocDevice **out) {
    if (dev < 0 || dev >= kNoallocMaxDevices) return TPGEMM_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    NoallocDevice &d = g_noalloc_dev[dev];
    if (!d.ready) {
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return TPGEMM_ERR_CUDA;
        if (prop.major != 10 || prop.minor != 3) return TPGEMM_ERR_UNSUPPORTED_DEVICE;
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
            (void)cudaGetLastError();
            return TPGEMM_ERR_CUDA;
        }
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return TPGEMM_ERR_CUDA;
        if (!tpg::tiled_set_limits_e0() ||
            cudaMemset(ptr, 0, sizeof(uint32_t) * kNoallocStatusWords) != cudaSuccess) {
            (void)cudaGetLastError();
            return TPGEMM_ERR_CUDA;
        }
        d.status = static_cast<uint32_t *>(ptr);
        d.num_sms = prop.multiProcessorCount;
        for (int f = 0; f < 2; ++f)
            for (int i = 0; i < 2; ++i) {
                const int split = i ? 4 : 2;
                const int n = tpg::tiled_clusters(false, f != 0, d.num_sms, split);
                d.ks_clusters[f][i] = n > 0 ? n : d.num_sms / split;
            }
        d.encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        d.ready = true;
    }
    *out = &d;
    return TPGEMM_OK;
}

} // namespace

extern "C" int gemm_run_noalloc(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B,
                                int64_t ldb, const void *C, int64_t ldc, void *D, int64_t ldd, float alpha,
                                float beta, int out_dtype, void *stream_ptr, int check_status) {
    const int chk = gemm_check_args(M, N, K, A, lda, B, ldb, C, ldc, D, ldd, beta, out_dtype);
    if (chk != TPGEMM_OK || M == 0 || N == 0) return chk;
    // The scratch this kernel needs is one status word whatever M, N and K are,
    // so the 16-byte array serves every size gemm_check_args accepts.
    int dev = -1;
    // cudaSetDevice on the current device binds its primary context to this
    // thread, which the tensor-map encoder below needs (see DeviceGuard).
    if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess) return TPGEMM_ERR_CUDA;
    NoallocDevice *nd = nullptr;
    const int st = noalloc_setup(dev, &nd);
    if (st != TPGEMM_OK) return st;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    const bool f32 = out_dtype == TPGEMM_OUT_F32;
    const int64_t elt = f32 ? 4 : 2;
    const bool use_c = beta != 0.0f;
    int rc;
    if (K == 0) {
        // D = beta*C: no pipeline, no scratch
        int64_t blocks = (M * N + 1023) / 1024;
        if (blocks > 8LL * nd->num_sms) blocks = 8LL * nd->num_sms;
        const int32_t m = static_cast<int32_t>(M), n = static_cast<int32_t>(N);
        const void *c = use_c ? C : nullptr;
        const tpg::EpiParams none{};
        rc = f32 ? launch(tpg::epilogue_only_kernel<true, false>, static_cast<int>(blocks), 256, 0, 1, stream, m, n,
                          beta, c, ldc, D, ldd, none)
                 : launch(tpg::epilogue_only_kernel<false, false>, static_cast<int>(blocks), 256, 0, 1, stream, m, n,
                          beta, c, ldc, D, ldd, none);
    } else {
        // The status word must start at zero: every call shares it.
        if (cudaMemsetAsync(nd->status, 0, sizeof(uint32_t), stream) != cudaSuccess) return TPGEMM_ERR_CUDA;
        CUtensorMap tmA, tmB, tmB1, tmC, tmD;
        tpg::TiledParams p;
        const TiledCall call{M, N, K, 1, 1, A, lda, 0, B, ldb, 0, C, ldc, 0, D, ldd, 0, alpha, beta, f32};
        if (build_tiled(nd->encode, call, &tmA, &tmB, &tmB1, &tmC, &tmD, &p) != TPGEMM_OK) return TPGEMM_ERR_CUDA;
        const int64_t mt = (M + tpg::tiled::BM - 1) / tpg::tiled::BM;
        const int64_t nt = (N + tpg::tiled::BN - 1) / tpg::tiled::BN;
        // the same K split as gemm_run would choose, so the two give the same bits
        const int ks = tiled_ksplit_choice(mt * nt, p.kb, nd->ks_clusters[f32 ? 1 : 0][0], nd->ks_clusters[f32 ? 1 : 0][1]);
        p.sched = ks > 1 ? tiled_schedule(mt, nt, mt * nt, false, false) : tiled_schedule(mt, nt, nd->num_sms, false, true);
        p.ksplit = ks;
        const int grid = static_cast<int>(p.sched.workers * ks);
        p.mt_batch = static_cast<int32_t>(mt);
        p.status = nd->status;
        p.timeout_ns = 2000000000ull;
        const tpg::TiledLaunch l{grid, static_cast<int>(tpg::tiled::SMEM_BYTES), ks, false, f32, stream,
                                 &tmA, &tmB, &tmB1, &tmC, &tmD, &p, nullptr};
        rc = tpg::tiled_launch_e0(l) == cudaSuccess ? TPGEMM_OK : TPGEMM_ERR_CUDA;
    }
    if (rc != TPGEMM_OK || !check_status) return rc;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return TPGEMM_ERR_CUDA;
    uint32_t word = 0;
    if (cudaMemcpy(&word, nd->status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return TPGEMM_ERR_CUDA;
    if (word != 0) {
        if (cudaMemset(nd->status, 0, sizeof(uint32_t)) != cudaSuccess) return TPGEMM_ERR_CUDA;
        return TPGEMM_ERR_TIMEOUT;
    }
    return TPGEMM_OK;
}
