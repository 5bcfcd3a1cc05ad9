// Persistent, warp-specialised bf16 GEMM for sm_103a:  D = alpha*A*B + beta*C.
//
// Two modes of one kernel template:
//   kPair = false  one CTA per SM owns 128 x 256 output tiles; MMAs are
//                  tcgen05.mma.cta_group::1 with M = 128.
//   kPair = true   the two CTAs of a cluster pair own a 256 x 256 tile; the even
//                  CTA issues tcgen05.mma.cta_group::2 with M = 256 for both. Each
//                  CTA stages its own 128 rows of A and its own half of B's
//                  columns, so per SM the ring holds 32 KB per K block instead
//                  of 48 KB and six stages fit where four did.
// Inside a CTA three roles run concurrently, connected by mbarriers:
//   warp 0      TMA producer: per 64-wide K block, one A box (128 rows x 64 K,
//               K-major) and the B boxes (64 K rows x 64 N each, N-major, two
//               per instruction when N is a multiple of 64; an odd last one,
//               of a 64-column piece, alone), all 128-byte swizzled, into the
//               shared-memory ring. The TMA unit's cost grows with the number
//               of instructions, not only with bytes, so fewer, larger boxes
//               keep the ring fuller.
//   warp 1      allocates all 512 TMEM columns (two 128 x 256 fp32
//               accumulators); one lane (of the even CTA, in pair mode) issues
//               the MMAs, K = 16 each, four per K block, and frees each ring
//               stage with tcgen05.commit when the MMAs reading it are done.
//   warps 2-5   epilogue: wait for a finished accumulator, read it from TMEM
//               (each warp its 32-lane quarter = 32 rows), apply alpha and
//               beta*C in fp32, round to the output type, write 128-byte
//               swizzled rows to a staging buffer and TMA-store them. The
//               accumulator is released as soon as it has been read, so the
//               next tile's MMAs overlap this tile's stores.
// The design levers are the ones "TorchInductor ganha suporte a GEMMs de alta
// performance com CuteDSL" lists for near-peak GEMMs (tile sizes matched to
// the tensor-core pipeline, explicit shared-memory stages, warp
// specialisation, TMA); the epilogue's auxiliary-tensor add is the page's
// epilogue-fusion roadmap. Each output tile (or tile piece) is owned by one
// CTA or CTA pair ("cuTile Rust explained", "Ownership crosses the launch
// boundary"); inside, the mbarrier full/empty protocol orders every load
// before the MMA that reads it and every MMA before the epilogue that reads
// its result ("Disjointness outside. Ordering inside.").
#pragma once

#include <cuda_bf16.h>

#include <type_traits>

#include "epilogue.cuh"
#include "ptx.cuh"
#include "schedule.cuh"

namespace tpg {

struct TiledParams {
    int32_t M, N, K; // M: rows per batch (uniform batches); grouped: unused
    int32_t kb;      // 64-wide K blocks
    Schedule sched;  // over all tile rows of all batches or groups
    int32_t mt_batch; // tile rows per batch (uniform batches)
    int32_t a_bcast, b_bcast, c_bcast; // 1: the operand has a single batch slice shared by all
    int64_t sC, sD;  // batch strides of C and D in elements (plain-store paths)
    // Columns [0, n_tma) of C and D go through the tensor maps; n_tma is N
    // rounded down to a multiple of 16 bytes, because a TMA store writes whole
    // 16-byte cells of the innermost dimension even past its bound. The last
    // n_tma..N-1 columns (fewer than one cell) use plain loads and stores.
    int32_t n_tma;
    // 1: B's tensor map is 4-D, [slice][N/64 groups][K][64 columns] (N a multiple
    // of 64), and each load brings two 64-column groups of one K block (one
    // TMA instruction where the 3-D map needs two); 0: B is loaded one 64 x 64
    // box at a time. The second map of B is always the 3-D one, [slice][K][N]:
    // it carries every box when this is 0 and the odd last 64-column group of a
    // narrow piece when it is 1.
    int32_t b_grouped;
    // 1-CTA mode only: the CTAs of a cluster of `ksplit` (2 or 4) share one
    // tile, each accumulating its own part of the K range; 1 otherwise. See the
    // kernel's K-split epilogue.
    int32_t ksplit;
    // Pair mode only, 1 or 0: the K split of the last partial round. Its tiles
    // are cut into two pieces as column halves, and each piece accumulates
    // half of the K range over the whole tile width instead of all of K over
    // half the width. The two pairs of a tile then trade, through `ws`, the
    // fp32 partial sums of each other's columns (see the epilogue).
    int32_t ktail;
    uint32_t epoch; // nonzero tag of this call in the workspace flags
    void *ws;       // workspace (caller-owned; flags, then 64 KB partial-sum slots)
    float alpha, beta;
    const void *C;
    int64_t ldc;
    void *D;
    int64_t ldd;
    uint32_t *status;
    uint64_t timeout_ns;
    EpiParams epi; // read only by the fused-epilogue instantiations
};

// Grouped GEMM (one B slice per group, the groups' rows stacked in A, C and
// D, as for mixture-of-experts layers): the group table travels as a kernel
// argument of the grouped instantiations only.
constexpr int kMaxGroups = 256;
struct GroupTable {
    int32_t groups;
    int32_t tile_prefix[kMaxGroups + 1]; // tile rows of the groups before g
    int32_t row_start[kMaxGroups];       // first row of group g in A, C and D
    int32_t rows[kMaxGroups];            // rows of group g
};
struct NoGroups {
    int32_t unused;
};
template <bool kGrouped>
using SegArg = typename std::conditional<kGrouped, GroupTable, NoGroups>::type;

// Where the tile row `tile_row` (of rows_per_tile rows) lives: the batch slice
// of A/C/D and of B, its first row and how many rows of the segment remain
// from there (more than the tile when the segment continues).
struct Segment {
    int32_t ab, bb, row0, rows_left;
};

template <bool kGrouped>
__device__ __forceinline__ Segment segment_of(int32_t tile_row, int32_t rows_per_tile, const TiledParams &p,
                                              const SegArg<kGrouped> &seg) {
    Segment s;
    if constexpr (kGrouped) {
        // the last group whose first tile row is <= tile_row (empty groups are skipped
        // because a later group with the same prefix wins)
        int32_t lo = 0, hi = seg.groups - 1;
        while (lo < hi) {
            const int32_t mid = (lo + hi + 1) >> 1;
            if (seg.tile_prefix[mid] <= tile_row)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int32_t local = tile_row - seg.tile_prefix[lo];
        s.ab = 0;
        s.bb = lo;
        s.row0 = seg.row_start[lo] + local * rows_per_tile;
        s.rows_left = seg.rows[lo] - local * rows_per_tile;
    } else {
        const int32_t b = tile_row / p.mt_batch;
        const int32_t local = tile_row - b * p.mt_batch;
        s.ab = b;
        s.bb = b;
        s.row0 = local * rows_per_tile;
        s.rows_left = p.M - local * rows_per_tile;
    }
    return s;
}

namespace tiled {

constexpr int kEpiUnitAlpha = 5; // see gemm_tiled_kernel's kEpi

constexpr int BM = 128;  // rows per CTA
constexpr int BN = 256;  // columns per tile
constexpr int BK = 64;
constexpr int THREADS = 192;
constexpr int EPI_THREADS = 128;
constexpr uint32_t A_STAGE_BYTES = BM * BK * 2; // 16 KB
constexpr uint32_t B_BOX_BYTES = BK * 64 * 2;   // 8 KB: 64 K rows x 64 N
constexpr uint32_t EPI_BUF_BYTES = BM * 128;    // 128 rows x 128 bytes
constexpr uint32_t TMEM_COLS = 512;

template <bool kPair>
struct Layout {
    static constexpr int STAGES = kPair ? 6 : 4;
    static constexpr int B_BOXES = kPair ? 2 : 4; // per CTA, full-width tile
    static constexpr uint32_t B_STAGE_BYTES = B_BOXES * B_BOX_BYTES;
    // Offsets from a 1024-byte aligned base (the 128-byte swizzle pattern
    // repeats every 1024 bytes and is computed from address bits).
    static constexpr uint32_t OFF_A = 0;
    static constexpr uint32_t OFF_B = OFF_A + STAGES * A_STAGE_BYTES;
    static constexpr uint32_t OFF_EPI = OFF_B + STAGES * B_STAGE_BYTES;
    static constexpr uint32_t OFF_BAR = OFF_EPI + 2 * EPI_BUF_BYTES;
    // full, empty, tfull, tempty, c, drain, K-split: peers' rings free, partials received
    static constexpr uint32_t NUM_BARS = 2 * STAGES + 2 + 2 + 2 + 1 + 2;
    static constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024; // + slack to align the base
};
static_assert(Layout<false>::SMEM_BYTES <= 232448, "exceeds the 227 KB shared-memory limit per CTA");
static_assert(Layout<true>::SMEM_BYTES <= 232448, "exceeds the 227 KB shared-memory limit per CTA");
constexpr uint32_t SMEM_BYTES = Layout<false>::SMEM_BYTES; // the 1-CTA mode

// Waits, without looking at the abort flag, for an operation this CTA itself
// started; used only on the abort path so nothing is in flight at exit.
__device__ __forceinline__ bool drain_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
    const uint32_t a = smem_addr(bar);
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 0; i < (1u << 28); ++i) {
        if (mbar_try_wait(a, parity)) return true;
        if ((i & 63u) == 63u && globaltimer_ns() - t0 > limit_ns) return false;
    }
    return false;
}

// The K blocks [lo, hi) a work item accumulates, and the columns its MMAs
// cover: all of K over the item's own columns, except for a piece of the K
// split tail, which covers its tile's full width over half of K.
struct KRange {
    int32_t lo, hi, n, width;
};
__device__ __forceinline__ KRange item_krange(const WorkItem &w, int32_t kb_lo, int32_t kb_hi, const TiledParams &p) {
    KRange r{kb_lo, kb_hi, w.n, w.width};
    if (p.ktail && w.width < BN) {
        const int32_t piece = (w.n % BN) / w.width; // 0 or 1
        r.lo = piece * p.kb / 2;
        r.hi = (piece + 1) * p.kb / 2;
        r.n = w.n - w.n % BN;
        r.width = BN;
    }
    return r;
}

// Workspace of the K split tail: 4 KB of flags, then one slot of 128 rows x
// 128 fp32 columns (64 KB) per (tail tile, CTA of the pair, piece). A slot is
// laid out [column / 4][row][4], so that the 32 rows of a warp write and read
// 512 contiguous bytes per column quad.
constexpr uint32_t kTailFlagBytes = 4096;
constexpr uint32_t kTailSlotBytes = 128u * 128u * 4u;
__device__ __forceinline__ uint32_t *tail_flag(const TiledParams &p, int64_t tile, uint32_t cta, uint32_t piece) {
    return static_cast<uint32_t *>(p.ws) + (tile * 2 + cta) * 2 + piece;
}
__device__ __forceinline__ float4 *tail_slot(const TiledParams &p, int64_t tile, uint32_t cta, uint32_t piece) {
    return reinterpret_cast<float4 *>(static_cast<uint8_t *>(p.ws) + kTailFlagBytes +
                                      static_cast<uint64_t>((tile * 2 + cta) * 2 + piece) * kTailSlotBytes);
}

// Busy-waits `ns` nanoseconds (abort path only).
__device__ __forceinline__ void settle(uint64_t ns) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 0; i < (1u << 26) && globaltimer_ns() - t0 < ns; ++i) {
    }
}

// kEpi: 0 plain alpha*acc + beta*C; 1 + activation for the fused epilogue
// (bias and aux are runtime options; the activation is compiled in, so each
// instantiation carries only its own math); kEpiUnitAlpha the plain epilogue
// for alpha == 1, without the multiply (the epilogue's work runs beside the
// next tile's MMAs and slows them, in proportion to how much of it there is).
// kKsplit: the 1-CTA mode's K split (p.ksplit CTAs of a cluster per tile);
// the other instantiations carry none of its code.
template <bool kOutF32, bool kPair, int kEpi, bool kGrouped = false, bool kKsplit = false>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_tiled_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmD,
                      const TiledParams p, const __grid_constant__ SegArg<kGrouped> seg) {
    using L = Layout<kPair>;
    constexpr int STAGES = L::STAGES;
    constexpr bool kFused = kEpi > 0 && kEpi != kEpiUnitAlpha; // bias / activation / aux
    constexpr int CHUNK = kOutF32 ? 32 : 64; // output columns per 128-byte staging row
    constexpr int CL = kPair ? 2 : 1;        // CTAs per worker

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);
    uint64_t *full = bars;
    uint64_t *empty = bars + STAGES;
    uint64_t *tfull = bars + 2 * STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *cbar = tempty + 2;
    uint64_t *drain = cbar + 2;
    uint64_t *ks_free = drain + 1; // K split: one arrive from each peer whose MMAs are done
    uint64_t *ks_recv = drain + 2; // K split (and its tail form in pair mode): the peers' partials have landed here
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + L::OFF_MISC + 4);

    const uint32_t warp = threadIdx.x / 32;
    const uint32_t lane = threadIdx.x % 32;
    const uint32_t rank = kPair ? cluster_ctarank() : 0u; // 0 = the even CTA, which issues the MMAs
    // K split (1-CTA mode): a cluster of ks CTAs is one worker; CTA krank
    // accumulates K blocks [kb_lo, kb_hi) of the worker's tile.
    const int32_t ks = (kPair || !kKsplit) ? 1 : p.ksplit;
    const int32_t krank = ks > 1 ? static_cast<int32_t>(cluster_ctarank()) : 0;
    const int32_t kb_lo = krank * p.kb / ks;
    const int32_t kb_hi = (krank + 1) * p.kb / ks;
    const int64_t worker = static_cast<int64_t>(blockIdx.x) / (CL * ks);
    const int64_t workers = static_cast<int64_t>(gridDim.x) / (CL * ks);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            // every epilogue warp of the worker hands the accumulator back
            mbar_init(&tempty[b], CL * EPI_THREADS / 32);
            mbar_init(&cbar[b], 1);
        }
        mbar_init(drain, 1);
        if (ks > 1) {
            mbar_init(ks_free, static_cast<uint32_t>(ks - 1));
            mbar_init(ks_recv, 1);
        }
        if (kPair && p.ktail) mbar_init(ks_recv, 1); // the K split tail's partner partial sums
        *abort_flag = 0u;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        if (p.b_grouped) prefetch_tensormap(&tmB1);
        prefetch_tensormap(&tmD);
        if (p.beta != 0.0f) prefetch_tensormap(&tmC);
    }
    if (warp == 1) {
        if constexpr (kPair) {
            tmem_alloc_pair(tmem_slot, TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(tmem_slot, TMEM_COLS);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    if (kPair || ks > 1)
        cluster_sync(); // every CTA's barriers initialised (and TMEM allocated in both of a pair)
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // Everything above touched only on-chip state; from here on global memory.
    grid_dependency_wait();
    grid_launch_dependents();

    const WaitCtl ctl{abort_flag, p.status, p.timeout_ns};

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            // In pair mode both CTAs' loads complete on the even CTA's barrier.
            const uint32_t full0 = kPair ? map_to_rank(smem_addr(full), 0) : 0u;
            uint32_t stage = 0, phase = 0;
            int64_t issued = 0;
            bool ok = true;
            WorkItem w;
            for (int64_t t = worker; ok && work_item(p.sched, t, BN, w); t += workers) {
                const KRange kr = item_krange(w, kb_lo, kb_hi, p);
                const Segment sg = segment_of<kGrouped>(w.m, BM * CL, p, seg);
                const int32_t m0 = sg.row0 + static_cast<int32_t>(rank) * BM;
                const int32_t ab = p.a_bcast ? 0 : sg.ab;
                const int32_t bb = p.b_bcast ? 0 : sg.bb;
                const int32_t cols = kr.width / CL; // B columns this CTA stages
                const int32_t nb = kr.n + static_cast<int32_t>(rank) * cols;
                // The CTA stages `groups` 64-column groups of B per K block: two
                // per instruction through the 4-D view while at least two remain,
                // and an odd last one (a 64-column piece of a split tile) through
                // the 3-D view, so that a narrow piece loads only the columns it
                // uses.
                const int32_t groups = cols / 64;
                const int32_t npair = p.b_grouped ? groups / 2 : 0;
                const uint32_t bbytes = static_cast<uint32_t>(groups) * B_BOX_BYTES;
                const uint32_t tx = CL * (A_STAGE_BYTES + bbytes);
                for (int32_t kb = kr.lo; kb < kr.hi; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, ctl, kStatusTimeoutProducer)) {
                        ok = false;
                        break;
                    }
                    const int32_t k0 = kb * BK;
                    uint8_t *adst = smem + L::OFF_A + stage * A_STAGE_BYTES;
                    uint8_t *bdst = smem + L::OFF_B + stage * L::B_STAGE_BYTES;
                    if constexpr (kPair) {
                        if (rank == 0) mbar_arrive_expect_tx(&full[stage], tx);
                        const uint32_t fb = full0 + stage * 8u;
                        tma_load_3d_pair(&tmA, fb, adst, k0, m0, ab);
                        for (int c = 0; c < npair; ++c)
                            tma_load_4d_pair(&tmB, fb, bdst + 2 * c * B_BOX_BYTES, 0, k0, (nb >> 6) + 2 * c, bb);
                        for (int c = 2 * npair; c < groups; ++c)
                            tma_load_3d_pair(&tmB1, fb, bdst + c * B_BOX_BYTES, nb + c * 64, k0, bb);
                    } else {
                        mbar_arrive_expect_tx(&full[stage], tx);
                        tma_load_3d(&tmA, &full[stage], adst, k0, m0, ab);
                        for (int c = 0; c < npair; ++c)
                            tma_load_4d(&tmB, &full[stage], bdst + 2 * c * B_BOX_BYTES, 0, k0, (nb >> 6) + 2 * c, bb);
                        for (int c = 2 * npair; c < groups; ++c)
                            tma_load_3d(&tmB1, &full[stage], bdst + c * B_BOX_BYTES, nb + c * 64, k0, bb);
                    }
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                if (!kPair || rank == 0) {
                    // Let the loads already issued land before the CTA exits.
                    const int64_t pending = issued < STAGES ? issued : STAGES;
                    uint32_t s = stage, ph = phase;
                    for (int64_t i = 0; i < pending; ++i) {
                        if (s == 0) {
                            s = STAGES - 1;
                            ph ^= 1u;
                        } else {
                            --s;
                        }
                        if (!drain_wait(&full[s], ph, p.timeout_ns) && p.status)
                            atomicOr(p.status, kStatusTimeoutDrain);
                    }
                }
                // The odd CTA's loads complete on the even CTA's barriers, which it
                // cannot wait on: give them time to land.
                if (kPair) settle(200000);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (even CTA only in pair mode)
        if (lane == 0 && rank == 0) {
            // The issuing thread's instructions per K block bound the tensor pipe:
            // each tcgen05.mma costs it about 107 cycles to issue, four of them
            // about 430 of the 512 cycles a 256-wide K block computes for. So the
            // stage-0 descriptors and barrier addresses are built once, and a
            // stage only adds offsets.
            const uint64_t adesc0 = make_smem_desc_sw128(smem_addr(smem + L::OFF_A), 16, 1024);
            // 64-wide N blocks of B are one 8 KB box apart
            const uint64_t bdesc0 = make_smem_desc_sw128(smem_addr(smem + L::OFF_B), B_BOX_BYTES, 1024);
            const uint32_t full_a = smem_addr(full), empty_a = smem_addr(empty);
            uint32_t stage = 0, phase = 0;
            uint32_t acc = 0, acc_phase = 0;
            bool ok = true;
            bool any = false;
            WorkItem w;
            for (int64_t t = worker; ok && work_item(p.sched, t, BN, w); t += workers) {
                const KRange kr = item_krange(w, kb_lo, kb_hi, p);
                const uint32_t idesc = make_idesc_bf16_f32(BM * CL, static_cast<uint32_t>(kr.width), false, true);
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, ctl, kStatusTimeoutMma)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                // Issues the MMAs of K block kb from the current stage and frees the stage.
                auto issue = [&](int32_t kb) {
                    // The stage's descriptors: stage 0's plus the stage's byte offset >> 4
                    // in the start-address field.
                    const uint64_t ad = adesc0 + stage * (A_STAGE_BYTES >> 4);
                    const uint64_t bd = bdesc0 + stage * (L::B_STAGE_BYTES >> 4);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        // A: K-major, advance 16 bf16 = 32 bytes inside the swizzle atom.
                        // B: N-major, advance 16 K rows = 2048 bytes.
                        const uint32_t accumulate = (kb != kr.lo || kk != 0) ? 1u : 0u;
                        if constexpr (kPair)
                            tc_mma_f16_pair(d_tmem, ad + kk * (32 >> 4), bd + kk * (2048 >> 4), idesc, accumulate);
                        else
                            tc_mma_f16(d_tmem, ad + kk * (32 >> 4), bd + kk * (2048 >> 4), idesc, accumulate);
                    }
                    any = true;
                    if constexpr (kPair)
                        tc_commit_pair_mc_addr(empty_a + stage * 8u, 0x3);
                    else
                        tc_commit_addr(empty_a + stage * 8u);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                };
                for (int32_t kb = kr.lo; kb < kr.hi;) {
                    // Wait for this stage and, in the same breath, test the next two: when
                    // they have landed, one wait serves up to three K blocks (the issuing
                    // thread's instructions per K block are what pace the tensor pipe).
                    const uint32_t s1 = stage + 1 == STAGES ? 0u : stage + 1;
                    const uint32_t p1 = stage + 1 == STAGES ? phase ^ 1u : phase;
                    const uint32_t s2 = s1 + 1 == STAGES ? 0u : s1 + 1;
                    const uint32_t p2 = s1 + 1 == STAGES ? p1 ^ 1u : p1;
                    const uint32_t st = mbar_try_wait_and_test2(full_a + stage * 8u, phase, full_a + s1 * 8u, p1,
                                                                full_a + s2 * 8u, p2);
                    if (!(st & 1u) && !mbar_wait(&full[stage], phase, ctl, kStatusTimeoutMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue(kb++);
                    if ((st & 2u) && kb < kr.hi) {
                        issue(kb++);
                        if ((st & 4u) && kb < kr.hi) issue(kb++);
                    }
                }
                if (!ok) break;
                if constexpr (kPair)
                    tc_commit_pair_mc(&tfull[acc], 0x3);
                else
                    tc_commit(&tfull[acc]);
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            if (!ok && any) {
                // Wait for every MMA issued so far before TMEM is freed.
                if constexpr (kPair)
                    tc_commit_pair_mc(drain, 0x1);
                else
                    tc_commit(drain);
                if (!drain_wait(drain, 0, p.timeout_ns) && p.status) atomicOr(p.status, kStatusTimeoutDrain);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue (warps 2..5)
        const uint32_t q = warp & 3u;        // TMEM lane quarter this warp may read
        const uint32_t row = q * 32u + lane; // row of the CTA's 128 rows held by this thread
        const bool leader = threadIdx.x == 64;
        const bool has_beta = p.beta != 0.0f;
        const uint32_t tempty0 = kPair ? map_to_rank(smem_addr(tempty), 0) : 0u;
        uint8_t *epi = smem + L::OFF_EPI;
        uint32_t acc = 0, acc_phase = 0;
        uint32_t slot = 0;
        uint32_t cphase = 0; // bit b: parity of the next wait on cbar[b]
        bool ok = true;
        bool tail_loading = false; // the leader issued the bulk load of the partner's partial sums
        // K split: CTA krank of the cluster owns (and stores) columns
        // [krank * ks_w, (krank + 1) * ks_w) of the tile. Once its own MMAs are
        // done its ring is idle, and holds ks - 1 receive slots (the other
        // CTAs' partial sums of its columns, one slot per sender) followed by
        // ks - 1 send slots (its partial sums of each peer's columns). A slot
        // is laid out [column / 4][row][4], so a warp's 32 rows write 512
        // contiguous bytes; one bulk copy per peer moves a send slot into the
        // peer's receive slot.
        const int32_t ks_w = BN / ks;
        const uint32_t ks_slot_bytes = static_cast<uint32_t>(BM * ks_w * 4);
        // Columns oc0 .. oc0+31 of this CTA's own window: part 0 + part 1 + ...
        // + part ks-1, always in that order, this CTA's part taken from r. A
        // peer's eight cells are loaded together, so their loads overlap.
        auto ks_combine = [&](uint32_t(&r)[32], int32_t oc0) {
            const float4 *recv = reinterpret_cast<const float4 *>(smem + L::OFF_A) + (oc0 / 4) * BM + row;
            const int32_t slot_f4 = static_cast<int32_t>(ks_slot_bytes / 16);
            float acc[32];
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
                if (rr >= ks) break;
                float part[32];
                if (rr == krank) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) part[e] = __uint_as_float(r[e]);
                } else {
                    const float4 *src = recv + (rr < krank ? rr : rr - 1) * slot_f4;
                    float4 t[8];
#pragma unroll
                    for (int g = 0; g < 8; ++g) t[g] = src[g * BM];
#pragma unroll
                    for (int g = 0; g < 8; ++g) {
                        part[4 * g] = t[g].x;
                        part[4 * g + 1] = t[g].y;
                        part[4 * g + 2] = t[g].z;
                        part[4 * g + 3] = t[g].w;
                    }
                }
#pragma unroll
                for (int e = 0; e < 32; ++e) acc[e] = rr == 0 ? part[e] : acc[e] + part[e];
            }
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(acc[e]);
        };
        WorkItem w;
        for (int64_t t = worker; ok && work_item(p.sched, t, BN, w); t += workers) {
            const int32_t own0 = krank * ks_w; // first TMEM column of this CTA's window
            if (ks > 1) {
                w.n += own0;
                w.width = ks_w;
            }
            const Segment sg = segment_of<kGrouped>(w.m, BM * CL, p, seg);
            const int32_t m0 = sg.row0 + static_cast<int32_t>(rank) * BM; // first row of this CTA's rows
            int32_t rows_valid = sg.rows_left - static_cast<int32_t>(rank) * BM;
            rows_valid = rows_valid < 0 ? 0 : (rows_valid > BM ? BM : rows_valid);
            // A tile that runs past its group's last row must not store through
            // the D map (its rows would land in the next group): plain stores.
            const bool direct_tile = kGrouped && rows_valid < BM;
            const int32_t cab = p.c_bcast ? 0 : sg.ab;
            int nchunks = (p.N - w.n + CHUNK - 1) / CHUNK;
            if (nchunks > w.width / CHUNK) nchunks = w.width / CHUNK;
            if (p.N <= w.n) nchunks = 0;
            // Every wait of the epilogue ends in a vote, so that all 128 threads
            // leave together if any of them gave up (no thread is left behind
            // at a later bar.sync).
            const bool got = mbar_wait(&tfull[acc], acc_phase, ctl, kStatusTimeoutEpilogue);
            if (named_barrier_or(1, EPI_THREADS, !got)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (ks > 1) {
                uint8_t *ring = smem + L::OFF_A;
                uint8_t *send = ring + static_cast<uint32_t>(ks - 1) * ks_slot_bytes;
                // This CTA's MMAs are done, so its ring is idle: stage each peer's
                // columns of the partial sum in the send slots.
                for (int32_t j = 0; j < ks; ++j) {
                    if (j == krank) continue;
                    uint8_t *slot = send + static_cast<uint32_t>(j < krank ? j : j - 1) * ks_slot_bytes;
                    for (int32_t g = 0; g < ks_w / 32; g += 2) {
                        uint32_t r[2][32];
                        const uint32_t ta = tmem_base + acc * BN + static_cast<uint32_t>(j * ks_w + g * 32) + ((q * 32u) << 16);
                        tmem_ld32(ta, r[0]);
                        tmem_ld32(ta + 32, r[1]);
                        tc_wait_ld();
#pragma unroll
                        for (int h = 0; h < 2; ++h)
#pragma unroll
                            for (int i = 0; i < 32; i += 4)
                                *reinterpret_cast<uint4 *>(slot + ((static_cast<uint32_t>((g + h) * 8 + i / 4) * BM + row) << 4)) =
                                    make_uint4(r[h][i], r[h][i + 1], r[h][i + 2], r[h][i + 3]);
                    }
                }
                fence_proxy_async_smem(); // the bulk copies read what these threads wrote
                if (leader) {
                    // the receive slots may be written: tell the peers; expect their bytes
                    for (int32_t j = 0; j < ks; ++j)
                        if (j != krank) mbar_arrive_cluster(map_to_rank(smem_addr(ks_free), static_cast<uint32_t>(j)));
                    mbar_arrive_expect_tx(ks_recv, static_cast<uint32_t>(ks - 1) * ks_slot_bytes);
                }
                const bool freed = mbar_wait_cluster(ks_free, 0u, ctl, kStatusTimeoutReduce);
                if (named_barrier_or(1, EPI_THREADS, !freed)) {
                    ok = false;
                    break;
                }
                if (leader) {
                    for (int32_t j = 0; j < ks; ++j) {
                        if (j == krank) continue;
                        const uint32_t src = smem_addr(send + static_cast<uint32_t>(j < krank ? j : j - 1) * ks_slot_bytes);
                        const uint32_t dst = map_to_rank(
                            smem_addr(ring + static_cast<uint32_t>(krank < j ? krank : krank - 1) * ks_slot_bytes),
                            static_cast<uint32_t>(j));
                        bulk_copy_to_peer(dst, src, ks_slot_bytes, map_to_rank(smem_addr(ks_recv), static_cast<uint32_t>(j)));
                    }
                }
                const bool parts = mbar_wait_cluster(ks_recv, 0u, ctl, kStatusTimeoutReduce);
                if (named_barrier_or(1, EPI_THREADS, !parts)) {
                    ok = false;
                    break;
                }
            }
            // K split tail: this pair accumulated half of K over the whole tile,
            // and owns (stores) the column half given by its piece. It hands the
            // partner pair its partial sums of the partner's columns through the
            // workspace, flags them with this call's epoch, and takes the
            // partner's partial sums of its own columns in return; the chunk loop
            // below adds them. Every element is still written by one CTA, and the
            // sum of two fp32 parts is the same in either order.
            const bool tail_piece = kPair && p.ktail && w.width < BN;
            // The partner's partial sums land in this CTA's ring, idle now: the
            // pair's MMAs are done and a tail piece is a worker's last item.
            const float4 *partner = reinterpret_cast<const float4 *>(smem + L::OFF_A) + row;
            if (tail_piece) {
                const int64_t tile_i = (t - p.sched.whole) / 2;
                const uint32_t piece = static_cast<uint32_t>((w.n % BN) / w.width);
                float4 *mine = tail_slot(p, tile_i, rank, piece);
                const uint32_t other0 = (1u - piece) * 128u; // TMEM column of the partner's half
                for (int32_t g = 0; g < 4; g += 2) {
                    uint32_t r[2][32];
                    const uint32_t ta = tmem_base + acc * BN + other0 + static_cast<uint32_t>(g * 32) + ((q * 32u) << 16);
                    tmem_ld32(ta, r[0]);
                    tmem_ld32(ta + 32, r[1]);
                    tc_wait_ld();
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int i = 0; i < 32; i += 4)
                            __stcg(mine + static_cast<uint32_t>((g + h) * 8 + i / 4) * BM + row,
                                   make_float4(__uint_as_float(r[h][i]), __uint_as_float(r[h][i + 1]),
                                               __uint_as_float(r[h][i + 2]), __uint_as_float(r[h][i + 3])));
                }
                // Every thread's stores come before the barrier, and the leader's
                // release store after it is cumulative over them: a reader that
                // acquires the flag sees the whole slot.
                named_barrier_sync(1, EPI_THREADS);
                bool have = true;
                if (leader) {
                    st_release_gpu(tail_flag(p, tile_i, rank, piece), p.epoch);
                    uint32_t *theirs = tail_flag(p, tile_i, rank, 1u - piece);
                    have = flag_wait(theirs, p.epoch, ctl, kStatusTimeoutReduce);
                    if (have) {
                        *theirs = 0u; // consumed: the next call starts from a clear flag
                        // one bulk copy brings the partner's 64 KB into the ring
                        fence_proxy_async_global();
                        mbar_arrive_expect_tx(ks_recv, kTailSlotBytes);
                        bulk_load_g2s(smem + L::OFF_A, tail_slot(p, tile_i, rank, 1u - piece), kTailSlotBytes, ks_recv);
                        tail_loading = true;
                    }
                }
                if (named_barrier_or(1, EPI_THREADS, !have)) {
                    ok = false;
                    break;
                }
                const bool landed = mbar_wait(ks_recv, 0u, ctl, kStatusTimeoutReduce);
                if (named_barrier_or(1, EPI_THREADS, !landed)) {
                    ok = false;
                    break;
                }
            }
            // Adds the partner's partial sums of columns col0 .. col0+31 of this
            // CTA's column half, from the ring ([column / 4][row][4] layout).
            auto tail_add = [&](uint32_t(&r)[32], int32_t col0) {
                float4 v[8];
#pragma unroll
                for (int g = 0; g < 8; ++g) v[g] = partner[static_cast<uint32_t>(col0 / 4 + g) * BM];
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                    r[4 * g] = __float_as_uint(__uint_as_float(r[4 * g]) + v[g].x);
                    r[4 * g + 1] = __float_as_uint(__uint_as_float(r[4 * g + 1]) + v[g].y);
                    r[4 * g + 2] = __float_as_uint(__uint_as_float(r[4 * g + 2]) + v[g].z);
                    r[4 * g + 3] = __float_as_uint(__uint_as_float(r[4 * g + 3]) + v[g].w);
                }
            };
            // first TMEM column of the columns this CTA stores
            const int32_t tcol0 = tail_piece ? (w.n % BN) : own0;
            const uint32_t acc_now = acc;
            auto release = [&]() {
                // Whole accumulator read: hand it back to the MMA warp.
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (kPair)
                        mbar_arrive_cluster_relaxed(tempty0 + acc_now * 8u); // hands over no memory
                    else
                        mbar_arrive(&tempty[acc_now]);
                }
            };
            if (nchunks == 0) release(); // a piece entirely right of N: nothing to store
            for (int c = 0; c < nchunks; ++c) {
                uint8_t *buf = epi + slot * EPI_BUF_BYTES;
                const int32_t cb = w.n + c * CHUNK; // first column of this chunk
                const bool chunk_tma = cb < p.n_tma && !direct_tile;
                // the ragged cell [n_tma, N) when it falls in this chunk, else -1
                const int tail_cell = (p.N > p.n_tma && cb <= p.n_tma && p.n_tma < cb + CHUNK)
                                          ? (p.n_tma - cb) / (16 / (kOutF32 ? 4 : 2))
                                          : -1;
                const int32_t grow = m0 + static_cast<int32_t>(row); // row of this thread within its batch
                const bool row_ok = static_cast<int32_t>(row) < rows_valid;
                const int64_t crow = static_cast<int64_t>(cab) * p.sC + static_cast<int64_t>(grow) * p.ldc;
                const int64_t drow = static_cast<int64_t>(sg.ab) * p.sD + static_cast<int64_t>(grow) * p.ldd;
                // Fused epilogue: this row's aux cells for the chunk, all in flight at once,
                // while the staging buffer frees up and C arrives.
                uint4 auxq[8];
                if constexpr (kFused) {
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        auxq[j] = load_aux_cell<kOutF32>(p.epi, p.N, grow, row_ok, cb + j * (kOutF32 ? 4 : 8));
                }
                // The store that last used this buffer must have finished reading it.
                if (leader) bulk_wait_group_read<1>();
                named_barrier_sync(1, EPI_THREADS);
                if (has_beta && chunk_tma) {
                    if (leader) {
                        mbar_arrive_expect_tx(&cbar[slot], EPI_BUF_BYTES);
                        tma_load_3d(&tmC, &cbar[slot], buf, cb, m0, cab);
                    }
                    const bool gotc = mbar_wait(&cbar[slot], (cphase >> slot) & 1u, ctl, kStatusTimeoutEpilogue);
                    if (named_barrier_or(1, EPI_THREADS, !gotc)) {
                        ok = false;
                        break;
                    }
                    cphase ^= 1u << slot;
                }
                const uint32_t taddr =
                    tmem_base + acc * BN + static_cast<uint32_t>(tcol0 + c * CHUNK) + ((q * 32u) << 16);
                uint32_t r0[32];
                uint32_t r1[32];
                tmem_ld32(taddr, r0);
                if (!kOutF32) tmem_ld32(taddr + 32, r1);
                tc_wait_ld();
                if (ks > 1) {
                    ks_combine(r0, c * CHUNK);
                    if (!kOutF32) ks_combine(r1, c * CHUNK + 32);
                }
                if (tail_piece) {
                    tail_add(r0, c * CHUNK);
                    if (!kOutF32) tail_add(r1, c * CHUNK + 32);
                }
                if (c == nchunks - 1) release();
                uint8_t *rowp = buf + row * 128u;
                if (!kOutF32 && !kFused && !has_beta && !direct_tile && tail_cell < 0) {
                    // The common bf16 chunk (no C, no fused ops, no ragged cell):
                    // a short loop of its own. The general loop below is large
                    // enough that running it once per tile cost 0.5-0.8 us per
                    // chunk, measured, against about 0.15 for this one.
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t *src = j < 4 ? &r0[j * 8] : &r1[(j - 4) * 8];
                        float v[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            v[e] = kEpi == kEpiUnitAlpha ? __uint_as_float(src[e]) : p.alpha * __uint_as_float(src[e]);
                        *reinterpret_cast<uint4 *>(rowp + ((j ^ (row & 7u)) << 4)) =
                            make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                                       pack_bf16x2(v[6], v[7]));
                    }
                } else
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    uint4 *cell = reinterpret_cast<uint4 *>(rowp + ((j ^ (row & 7u)) << 4));
                    const bool tail = direct_tile || j == tail_cell;
                    if constexpr (kOutF32) {
                        float v[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            v[e] = kEpi == kEpiUnitAlpha ? __uint_as_float(r0[j * 4 + e])
                                                         : p.alpha * __uint_as_float(r0[j * 4 + e]);
                        if (tail) {
                            // ragged last columns: plain loads and stores of this row
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int32_t col = cb + j * 4 + e;
                                if (has_beta && row_ok && col < p.N)
                                    v[e] = fmaf(p.beta, static_cast<const float *>(p.C)[crow + col], v[e]);
                            }
                            if constexpr (kFused) epilogue_cell<4, true, kFused ? kEpi - 1 : 0>(p.epi, p.N, grow, row_ok, cb + j * 4, v, auxq[j]);
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int32_t col = cb + j * 4 + e;
                                if (row_ok && col < p.N) static_cast<float *>(p.D)[drow + col] = v[e];
                            }
                            continue;
                        }
                        if (has_beta) {
                            const uint4 cv = *cell;
                            v[0] = fmaf(p.beta, __uint_as_float(cv.x), v[0]);
                            v[1] = fmaf(p.beta, __uint_as_float(cv.y), v[1]);
                            v[2] = fmaf(p.beta, __uint_as_float(cv.z), v[2]);
                            v[3] = fmaf(p.beta, __uint_as_float(cv.w), v[3]);
                        }
                        if constexpr (kFused) epilogue_cell<4, true, kFused ? kEpi - 1 : 0>(p.epi, p.N, grow, row_ok, cb + j * 4, v, auxq[j]);
                        *cell = make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                                           __float_as_uint(v[3]));
                    } else {
                        float v[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const uint32_t bits = (j < 4) ? r0[j * 8 + e] : r1[(j - 4) * 8 + e];
                            v[e] = kEpi == kEpiUnitAlpha ? __uint_as_float(bits) : p.alpha * __uint_as_float(bits);
                        }
                        if (tail) {
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const int32_t col = cb + j * 8 + e;
                                if (has_beta && row_ok && col < p.N) {
                                    const uint16_t cbits = static_cast<const uint16_t *>(p.C)[crow + col];
                                    v[e] = fmaf(p.beta, __uint_as_float(static_cast<uint32_t>(cbits) << 16), v[e]);
                                }
                            }
                            if constexpr (kFused) epilogue_cell<8, false, kFused ? kEpi - 1 : 0>(p.epi, p.N, grow, row_ok, cb + j * 8, v, auxq[j]);
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const int32_t col = cb + j * 8 + e;
                                if (row_ok && col < p.N)
                                    static_cast<uint16_t *>(p.D)[drow + col] =
                                        static_cast<uint16_t>(pack_bf16x2(v[e], 0.0f) & 0xFFFFu);
                            }
                            continue;
                        }
                        if (has_beta) {
                            const uint4 cv = *cell;
                            const uint32_t cw[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                v[2 * e] = fmaf(p.beta, bf16lo_to_f32(cw[e]), v[2 * e]);
                                v[2 * e + 1] = fmaf(p.beta, bf16hi_to_f32(cw[e]), v[2 * e + 1]);
                            }
                        }
                        if constexpr (kFused) epilogue_cell<8, false, kFused ? kEpi - 1 : 0>(p.epi, p.N, grow, row_ok, cb + j * 8, v, auxq[j]);
                        *cell = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                                           pack_bf16x2(v[6], v[7]));
                    }
                }
                fence_proxy_async_smem();
                named_barrier_sync(1, EPI_THREADS);
                if (leader && chunk_tma) {
                    tma_store_3d(&tmD, buf, cb, m0, sg.ab);
                    bulk_commit_group();
                }
                slot ^= 1u;
            }
            if (!ok) break;
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        // The stores must have read the staging buffers before the CTA exits;
        // their global writes are complete when the grid is.
        if (leader) bulk_wait_group_read<0>();
        // K split: a CTA that gave up early must still not exit while a peer's
        // bulk copy into its ring may be in flight (a no-op once the copies
        // have landed). The same holds for the tail's bulk load.
        if ((ks > 1 || tail_loading) && leader && !drain_wait(ks_recv, 0u, p.timeout_ns) && p.status)
            atomicOr(p.status, kStatusTimeoutDrain);
    }

    tc_fence_before();
    if (kPair || ks > 1)
        cluster_sync(); // a peer may still arrive on this CTA's barriers (or write its ring) until here
    else
        __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        if constexpr (kPair)
            tmem_dealloc_pair(tmem_base, TMEM_COLS);
        else
            tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

} // namespace tiled
} // namespace tpg
