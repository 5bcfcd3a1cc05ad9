// Persistent, warp-specialised block-scaled (MX) GEMM for sm_103a:
//
//     D = alpha * sum over K blocks b of (SA[:, b] SB[:, b]^T) .* (A_b * B_b) + beta * C
//
// the scaled_mm of "TorchInductor ganha suporte a GEMMs de alta performance
// com CuteDSL" (the enablement paragraph names scaled_mm; the results paragraph
// measures MXFP8). A and B hold FP8 elements (E4M3 or E5M2) and every 32
// consecutive elements along K share one E8M0 scale per row of A and per
// column of B, the MX formats of the OCP Microscaling specification. The
// tensor cores apply the scales themselves: tcgen05.mma kind::mxf8f6f4 with
// scale_vec::1X reads one scale byte per row (of A) and per column (of B) from
// TMEM for each K = 32 instruction.
//
// Two modes of one kernel template, on the grouped-raster persistent schedule
// of the bf16 kernel; each tile has one owner ("cuTile Rust explained",
// "Ownership crosses the launch boundary"):
//   kPair = false  one CTA per SM owns 128 x kBN tiles (kBN = 128 or 192).
//   kPair = true   the two CTAs of a cluster pair own a 256 x 256 tile through
//                  tcgen05.mma.cta_group::2 (M = 256, N = 256) issued by the
//                  even CTA; each CTA stages its own 128 rows of A and of B's
//                  transpose. A 256-wide block-scaled MMA gives the tensor pipe
//                  128 cycles of work per SM, more than issuing it costs the
//                  issuing thread (192-wide ones, 96 cycles, capped the kernel
//                  near 80% of the FP8 rate). Two 256-column accumulators would
//                  fill TMEM and leave no room for the scales, so a pair has one;
//                  the epilogue reads it whole into registers (packed bf16)
//                  before it stages anything, so the next tile's MMAs wait only
//                  for that read.
// Roles, connected by mbarriers:
//   warp 0      TMA producer: per 128-wide K block, one A box (128 rows x 128
//               bytes) and one B box (kBN / CTAs rows of B's transpose x 128
//               bytes), both K-major with 128-byte swizzle, plus the K block's
//               scale chunks: 512 bytes for the CTA's 128 rows of A and one or
//               two for the tile's rows of B (all of them, in both CTAs of a
//               pair), copied as they are from the caller's blocked layout. The
//               scale chunks are issued first and complete on a barrier of
//               their own, so they reach TMEM while the operands are in flight.
//   warp 6      scale copier (even CTA): once a stage's scales have landed,
//               one lane copies its scale chunks into the stage's TMEM scale columns
//               (tcgen05.cp, 32 lanes x 16 bytes, repeated in all four lane
//               quarters, into both CTAs' TMEM in pair mode) and commits them
//               to the stage's scales-ready barrier. Keeping the copies off the
//               MMA thread leaves that thread four MMAs, one wait and one
//               commit per stage. FP4 stages hold three or four times as
//               many chunks, so warps 6 and 7 share them: each copies the
//               chunks of two of the four MMAs and signals its own barrier,
//               and the MMA thread issues each pair of MMAs once its half of
//               the scales is in.
//   warp 1      allocates TMEM (fp32 accumulators of kBN columns, two or, for
//               pairs, one, and per ring stage 4 scale columns for A and 8 for
//               B); one lane (of the even CTA) issues the four K = 32 MMAs of a
//               stage once its operands have landed and its scales are in TMEM,
//               scale byte j of each TMEM cell going with MMA j; tcgen05.commit
//               frees the stage (in both CTAs).
//   warps 2-5   epilogue, as in the bf16 kernel: TMEM -> registers -> alpha,
//               beta*C -> one rounding -> swizzled staging -> TMA store, each
//               CTA its own 128 rows.
//
// The scale layout, per operand of R rows and K/32 scale columns: chunks of 128
// rows x 4 scale columns (512 bytes), chunk (row block rb, column block cb)
// at byte (rb * ceil(K/128) + cb) * 512, and inside a chunk the scale of row r,
// column c at byte (r % 32) * 16 + (r / 32) * 4 + c. A chunk is therefore the
// 32 x 16-byte matrix that tcgen05.cp places so that TMEM lane r % 32, column
// r / 32, byte c holds scale (r, c): row r's scale for MMA c of the K block.
// For B tiles of 192 columns a tile may start 64 rows into a chunk; its scale
// columns then start two TMEM columns into the copied pair of chunks.
//
// FP4 (kFmt = kFmtNvf4 or kFmtMxf4), the same page's NVFP4 and MXF4 GEMMs:
// A and B hold E2M1 elements two to a byte (the even element in the low four
// bits), so a 128-byte stage row is 256 elements and each of a stage's four
// MMAs (kind::mxf4nvf4, K = 64) takes 32 bytes, the same descriptor steps as
// FP8. NVFP4 scales every 16 elements with an E4M3 byte (scale_vec::4X: the
// four bytes of a TMEM cell are the four scales of one MMA, one 512-byte chunk
// per MMA and 128 rows); MXFP4 every 32 with an E8M0 byte (scale_vec::2X: one
// chunk serves two MMAs, which take bytes 0-1 and 2-3 of each cell). Tiles are
// 256 x 256 or 256 x 192 on CTA pairs, 128 x 192 or 128 x 128 on one CTA; a
// tile's B scales are the one or two row blocks of 128 it reaches (a 192-wide
// tile starts 0 or 64 rows into the first). The scale maps are rank 3 ([row
// block][chunk][128 words]): a stage's chunks arrive in one box per operand,
// and chunks past the end of a row block (K not a multiple of the stage's 256
// elements) or past the last row block read as zero scales rather than the
// next row block's. 192-wide FP4 tiles have one accumulator, as pairs do.
#pragma once

#include <cuda_bf16.h>

#include "ptx.cuh"
#include "schedule.cuh"

namespace tpg {

struct MxParams {
    int32_t M, N, K;
    int32_t kb;       // K blocks of 128
    Schedule sched;   // tiles of 128 (CTA pairs: 256) x kBN, no column pieces
    int32_t n_tma;    // columns [0, n_tma) of C and D go through the tensor maps (see TiledParams)
    int32_t sfb_rows; // row blocks of 128 in B's scales: chunks past the last are not loaded
    int32_t sf_kc;    // scale chunks per row block: ceil(K / 128)
    uint32_t idesc;   // instruction descriptor without the scale-factor IDs
    float alpha, beta;
    const void *C;
    int64_t ldc;
    void *D;
    int64_t ldd;
    uint32_t *status;
    uint64_t timeout_ns;
};

namespace mx {

// Element and scale formats (the kernel's kFmt template argument).
constexpr int kFmtMxf8 = 0; // FP8 elements, one E8M0 scale per 32 (kind::mxf8f6f4, scale_vec::1X)
constexpr int kFmtNvf4 = 1; // packed E2M1, one E4M3 scale per 16 (kind::mxf4nvf4, scale_vec::4X)
constexpr int kFmtMxf4 = 2; // packed E2M1, one E8M0 scale per 32 (kind::mxf4nvf4, scale_vec::2X)

constexpr int BM = 128; // rows per CTA
constexpr int BK = 128; // K elements (bytes) per stage: four MMAs of K = 32, four scale columns
constexpr int EPI_THREADS = 128;
constexpr uint32_t SF_CHUNK = 512;
constexpr uint32_t EPI_BUF_BYTES = BM * 128;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t SF_TMEM_STRIDE = 16; // TMEM columns per stage: A at +0 (4), B at +4 (8)

// kARows < 128 (1-CTA, M <= kARows): A's TMA box is kARows rows (64 or 32),
// so a stage holds 8 or 4 KB of A instead of 16 and the ring one or two
// stages more; the MMA still reads 128 rows, and the rows past the box (the
// next stages' bytes) only reach accumulator rows that are never stored.
template <int kBN, bool kPair, int kARows = 128, int kFmt = kFmtMxf8>
struct Layout {
    static constexpr bool FP4 = kFmt != kFmtMxf8;
    static_assert(kFmt == kFmtMxf8 || kFmt == kFmtNvf4 || kFmt == kFmtMxf4, "format");
    static_assert(kPair ? (kBN == 256 || (FP4 && kBN == 192)) : (kBN == 128 || kBN == 192), "tile width");
    static_assert(kARows == 128 || (!kPair && kBN == 192 && (kARows == 64 || kARows == 32)),
                  "the small-M rings are 1-CTA, 192 wide");
    static constexpr int CL = kPair ? 2 : 1;
    // FP4: scale chunks per stage and row block (a stage is 256 elements of K:
    // four NVFP4 chunks of 64, two MXFP4 chunks of 128), and row blocks of B's
    // scales a tile reaches (a 192-wide tile starts 0 or 64 rows into one and
    // ends in the next).
    static constexpr int CPS = kFmt == kFmtNvf4 ? 4 : 2;
    static constexpr int NRB = kBN == 128 ? 1 : 2;
    // One accumulator in pair mode (two of 256 columns would fill TMEM and
    // leave no room for the scales) and for FP4's 192-wide tiles (two would
    // leave room for two stages of scales); then one epilogue staging buffer.
    static constexpr int ACCS = (kPair || (FP4 && kBN == 192)) ? 1 : 2;
    static constexpr int STAGES =
        FP4 ? (kPair ? (kBN == 256 ? 5 : 6)
                     : (kBN == 128 ? 5 : (kARows == 32 ? 6 : (kARows == 64 ? 5 : 4))))
            : (kPair ? 6 : (kARows == 32 ? 6 : (kARows == 64 ? 5 : (kBN == 192 ? 4 : 5))));
    static constexpr int EPI_BUFS = ACCS == 1 ? 1 : 2;
    static constexpr uint32_t A_ROWS = kARows; // rows of A's box
    static constexpr uint32_t A_BYTES = A_ROWS * BK;
    static constexpr uint32_t B_ROWS = kBN / CL; // rows of B's transpose this CTA stages
    static constexpr uint32_t B_BYTES = B_ROWS * BK;
    // FP8: A chunk at 0, B chunks at 512 and 1024 (and 1536 for 192-wide tiles
    // that straddle two row blocks). FP4: A's chunks, then B's, row block by
    // row block.
    static constexpr uint32_t SF_BYTES = FP4 ? CPS * SF_CHUNK * (1 + NRB) : (kPair ? 1536 : 2048);
    // TMEM columns per stage: FP8 A at +0 (4), B at +4 (8); FP4 four per chunk,
    // A's CPS chunks first, then B's, the NRB row blocks of one chunk together.
    static constexpr uint32_t SF_TSTRIDE = FP4 ? 4 * CPS * (1 + NRB) : SF_TMEM_STRIDE;
    static constexpr uint32_t OFF_A = 0;
    static constexpr uint32_t OFF_B = OFF_A + STAGES * A_BYTES;
    static_assert(OFF_A + (STAGES - 1) * A_BYTES + BM * BK <= OFF_B + STAGES * (kBN / CL) * BK,
                  "the MMA's 128-row reads of A stay inside the operand ring");
    static constexpr uint32_t OFF_SF = OFF_B + STAGES * B_BYTES;
    // the staging buffers are 128-byte swizzled, a pattern taken from address
    // bits 7-9: they start on a 1024-byte boundary
    static constexpr uint32_t OFF_EPI = (OFF_SF + STAGES * SF_BYTES + 1023) / 1024 * 1024;
    static constexpr uint32_t OFF_BAR = OFF_EPI + EPI_BUFS * EPI_BUF_BYTES;
    // full, empty, scales ready, tfull, tempty, c, drain, scale-copy drain
    // FP4 splits a stage's scale copies over two warps, each with its own
    // scales-ready barrier: the first copies the chunks of MMAs 0 and 1, the
    // second those of MMAs 2 and 3, and the MMAs of each half start as soon
    // as their scales are in.
    static constexpr int COPIERS = FP4 ? 2 : 1;
    static constexpr int THREADS = (6 + COPIERS) * 32;
    // full (operands), empty, scales landed, scales ready (per copier), tfull,
    // tempty, c, drain, scale-copy drain (per copier)
    static constexpr uint32_t NUM_BARS = (3 + COPIERS) * STAGES + 2 + 2 + 2 + 1 + COPIERS;
    static constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;
    static constexpr uint32_t SF_COL0 = ACCS * kBN; // first TMEM column of the scale region
    static_assert(SF_COL0 + STAGES * SF_TSTRIDE <= TMEM_COLS, "TMEM overflow");
    static_assert(SMEM_BYTES <= 232448, "exceeds the 227 KB shared-memory limit per CTA");
    static_assert(OFF_A % 1024 == 0 && OFF_B % 1024 == 0 && A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0,
                  "128-byte swizzled operand stages start on 1024-byte boundaries");
    static_assert(OFF_SF % 128 == 0 && SF_BYTES % 128 == 0, "scale boxes land on 128-byte boundaries");
};

__device__ __forceinline__ bool mx_drain_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
    const uint32_t a = smem_addr(bar);
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 0; i < (1u << 28); ++i) {
        if (mbar_try_wait(a, parity)) return true;
        if ((i & 63u) == 63u && globaltimer_ns() - t0 > limit_ns) return false;
    }
    return false;
}

// Busy-waits `ns` nanoseconds (abort path only).
__device__ __forceinline__ void mx_settle(uint64_t ns) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 0; i < (1u << 26) && globaltimer_ns() - t0 < ns; ++i) {
    }
}

template <bool kOutF32, int kBN, bool kPair, int kARows = 128, int kFmt = kFmtMxf8>
__global__ void __launch_bounds__(Layout<kBN, kPair, kARows, kFmt>::THREADS, 1)
    gemm_mx_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                   const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmD,
                   const MxParams p) {
    using L = Layout<kBN, kPair, kARows, kFmt>;
    constexpr int STAGES = L::STAGES;
    constexpr int CL = L::CL;
    constexpr int CHUNK = kOutF32 ? 32 : 64; // output columns per 128-byte staging row

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);
    uint64_t *full = bars;
    uint64_t *empty = bars + STAGES;
    uint64_t *sffull = bars + 2 * STAGES;  // a stage's scale chunks have landed
    uint64_t *sfready = bars + 3 * STAGES; // copier c's barrier of stage s: sfready[c * STAGES + s]
    uint64_t *tfull = bars + (3 + L::COPIERS) * STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *cbar = tempty + 2;
    uint64_t *drain = cbar + 2;
    uint64_t *sfdrain = drain + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + L::OFF_MISC + 4);

    const uint32_t warp = threadIdx.x / 32;
    const uint32_t lane = threadIdx.x % 32;
    const uint32_t rank = kPair ? cluster_ctarank() : 0u; // 0 = the even CTA, which issues copies and MMAs
    const int64_t worker = static_cast<int64_t>(blockIdx.x) / CL;
    const int64_t workers = static_cast<int64_t>(gridDim.x) / CL;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&sffull[s], 1);
            for (int c = 0; c < L::COPIERS; ++c) mbar_init(&sfready[c * STAGES + s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            // every epilogue warp of the worker hands the accumulator back
            mbar_init(&tempty[b], CL * EPI_THREADS / 32);
            mbar_init(&cbar[b], 1);
        }
        mbar_init(drain, 1);
        for (int c = 0; c < L::COPIERS; ++c) mbar_init(&sfdrain[c], 1);
        *abort_flag = 0u;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        prefetch_tensormap(&tmSA);
        prefetch_tensormap(&tmSB);
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
    if constexpr (kPair)
        cluster_sync(); // both CTAs' barriers initialised and TMEM allocated
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    grid_dependency_wait();
    grid_launch_dependents();

    const WaitCtl ctl{abort_flag, p.status, p.timeout_ns};

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (both CTAs)
        if (lane == 0) {
            // In pair mode both CTAs' loads complete on the even CTA's barriers.
            // A stage's scale chunks go first, on their own barrier, so that the
            // copier can move them into TMEM while the operands are in flight.
            const uint32_t full0 = kPair ? map_to_rank(smem_addr(full), 0) : 0u;
            const uint32_t sffull0 = kPair ? map_to_rank(smem_addr(sffull), 0) : 0u;
            uint32_t stage = 0, phase = 0;
            int64_t issued = 0;
            bool ok = true;
            WorkItem w;
            for (int64_t t = worker; ok && work_item(p.sched, t, kBN, w); t += workers) {
                const int32_t arow = w.m * CL + static_cast<int32_t>(rank); // this CTA's 128-row block of A
                const int32_t m0 = arow * BM;
                const int32_t n0 = w.n + static_cast<int32_t>(rank * L::B_ROWS);
                const int32_t rb = w.n / 128; // B's first scale row block
                // a 192-wide FP8 tile may reach into the next row block of B's scales
                const bool two = !L::FP4 && kBN + (w.n % 128) > 128 && rb + 1 < p.sfb_rows;
                // FP4 scale boxes are whole (zero-filled past the ends), so always complete
                const uint32_t sf_tx = CL * (L::FP4 ? L::SF_BYTES : SF_CHUNK * (two ? 3u : 2u));
                const uint32_t tx = CL * (L::A_BYTES + L::B_BYTES);
                const int32_t ca = static_cast<int32_t>(arow * p.sf_kc);
                const int32_t cb = static_cast<int32_t>(rb * p.sf_kc);
                for (int32_t kb = 0; kb < p.kb; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, ctl, kStatusTimeoutProducer)) {
                        ok = false;
                        break;
                    }
                    uint8_t *adst = smem + L::OFF_A + stage * L::A_BYTES;
                    uint8_t *bdst = smem + L::OFF_B + stage * L::B_BYTES;
                    uint8_t *sf = smem + L::OFF_SF + stage * L::SF_BYTES;
                    if constexpr (kPair) {
                        if (rank == 0) {
                            mbar_arrive_expect_tx(&sffull[stage], sf_tx);
                            mbar_arrive_expect_tx(&full[stage], tx);
                        }
                        const uint32_t sb = sffull0 + stage * 8u, fb = full0 + stage * 8u;
                        if constexpr (L::FP4) {
                            // this CTA's row block of A's scales; all of the tile's row blocks of B's
                            const int32_t sc = kb * L::CPS;
                            tma_load_3d_pair(&tmSA, sb, sf, 0, sc, arow);
                            tma_load_3d_pair(&tmSB, sb, sf + L::CPS * SF_CHUNK, 0, sc, rb);
                        } else {
                            tma_load_2d_pair(&tmSA, sb, sf, 0, ca + kb);
                            tma_load_2d_pair(&tmSB, sb, sf + SF_CHUNK, 0, cb + kb);
                            if (two)
                                tma_load_2d_pair(&tmSB, sb, sf + 2 * SF_CHUNK, 0,
                                                 cb + static_cast<int32_t>(p.sf_kc) + kb);
                        }
                        tma_load_2d_pair(&tmA, fb, adst, kb * BK, m0);
                        tma_load_2d_pair(&tmB, fb, bdst, kb * BK, n0);
                    } else {
                        mbar_arrive_expect_tx(&sffull[stage], sf_tx);
                        mbar_arrive_expect_tx(&full[stage], tx);
                        if constexpr (L::FP4) {
                            const int32_t sc = kb * L::CPS;
                            tma_load_3d(&tmSA, &sffull[stage], sf, 0, sc, arow);
                            tma_load_3d(&tmSB, &sffull[stage], sf + L::CPS * SF_CHUNK, 0, sc, rb);
                        } else {
                            tma_load_2d(&tmSA, &sffull[stage], sf, 0, ca + kb);
                            tma_load_2d(&tmSB, &sffull[stage], sf + SF_CHUNK, 0, cb + kb);
                            if (two)
                                tma_load_2d(&tmSB, &sffull[stage], sf + 2 * SF_CHUNK, 0,
                                            cb + static_cast<int32_t>(p.sf_kc) + kb);
                        }
                        tma_load_2d(&tmA, &full[stage], adst, kb * BK, m0);
                        tma_load_2d(&tmB, &full[stage], bdst, kb * BK, n0);
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
                        if (!mx_drain_wait(&sffull[s], ph, p.timeout_ns) && p.status)
                            atomicOr(p.status, kStatusTimeoutDrain);
                        if (!mx_drain_wait(&full[s], ph, p.timeout_ns) && p.status)
                            atomicOr(p.status, kStatusTimeoutDrain);
                    }
                }
                // The odd CTA's loads complete on the even CTA's barriers, which it
                // cannot wait on: give them time to land.
                if (kPair) mx_settle(200000);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issue (even CTA only in pair mode)
        if (lane == 0 && rank == 0) {
            const uint64_t adesc0 = make_smem_desc_sw128(smem_addr(smem + L::OFF_A), 16, 1024);
            const uint64_t bdesc0 = make_smem_desc_sw128(smem_addr(smem + L::OFF_B), 16, 1024);
            const uint32_t ready_a = smem_addr(sfready), empty_a = smem_addr(empty), full_a = smem_addr(full);
            uint32_t stage = 0, phase = 0;
            uint32_t acc = 0, acc_phase = 0;
            bool ok = true;
            bool any = false;
            WorkItem w;
            for (int64_t t = worker; ok && work_item(p.sched, t, kBN, w); t += workers) {
                // B's scale columns start (w.n % 128) / 32 TMEM columns into the copied chunks
                const uint32_t sfb_skip = static_cast<uint32_t>((w.n % 128) / 32);
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, ctl, kStatusTimeoutMma)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * kBN;
                // FP8: issues the four MMAs of K block kb from the current stage and frees the stage.
                auto issue = [&](int32_t kb) {
                    const uint32_t sfa_t = tmem_base + L::SF_COL0 + stage * L::SF_TSTRIDE;
                    const uint32_t sfb_t = sfa_t + 4 + sfb_skip;
                    const uint64_t ad = adesc0 + stage * (L::A_BYTES >> 4);
                    const uint64_t bd = bdesc0 + stage * (L::B_BYTES >> 4);
#pragma unroll
                    for (int kk = 0; kk < BK / 32; ++kk) {
                        // K = 32 FP8 elements are 32 bytes: +2 in the descriptors' address field
                        const uint32_t accumulate = (kb != 0 || kk != 0) ? 1u : 0u;
                        const uint32_t idesc = p.idesc | idesc_mx_sf_ids(kk, kk);
                        if constexpr (kPair)
                            tc_mma_mxf8_pair(d_tmem, ad + kk * 2, bd + kk * 2, idesc, sfa_t, sfb_t, accumulate);
                        else
                            tc_mma_mxf8(d_tmem, ad + kk * 2, bd + kk * 2, idesc, sfa_t, sfb_t, accumulate);
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
                if constexpr (L::FP4) {
                    for (int32_t kb = 0; kb < p.kb && ok; ++kb) {
                        const uint32_t sfa_t = tmem_base + L::SF_COL0 + stage * L::SF_TSTRIDE;
                        // a 192-wide tile's B scales start (w.n % 128) / 32 columns into each MMA's group
                        const uint32_t sfb_t = sfa_t + 4 * L::CPS + sfb_skip;
                        const uint64_t ad = adesc0 + stage * (L::A_BYTES >> 4);
                        const uint64_t bd = bdesc0 + stage * (L::B_BYTES >> 4);
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            // this half's scales are in TMEM (and, before the first half, the
                            // stage's operands have landed)
                            if (!mbar_wait(&sfready[half * STAGES + stage], phase, ctl, kStatusTimeoutMma) ||
                                (half == 0 && !mbar_wait(&full[stage], phase, ctl, kStatusTimeoutMma))) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
#pragma unroll
                            for (int k2 = 0; k2 < 2; ++k2) {
                                // K = 64 FP4 elements are 32 bytes: +2 in the descriptors' address
                                // field. NVFP4: chunk kk, all four bytes; MXFP4: chunk kk / 2,
                                // bytes 2 (kk % 2) and up.
                                const int kk = 2 * half + k2;
                                const uint32_t accumulate = (kb != 0 || kk != 0) ? 1u : 0u;
                                const uint32_t g = kFmt == kFmtNvf4 ? kk : kk / 2;
                                const uint32_t id = kFmt == kFmtNvf4 ? 0u : 2u * (kk % 2);
                                const uint32_t idesc = p.idesc | idesc_mx_sf_ids(id, id);
                                tc_mma_fp4<kPair, kFmt == kFmtNvf4>(d_tmem, ad + kk * 2, bd + kk * 2, idesc,
                                                                  sfa_t + 4 * g, sfb_t + 4 * L::NRB * g, accumulate);
                            }
                            any = true;
                        }
                        if (!ok) break;
                        if constexpr (kPair)
                            tc_commit_pair_mc_addr(empty_a + stage * 8u, 0x3);
                        else
                            tc_commit_addr(empty_a + stage * 8u);
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                } else {
                    for (int32_t kb = 0; kb < p.kb;) {
                        // Wait until the stage's operands have landed and its scales are in
                        // TMEM, and test the next stage in the same breath: when both are
                        // ready, one wait serves two K blocks.
                        const uint32_t nstage = stage + 1 == STAGES ? 0u : stage + 1;
                        const uint32_t nphase = stage + 1 == STAGES ? phase ^ 1u : phase;
                        const uint32_t st2 =
                            mbar_try_wait_and_test(ready_a + stage * 8u, phase, ready_a + nstage * 8u, nphase);
                        if ((!(st2 & 1u) && !mbar_wait(&sfready[stage], phase, ctl, kStatusTimeoutMma)) ||
                            !mbar_wait(&full[stage], phase, ctl, kStatusTimeoutMma)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        issue(kb++);
                        // the next stage too, if its scales are in and its operands have landed
                        if ((st2 & 2u) && kb < p.kb && mbar_try_wait(full_a + stage * 8u, phase)) {
                            tc_fence_after();
                            issue(kb++);
                        }
                    }
                }
                if (!ok) break;
                if constexpr (kPair)
                    tc_commit_pair_mc(&tfull[acc], 0x3);
                else
                    tc_commit(&tfull[acc]);
                if (++acc == static_cast<uint32_t>(L::ACCS)) {
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
                if (!mx_drain_wait(drain, 0, p.timeout_ns) && p.status) atomicOr(p.status, kStatusTimeoutDrain);
            }
        }
        __syncwarp();
    } else if (warp >= 6) {
        // ------------------------------------------------ scale copies into TMEM (even CTA)
        const int cw = static_cast<int>(warp) - 6; // copier index
        if (lane == 0 && rank == 0) {
            // a scale chunk: 32 rows of 16 bytes, groups of 8 rows 128 bytes apart
            const uint64_t sdesc0 = make_smem_desc_plain(smem_addr(smem + L::OFF_SF), 512, 128);
            const uint32_t sffull_a = smem_addr(sffull);
            uint64_t *ready = sfready + cw * STAGES;
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            bool any = false;
            WorkItem w;
            for (int64_t t = worker; ok && work_item(p.sched, t, kBN, w); t += workers) {
                for (int32_t kb = 0; kb < p.kb; ++kb) {
                    // Stage s was last read by MMAs that completed before the producer
                    // could refill it, so its TMEM scale columns are free once its
                    // scales have landed.
                    if (!mbar_try_wait(sffull_a + stage * 8u, phase) &&
                        !mbar_wait(&sffull[stage], phase, ctl, kStatusTimeoutMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sfa_t = tmem_base + L::SF_COL0 + stage * L::SF_TSTRIDE;
                    const uint64_t sd = sdesc0 + stage * (L::SF_BYTES >> 4);
                    if constexpr (L::FP4) {
                        // A's chunk j to column 4j; B's chunk j of row block r to
                        // 4 CPS + 4 (NRB j + r), so that one MMA's B scales are NRB * 4
                        // consecutive columns, row r of the tile in column r / 32. Copier
                        // cw takes chunks [cw CPS / 2, (cw + 1) CPS / 2): those of MMAs
                        // 2 cw and 2 cw + 1.
#pragma unroll
                        for (int j = cw * L::CPS / 2; j < (cw + 1) * L::CPS / 2; ++j) {
                            const uint64_t src = sd + ((j * SF_CHUNK) >> 4);
                            if constexpr (kPair)
                                tc_cp_32x128b_x4_pair(sfa_t + 4 * j, src);
                            else
                                tc_cp_32x128b_x4(sfa_t + 4 * j, src);
#pragma unroll
                            for (int r = 0; r < L::NRB; ++r) {
                                const uint64_t srcb = sd + ((((1 + r) * L::CPS + j) * SF_CHUNK) >> 4);
                                const uint32_t dst = sfa_t + 4 * L::CPS + 4 * (L::NRB * j + r);
                                if constexpr (kPair)
                                    tc_cp_32x128b_x4_pair(dst, srcb);
                                else
                                    tc_cp_32x128b_x4(dst, srcb);
                            }
                        }
                        if constexpr (kPair)
                            tc_commit_pair_mc(&ready[stage], 0x1);
                        else
                            tc_commit(&ready[stage]);
                    } else if constexpr (kPair) {
                        tc_cp_32x128b_x4_pair(sfa_t, sd);
                        tc_cp_32x128b_x4_pair(sfa_t + 4, sd + (SF_CHUNK >> 4));
                        tc_cp_32x128b_x4_pair(sfa_t + 8, sd + (2 * SF_CHUNK >> 4));
                        tc_commit_pair_mc(&ready[stage], 0x1);
                    } else {
                        tc_cp_32x128b_x4(sfa_t, sd);
                        tc_cp_32x128b_x4(sfa_t + 4, sd + (SF_CHUNK >> 4));
                        if constexpr (kBN > 128) tc_cp_32x128b_x4(sfa_t + 8, sd + (2 * SF_CHUNK >> 4));
                        tc_commit(&ready[stage]);
                    }
                    any = true;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok && any) {
                // Wait for every copy issued so far before TMEM is freed.
                if constexpr (kPair)
                    tc_commit_pair_mc(&sfdrain[cw], 0x1);
                else
                    tc_commit(&sfdrain[cw]);
                if (!mx_drain_wait(&sfdrain[cw], 0, p.timeout_ns) && p.status)
                    atomicOr(p.status, kStatusTimeoutDrain);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue (warps 2..5, both CTAs)
        const uint32_t q = warp & 3u;        // TMEM lane quarter this warp may read
        const uint32_t row = q * 32u + lane; // row of the CTA's 128 rows held by this thread
        const bool leader = threadIdx.x == 64;
        const bool has_beta = p.beta != 0.0f;
        const uint32_t tempty0 = kPair ? map_to_rank(smem_addr(tempty), 0) : 0u;
        uint8_t *epi = smem + L::OFF_EPI;
        uint32_t acc = 0, acc_phase = 0;
        uint32_t slot = 0;
        uint32_t cphase = 0;
        bool ok = true;
        WorkItem w;
        for (int64_t t = worker; ok && work_item(p.sched, t, kBN, w); t += workers) {
            const int32_t m0 = (w.m * CL + static_cast<int32_t>(rank)) * BM;
            int32_t rows_valid = p.M - m0;
            rows_valid = rows_valid < 0 ? 0 : (rows_valid > BM ? BM : rows_valid);
            int nchunks = (p.N - w.n + CHUNK - 1) / CHUNK;
            if (nchunks > kBN / CHUNK) nchunks = kBN / CHUNK;
            const bool got = mbar_wait(&tfull[acc], acc_phase, ctl, kStatusTimeoutEpilogue);
            if (named_barrier_or(1, EPI_THREADS, !got)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t acc_now = acc;
            auto release = [&]() {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (kPair)
                        mbar_arrive_cluster_relaxed(tempty0 + acc_now * 8u); // hands over no memory
                    else
                        mbar_arrive(&tempty[acc_now]);
                }
            };
            if (nchunks == 0) release();
            if constexpr (L::ACCS == 1 && !kOutF32) {
                if (!has_beta && p.n_tma == p.N) {
                    // One accumulator: the next tile's MMAs wait until this one is
                    // read. So read all kBN columns first, packed to bf16 in registers
                    // (alpha applied, one rounding), hand the accumulator back, and
                    // only then stage and store the chunks.
                    uint32_t packed[kBN / 2];
                    // two 32-column loads in flight per wait: the drain's length is
                    // the loads' latency, one wait per pair of groups
#pragma unroll
                    for (int g = 0; g < kBN / 32; g += 2) {
                        uint32_t ra[32], rb[32];
                        const uint32_t ta = tmem_base + acc * kBN + static_cast<uint32_t>(g * 32) + ((q * 32u) << 16);
                        tmem_ld32(ta, ra);
                        tmem_ld32(ta + 32, rb);
                        tc_wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            packed[g * 16 + e] = pack_bf16x2(p.alpha * __uint_as_float(ra[2 * e]),
                                                             p.alpha * __uint_as_float(ra[2 * e + 1]));
                            packed[g * 16 + 16 + e] = pack_bf16x2(p.alpha * __uint_as_float(rb[2 * e]),
                                                                  p.alpha * __uint_as_float(rb[2 * e + 1]));
                        }
                    }
                    release();
                    // N is a whole number of 16-byte cells here, so every chunk goes
                    // through the tensor map; rows past M are clipped by the store.
                    uint8_t *rowp = epi + row * 128u;
#pragma unroll
                    for (int c = 0; c < kBN / CHUNK; ++c) {
                        if (c >= nchunks) break;
                        if (leader) bulk_wait_group_read<0>(); // the last store has read the buffer
                        named_barrier_sync(1, EPI_THREADS);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int base = c * 32 + j * 4; // packed[base .. base+3]: this cell's 8 columns
                            *reinterpret_cast<uint4 *>(rowp + ((j ^ (row & 7u)) << 4)) =
                                make_uint4(packed[base], packed[base + 1], packed[base + 2], packed[base + 3]);
                        }
                        fence_proxy_async_smem();
                        named_barrier_sync(1, EPI_THREADS);
                        if (leader) {
                            tma_store_2d(&tmD, epi, w.n + c * CHUNK, m0);
                            bulk_commit_group();
                        }
                    }
                    if (++acc == static_cast<uint32_t>(L::ACCS)) {
                        acc = 0;
                        acc_phase ^= 1u;
                    }
                    continue;
                }
            }
            for (int c = 0; c < nchunks; ++c) {
                uint8_t *buf = epi + slot * EPI_BUF_BYTES;
                const int32_t cb = w.n + c * CHUNK;
                const bool chunk_tma = cb < p.n_tma;
                const int tail_cell = (p.N > p.n_tma && cb <= p.n_tma && p.n_tma < cb + CHUNK)
                                          ? (p.n_tma - cb) / (16 / (kOutF32 ? 4 : 2))
                                          : -1;
                const int32_t grow = m0 + static_cast<int32_t>(row);
                const bool row_ok = static_cast<int32_t>(row) < rows_valid;
                const int64_t crow = static_cast<int64_t>(grow) * p.ldc;
                const int64_t drow = static_cast<int64_t>(grow) * p.ldd;
                // The store that last used this buffer must have finished reading it.
                if (leader) {
                    if constexpr (L::EPI_BUFS == 2)
                        bulk_wait_group_read<1>();
                    else
                        bulk_wait_group_read<0>();
                }
                named_barrier_sync(1, EPI_THREADS);
                if (has_beta && chunk_tma) {
                    if (leader) {
                        mbar_arrive_expect_tx(&cbar[slot], EPI_BUF_BYTES);
                        tma_load_2d(&tmC, &cbar[slot], buf, cb, m0);
                    }
                    const bool gotc = mbar_wait(&cbar[slot], (cphase >> slot) & 1u, ctl, kStatusTimeoutEpilogue);
                    if (named_barrier_or(1, EPI_THREADS, !gotc)) {
                        ok = false;
                        break;
                    }
                    cphase ^= 1u << slot;
                }
                const uint32_t taddr = tmem_base + acc * kBN + static_cast<uint32_t>(c * CHUNK) + ((q * 32u) << 16);
                uint32_t r0[32];
                uint32_t r1[32];
                tmem_ld32(taddr, r0);
                if (!kOutF32) tmem_ld32(taddr + 32, r1);
                tc_wait_ld();
                if (c == nchunks - 1) release();
                uint8_t *rowp = buf + row * 128u;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    uint4 *cell = reinterpret_cast<uint4 *>(rowp + ((j ^ (row & 7u)) << 4));
                    const bool tail = j == tail_cell;
                    if constexpr (kOutF32) {
                        float v[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) v[e] = p.alpha * __uint_as_float(r0[j * 4 + e]);
                        if (tail) {
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int32_t col = cb + j * 4 + e;
                                if (row_ok && col < p.N) {
                                    if (has_beta) v[e] = fmaf(p.beta, static_cast<const float *>(p.C)[crow + col], v[e]);
                                    static_cast<float *>(p.D)[drow + col] = v[e];
                                }
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
                        *cell = make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                                           __float_as_uint(v[3]));
                    } else {
                        float v[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const uint32_t bits = (j < 4) ? r0[j * 8 + e] : r1[(j - 4) * 8 + e];
                            v[e] = p.alpha * __uint_as_float(bits);
                        }
                        if (tail) {
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const int32_t col = cb + j * 8 + e;
                                if (row_ok && col < p.N) {
                                    if (has_beta) {
                                        const uint16_t cbits = static_cast<const uint16_t *>(p.C)[crow + col];
                                        v[e] = fmaf(p.beta, __uint_as_float(static_cast<uint32_t>(cbits) << 16), v[e]);
                                    }
                                    static_cast<uint16_t *>(p.D)[drow + col] =
                                        static_cast<uint16_t>(pack_bf16x2(v[e], 0.0f) & 0xFFFFu);
                                }
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
                        *cell = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                                           pack_bf16x2(v[6], v[7]));
                    }
                }
                fence_proxy_async_smem();
                named_barrier_sync(1, EPI_THREADS);
                if (leader && chunk_tma) {
                    tma_store_2d(&tmD, buf, cb, m0);
                    bulk_commit_group();
                }
                if constexpr (L::EPI_BUFS == 2) slot ^= 1u;
            }
            if (!ok) break;
            if (++acc == static_cast<uint32_t>(L::ACCS)) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (leader) bulk_wait_group_read<0>();
    }

    tc_fence_before();
    if constexpr (kPair)
        cluster_sync(); // the peer may still arrive on this CTA's barriers until here
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

} // namespace mx
} // namespace tpg
