// Small-M weight-streaming bf16 GEMM for sm_103a (decode shapes, M <= 64).
//
// With a handful of token rows the GEMM is bound by reading B once from HBM,
// not by the tensor cores ("TorchInductor ganha suporte a GEMMs de alta
// performance com CuteDSL", BF16 results paragraph: decode shapes with M from 8
// to 64; "Implementing Tensor Parallelism Communication Overlays ...",
// "Performance Tradeoffs": as M shrinks the GEMM turns memory-bound). The
// kernel therefore computes the transposed product
//     D^T [N x M] = B^T [N x K] * A^T [K x M]
// so that the tensor core's 128-row M dimension runs over N (B is read as an
// N-major operand straight from its row-major layout) and the MMA's N
// dimension is the padded token count MT = roundup(M, 16). Each CTA streams
// 128-column panels of B through a deep TMA ring; A (a few hundred KB) stays
// in L2.
//
// Output ownership is per 128-column panel. With SPLIT > 1 (2, 3 or 4) the
// panel's K range is cut into SPLIT nearly equal parts between the CTAs of a
// cluster: the other CTAs send their fp32 partial sums through distributed
// shared memory and the first adds them in a fixed order (part 0 + part 1 +
// ...) and writes the panel, so the result is deterministic and no panel is
// written by two CTAs (no atomics, no global split-K buffer). Few panels (a
// narrow N) get a larger SPLIT, so that every SM streams part of B.
//
// Warp roles as in the tiled kernel: warp 0 TMA producer, warp 1 TMEM owner
// and MMA issuer, warps 2-5 epilogue (one TMEM lane quarter each, i.e. 32
// columns of D per warp, MT token rows per thread).
#pragma once

#include "epilogue.cuh"
#include "ptx.cuh"

namespace tpg {

struct StreamParams {
    int32_t M, N, K;
    int32_t nt;     // 128-wide panels along N
    int32_t kb;     // 64-wide K blocks in total
    int32_t mt_pad; // MMA N: M rounded up to a multiple of 16 (16..64)
    int32_t stages; // ring depth (host-computed from shared memory)
    float alpha, beta;
    const void *C;
    int64_t ldc;
    void *D;
    int64_t ldd;
    uint32_t *status;
    uint64_t timeout_ns;
    EpiParams epi; // read only by the kEpi instantiations
};

namespace stream {

constexpr int BN = 128; // output columns per panel (the MMA's M)
constexpr int BK = 64;
constexpr int MAX_STAGES = 12;
constexpr int THREADS = 192;
constexpr int EPI_THREADS = 128;
constexpr uint32_t B_BOX_BYTES = BK * 64 * 2;   // 64 K rows x 64 N
constexpr uint32_t B_STAGE_BYTES = 2 * B_BOX_BYTES;
constexpr uint32_t TMEM_COLS = 128;             // two accumulators of up to 64 columns
constexpr int MAX_SPLIT = 4;
// K blocks of a CTA's first panel whose B boxes are prefetched into L2 before
// the wait on the previous grid.
constexpr int PREFETCH_KB = 16;
// full, empty; tfull, tempty; red_full (per sending CTA, two slots); red_empty; drain
constexpr uint32_t NUM_BARS = 2 * MAX_STAGES + 2 + 2 + 2 * (MAX_SPLIT - 1) + 2 + 1;
constexpr uint32_t BAR_BYTES = NUM_BARS * 8 + 16;
constexpr uint32_t SMEM_LIMIT = 232448;

__host__ __device__ constexpr uint32_t a_slot_bytes(int mt) { return static_cast<uint32_t>(mt) * 128u; }
__host__ __device__ constexpr uint32_t stage_bytes(int mt) { return B_STAGE_BYTES + a_slot_bytes(mt); }
// One fp32 partial sum of a panel, laid out [MT / 4][BN][4]: the thread of D
// column c keeps its token rows 4g .. 4g+3 in the 16 bytes at (g * BN + c) * 16,
// so a warp's 32 columns fill 512 contiguous bytes (no bank conflicts).
__host__ __device__ constexpr uint32_t red_slot_bytes(int mt) { return static_cast<uint32_t>(BN) * mt * 4u; }

// Partial-sum slots of the first CTA of a cluster: two per sending CTA.
__host__ __device__ constexpr uint32_t red_bytes(int mt, int split) {
    return split > 1 ? static_cast<uint32_t>(split - 1) * 2u * red_slot_bytes(mt) : 0u;
}

// Stage count that fits beside the barrier block and the reduction slots,
// leaving 1 KB to align the base.
__host__ __device__ constexpr int max_stages(int mt, int split) {
    const uint32_t fixed = 1024 + BAR_BYTES + red_bytes(mt, split);
    const int s = fixed < SMEM_LIMIT ? static_cast<int>((SMEM_LIMIT - fixed) / stage_bytes(mt)) : 0;
    return s > MAX_STAGES ? MAX_STAGES : s;
}

__host__ __device__ constexpr uint32_t smem_bytes(int mt, int stages, int split) {
    return 1024 + stages * stage_bytes(mt) + red_bytes(mt, split) + BAR_BYTES;
}

__device__ __forceinline__ bool drain_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
    const uint32_t a = smem_addr(bar);
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 0; i < (1u << 28); ++i) {
        if (mbar_try_wait(a, parity)) return true;
        if ((i & 63u) == 63u && globaltimer_ns() - t0 > limit_ns) return false;
    }
    return false;
}

template <bool kOutF32, int SPLIT, bool kEpi>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_stream_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const StreamParams p) {
    static_assert(SPLIT >= 1 && SPLIT <= MAX_SPLIT, "K split of 1 to 4");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const int MT = p.mt_pad;
    const int S = p.stages;
    const uint32_t a_bytes = a_slot_bytes(MT);
    const uint32_t st_bytes = stage_bytes(MT);
    uint8_t *ring = smem;                                  // stage s: B boxes, then the A box
    uint8_t *red = smem + S * st_bytes;                    // SPLIT > 1: partial-sum slots
    uint8_t *barblk = red + red_bytes(MT, SPLIT);
    uint64_t *bars = reinterpret_cast<uint64_t *>(barblk);
    uint64_t *full = bars;
    uint64_t *empty = bars + MAX_STAGES;
    uint64_t *tfull = bars + 2 * MAX_STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *red_full = tempty + 2;  // in the first CTA, [sender - 1][slot]: that CTA's partial has landed
    uint64_t *red_empty = red_full + 2 * (MAX_SPLIT - 1); // in each sender, [slot]: the first CTA has consumed it
    uint64_t *drain = red_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(barblk + NUM_BARS * 8);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(barblk + NUM_BARS * 8 + 4);

    const uint32_t warp = threadIdx.x / 32;
    const uint32_t lane = threadIdx.x % 32;
    const uint32_t rank = SPLIT > 1 ? cluster_ctarank() : 0u;
    const int32_t cluster_id = static_cast<int32_t>(blockIdx.x) / SPLIT;
    const int32_t num_clusters = static_cast<int32_t>(gridDim.x) / SPLIT;

    // K blocks of this CTA: part `rank` of SPLIT nearly equal parts, in order.
    const int32_t kb_begin = static_cast<int32_t>(rank) * p.kb / SPLIT;
    const int32_t kb_end = (static_cast<int32_t>(rank) + 1) * p.kb / SPLIT;
    const int32_t my_kb = kb_end - kb_begin; // the host guarantees kb >= SPLIT, so >= 1

    if (threadIdx.x == 0) {
        for (int s = 0; s < MAX_STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], EPI_THREADS / 32);
            mbar_init(&red_empty[b], EPI_THREADS);
        }
        for (int b = 0; b < 2 * (MAX_SPLIT - 1); ++b) mbar_init(&red_full[b], EPI_THREADS);
        mbar_init(drain, 1);
        *abort_flag = 0u;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        // B is only read, and the prefetch is a hint (see tma_prefetch_2d), so
        // the first K blocks of this CTA's first panel can start on their way
        // from HBM while the previous grid in the stream is still finishing:
        // this CTA runs on an SM that grid has already left, during the
        // ragged end of its last panels. Only clusters that stream more than
        // one panel do it. A cluster with a single panel is short, and its
        // first loads would queue behind the prefetches.
        const int32_t n0 = cluster_id * BN;
        const int32_t pf_end =
            p.nt > num_clusters ? kb_begin + (my_kb < PREFETCH_KB ? my_kb : PREFETCH_KB) : kb_begin;
        for (int32_t kb = kb_begin; kb < pf_end; ++kb) {
            tma_prefetch_2d(&tmB, n0, kb * BK);
            if (n0 + 64 < p.N) tma_prefetch_2d(&tmB, n0 + 64, kb * BK);
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    if (SPLIT > 1)
        cluster_sync(); // the peers' barriers are initialised before any remote arrive
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
            const uint64_t stream_policy = policy_evict_first(); // B is read once
            const uint64_t keep_policy = policy_evict_last();    // A is read by every CTA
            uint32_t stage = 0, phase = 0;
            int64_t issued = 0;
            bool ok = true;
            for (int32_t t = cluster_id; t < p.nt && ok; t += num_clusters) {
                const int32_t n0 = t * BN;
                for (int32_t kb = kb_begin; kb < kb_end; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, ctl, kStatusTimeoutProducer)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[stage], B_STAGE_BYTES + a_bytes);
                    const int32_t k0 = kb * BK;
                    uint8_t *dst = ring + stage * st_bytes;
                    tma_load_2d_hint(&tmB, &full[stage], dst, n0, k0, stream_policy);
                    tma_load_2d_hint(&tmB, &full[stage], dst + B_BOX_BYTES, n0 + 64, k0, stream_policy);
                    tma_load_2d_hint(&tmA, &full[stage], dst + B_STAGE_BYTES, k0, 0, keep_policy);
                    ++issued;
                    if (++stage == static_cast<uint32_t>(S)) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                const int64_t pending = issued < S ? issued : S;
                uint32_t s = stage, ph = phase;
                for (int64_t i = 0; i < pending; ++i) {
                    if (s == 0) {
                        s = S - 1;
                        ph ^= 1u;
                    } else {
                        --s;
                    }
                    if (!drain_wait(&full[s], ph, p.timeout_ns) && p.status)
                        atomicOr(p.status, kStatusTimeoutDrain);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            // A operand = B^T panel (N-major), B operand = A^T (K-major rows of A).
            const uint32_t idesc = make_idesc_bf16_f32(BN, static_cast<uint32_t>(MT), true, false);
            uint32_t stage = 0, phase = 0;
            uint32_t acc = 0, acc_phase = 0;
            bool ok = true, any = false;
            for (int32_t t = cluster_id; t < p.nt && ok; t += num_clusters) {
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, ctl, kStatusTimeoutMma)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * 64u;
                for (int32_t i = 0; i < my_kb; ++i) {
                    if (!mbar_wait(&full[stage], phase, ctl, kStatusTimeoutMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t b_addr = smem_addr(ring + stage * st_bytes);
                    const uint32_t a_addr = b_addr + B_STAGE_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint64_t wdesc = make_smem_desc_sw128(b_addr + kk * 2048, B_BOX_BYTES, 1024);
                        const uint64_t xdesc = make_smem_desc_sw128(a_addr + kk * 32, 16, 1024);
                        tc_mma_f16(d_tmem, wdesc, xdesc, idesc, (i | kk) != 0 ? 1u : 0u);
                    }
                    any = true;
                    tc_commit(&empty[stage]);
                    if (++stage == static_cast<uint32_t>(S)) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit(&tfull[acc]);
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            if (!ok && any) {
                tc_commit(drain);
                if (!drain_wait(drain, 0, p.timeout_ns) && p.status)
                    atomicOr(p.status, kStatusTimeoutDrain);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue (warps 2..5)
        const uint32_t q = warp & 3u;
        const uint32_t col = q * 32u + lane; // D column within the panel = TMEM lane
        const bool has_beta = p.beta != 0.0f;
        uint32_t acc = 0, acc_phase = 0;
        uint32_t rslot = 0, rphase = 0;
        bool ok = true;
        for (int32_t t = cluster_id; t < p.nt && ok; t += num_clusters) {
            const int32_t n = t * BN + static_cast<int32_t>(col);
            const bool got = mbar_wait(&tfull[acc], acc_phase, ctl, kStatusTimeoutEpilogue);
            if (named_barrier_or(1, EPI_THREADS, !got)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float v[64];
            const uint32_t taddr = tmem_base + acc * 64u + ((q * 32u) << 16);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (c * 16 < MT) {
                    uint32_t r[16];
                    tmem_ld16(taddr + c * 16, r);
                    tc_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) v[c * 16 + e] = __uint_as_float(r[e]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }

            if (SPLIT > 1) {
                const uint32_t col_off = col * 16u;
                if (rank != 0) {
                    // Hand this part's partial sum to the first CTA.
                    uint8_t *slot = red + ((rank - 1) * 2 + rslot) * red_slot_bytes(MT);
                    const bool free_ok =
                        mbar_wait_cluster(&red_empty[rslot], rphase ^ 1u, ctl, kStatusTimeoutReduce);
                    if (named_barrier_or(1, EPI_THREADS, !free_ok)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dst = map_to_rank(smem_addr(slot + col_off), 0);
#pragma unroll
                    for (int m = 0; m < 64; m += 4)
                        if (m < MT) st_cluster_v4(dst + m * (BN * 4), v[m], v[m + 1], v[m + 2], v[m + 3]);
                    mbar_arrive_cluster(map_to_rank(smem_addr(&red_full[(rank - 1) * 2 + rslot]), 0));
                } else {
                    // part 0 + part 1 + ... + part SPLIT-1, always in this order
                    for (int r = 1; r < SPLIT && ok; ++r) {
                        const uint8_t *slot = red + ((r - 1) * 2 + rslot) * red_slot_bytes(MT);
                        const bool have =
                            mbar_wait_cluster(&red_full[(r - 1) * 2 + rslot], rphase, ctl, kStatusTimeoutReduce);
                        if (named_barrier_or(1, EPI_THREADS, !have)) {
                            ok = false;
                            break;
                        }
                        const float4 *src = reinterpret_cast<const float4 *>(slot + col_off);
#pragma unroll
                        for (int m = 0; m < 64; m += 4) {
                            if (m >= MT) break;
                            const float4 w = src[(m / 4) * BN];
                            v[m] += w.x;
                            v[m + 1] += w.y;
                            v[m + 2] += w.z;
                            v[m + 3] += w.w;
                        }
                        mbar_arrive_cluster(map_to_rank(smem_addr(&red_empty[rslot]), static_cast<uint32_t>(r)));
                    }
                    if (!ok) break;
                }
                if (++rslot == 2) {
                    rslot = 0;
                    rphase ^= 1u;
                }
                if (rank != 0) continue; // the first CTA owns and writes the panel
            }

            if (n < p.N) {
#pragma unroll
                for (int m = 0; m < 64; ++m) {
                    if (m >= p.M) break;
                    float x = p.alpha * v[m];
                    if constexpr (kOutF32) {
                        if (has_beta)
                            x = fmaf(p.beta, static_cast<const float *>(p.C)[m * p.ldc + n], x);
                        if constexpr (kEpi) x = epilogue_one<true>(p.epi, m, n, x);
                        static_cast<float *>(p.D)[m * p.ldd + n] = x;
                    } else {
                        if (has_beta) {
                            const uint16_t cb = static_cast<const uint16_t *>(p.C)[m * p.ldc + n];
                            x = fmaf(p.beta, __uint_as_float(static_cast<uint32_t>(cb) << 16), x);
                        }
                        if constexpr (kEpi) x = epilogue_one<false>(p.epi, m, n, x);
                        static_cast<uint16_t *>(p.D)[m * p.ldd + n] =
                            static_cast<uint16_t>(pack_bf16x2(x, 0.0f) & 0xFFFFu);
                    }
                }
            }
        }
    }

    tc_fence_before();
    if (SPLIT > 1)
        cluster_sync(); // no CTA leaves while a peer may still arrive on its barriers
    else
        __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

} // namespace stream
} // namespace tpg
