// Inline-PTX building blocks for sm_103a: mbarriers with bounded waits, TMA
// (cp.async.bulk.tensor) loads and stores, and the tcgen05 tensor-core family
// (TMEM allocation, MMA, commit, TMEM loads, fences). Encodings follow the
// public PTX ISA documentation for tcgen05 and the tensor-map API of CUDA 13.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace tpg {

// ---------------------------------------------------------------- status bits
// Written (atomicOr) into the handle's device status word by a kernel that
// gave up on a wait. The host maps any non-zero word to TPGEMM_ERR_TIMEOUT.
enum : uint32_t {
    kStatusTimeoutProducer = 1u << 0,
    kStatusTimeoutMma = 1u << 1,
    kStatusTimeoutEpilogue = 1u << 2,
    kStatusTimeoutDrain = 1u << 3,
    kStatusTimeoutReduce = 1u << 4,
    kStatusSelftest = 1u << 8,
};

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t lane_id() {
    uint32_t l;
    asm volatile("mov.u32 %0, %%laneid;" : "=r"(l));
    return l;
}

__device__ __forceinline__ bool elect_one() {
    uint32_t pred = 0;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "elect.sync _|p, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(pred));
    return pred != 0;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Makes barrier initialisation visible to the async proxy (TMA, tcgen05) and to
// the other CTAs of the cluster.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Arrive on the barrier at shared::cluster address `cluster_addr` (possibly in
// a peer CTA), with release semantics at cluster scope.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}

// The same arrive without release semantics, for a signal that hands over no
// memory: an epilogue's "accumulator read" signal, given after
// tcgen05.wait::ld has completed the TMEM loads (so the next MMAs cannot
// overwrite columns still being read) and tcgen05.fence::before_thread_sync.
// A cluster-scope release there waited for the thread's earlier memory
// operations to reach cluster scope, measured at 1-2 us per tile.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(addr), "r"(parity)
        : "memory");
    return ok != 0;
}

// Two ring stages at once: a (possibly blocking) wait on the first barrier and
// a non-blocking test of the second, issued together so that their latencies
// overlap. Bit 0 of the result: the first phase is complete; bit 1: the second.
__device__ __forceinline__ uint32_t mbar_try_wait_and_test(uint32_t a1, uint32_t p1, uint32_t a2, uint32_t p2) {
    uint32_t r1, r2;
    asm volatile(
        "{\n\t.reg .pred q1, q2;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 q1, [%2], %3;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 q2, [%4], %5;\n\t"
        "selp.u32 %0, 1, 0, q1;\n\t"
        "selp.u32 %1, 2, 0, q2;\n\t}\n"
        : "=r"(r1), "=r"(r2)
        : "r"(a1), "r"(p1), "r"(a2), "r"(p2)
        : "memory");
    return r1 | r2;
}

// The same over three stages: bit 0 the first (waited on), bits 1 and 2 the
// next two (tested).
__device__ __forceinline__ uint32_t mbar_try_wait_and_test2(uint32_t a1, uint32_t p1, uint32_t a2, uint32_t p2,
                                                            uint32_t a3, uint32_t p3) {
    uint32_t r1, r2, r3;
    asm volatile(
        "{\n\t.reg .pred q1, q2, q3;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 q1, [%3], %4;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 q2, [%5], %6;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 q3, [%7], %8;\n\t"
        "selp.u32 %0, 1, 0, q1;\n\t"
        "selp.u32 %1, 2, 0, q2;\n\t"
        "selp.u32 %2, 4, 0, q3;\n\t}\n"
        : "=r"(r1), "=r"(r2), "=r"(r3)
        : "r"(a1), "r"(p1), "r"(a2), "r"(p2), "r"(a3), "r"(p3)
        : "memory");
    return r1 | r2 | r3;
}

// Cluster-scope acquire form, for barriers that peers arrive on remotely.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(addr), "r"(parity)
        : "memory");
    return ok != 0;
}

// Shared state of one CTA's bounded waits: a flag any role sets when it gives
// up, so that the others stop waiting too, and the time limit.
struct WaitCtl {
    volatile uint32_t *abort_flag; // shared memory
    uint32_t *status;              // global status word (may be null)
    uint64_t timeout_ns;
};

// Slow path of a bounded wait: polls the barrier, and every 64 polls checks the
// CTA's abort flag and the elapsed %globaltimer time. Gives up (returns false)
// when the time limit passes, when another role has aborted, or after 2^31
// polls in case the timer does not advance. On a timeout it records `code` in
// the status word and raises the abort flag.
template <bool kCluster>
__device__ __noinline__ bool mbar_wait_slow(uint32_t addr, uint32_t parity, WaitCtl ctl,
                                            uint32_t code) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1; i < (1u << 31); ++i) {
        if (kCluster ? mbar_try_wait_cluster(addr, parity) : mbar_try_wait(addr, parity))
            return true;
        if ((i & 63u) == 0) {
            if (*ctl.abort_flag) return false;
            if (globaltimer_ns() - t0 > ctl.timeout_ns) break;
        }
    }
    *ctl.abort_flag = 1u;
    if (ctl.status) atomicOr(ctl.status, code);
    return false;
}

__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, const WaitCtl &ctl,
                                          uint32_t code) {
    const uint32_t a = smem_addr(bar);
    if (mbar_try_wait(a, parity)) return true;
    return mbar_wait_slow<false>(a, parity, ctl, code);
}

__device__ __forceinline__ bool mbar_wait_cluster(uint64_t *bar, uint32_t parity,
                                                  const WaitCtl &ctl, uint32_t code) {
    const uint32_t a = smem_addr(bar);
    if (mbar_try_wait_cluster(a, parity)) return true;
    return mbar_wait_slow<true>(a, parity, ctl, code);
}

// ---------------------------------------------------------------- flags in global memory
// A flag another CTA of the grid sets after writing data that this CTA then
// reads (release store / acquire load at GPU scope).
__device__ __forceinline__ void st_release_gpu(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Bounded wait until *flag == want, with the same give-up rules as the
// mbarrier waits (time limit, another role's abort, a hard poll cap).
static __device__ __noinline__ bool flag_wait(const uint32_t *flag, uint32_t want, WaitCtl ctl, uint32_t code) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1; i < (1u << 31); ++i) {
        if (ld_acquire_gpu(flag) == want) return true;
        if ((i & 15u) == 0) {
            if (*ctl.abort_flag) return false;
            if (globaltimer_ns() - t0 > ctl.timeout_ns) break;
        }
    }
    *ctl.abort_flag = 1u;
    if (ctl.status) atomicOr(ctl.status, code);
    return false;
}

// ---------------------------------------------------------------- programmatic dependent launch
// A kernel launched with programmatic stream serialisation may start while the
// previous kernel in the stream is still running. It does its prologue (barrier
// init, TMEM allocation, tensor-map prefetch), then waits here until the
// previous grid has completed and its memory is visible, before it reads any
// input or writes any output.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Lets the next kernel in the stream be scheduled as soon as SMs free up.
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- cluster
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// shared::cta address -> shared::cluster address of the same offset in CTA `rank`.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t cta_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(cta_addr), "r"(rank));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

__device__ __forceinline__ void st_cluster_v4(uint32_t cluster_addr, float a, float b, float c,
                                              float d) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(cluster_addr), "f"(a),
                 "f"(b), "f"(c), "f"(d)
                 : "memory");
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 2-D tiled load global -> shared; completion is signalled on `bar` as
// transaction bytes. c0 is the innermost (contiguous) coordinate.
__device__ __forceinline__ void tma_load_2d(const CUtensorMap *m, uint64_t *bar, void *dst,
                                            int32_t c0, int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_addr(bar)), "r"(c0), "r"(c1)
        : "memory");
}

// L2 prefetch of one box of a 2-D tensor map: a hint that moves no data into
// shared memory and completes on no barrier. L2 is the point of coherence for
// every load of this GPU, so a prefetch issued before an earlier grid has
// finished writing the same bytes can never make a later load see stale data.
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap *m, int32_t c0, int32_t c1) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(m)),
                 "r"(c0), "r"(c1)
                 : "memory");
}

__device__ __forceinline__ void tma_load_2d_hint(const CUtensorMap *m, uint64_t *bar, void *dst,
                                                 int32_t c0, int32_t c1, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_addr(bar)), "r"(c0), "r"(c1), "l"(policy)
        : "memory");
}

// 3-D forms: the third coordinate selects a batch (or group) slice.
__device__ __forceinline__ void tma_load_3d(const CUtensorMap *m, uint64_t *bar, void *dst, int32_t c0,
                                            int32_t c1, int32_t c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_addr(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// 4-D forms: B viewed as [slice][64-column group][K row][64 columns], so that
// one box brings several 64-column groups of one K block.
__device__ __forceinline__ void tma_load_4d(const CUtensorMap *m, uint64_t *bar, void *dst, int32_t c0,
                                            int32_t c1, int32_t c2, int32_t c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_addr(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d_pair(const CUtensorMap *m, uint32_t bar_cluster_addr, void *dst,
                                                 int32_t c0, int32_t c1, int32_t c2, int32_t c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster_addr), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d_pair(const CUtensorMap *m, uint32_t bar_cluster_addr, void *dst,
                                                 int32_t c0, int32_t c1, int32_t c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster_addr), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap *m, const void *src, int32_t c0, int32_t c1,
                                             int32_t c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(m)),
                 "r"(smem_addr(src)), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

// 2-D tiled store shared -> global (out-of-range elements are clipped).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *m, const void *src, int32_t c0,
                                             int32_t c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::
                     "l"(reinterpret_cast<uint64_t>(m)),
                 "r"(smem_addr(src)), "r"(c0), "r"(c1)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Waits until at most N committed bulk groups of this thread still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait_group() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) reads of the same memory.
// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned) from
// this CTA's shared memory to another CTA's of the cluster; the bytes complete
// as transactions on the destination CTA's mbarrier `mbar_cluster`.
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst_cluster, uint32_t src_cta, uint32_t bytes,
                                                  uint32_t mbar_cluster) {
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     dst_cluster),
                 "r"(src_cta), "r"(bytes), "r"(mbar_cluster)
                 : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Orders this thread's generic-proxy view of global memory (e.g. an acquire
// load of a flag) before the async-proxy operations it issues next (a bulk
// copy that reads what the flag guards).
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Bulk copy (TMA, no tensor map) of `bytes` (a multiple of 16, both addresses
// 16-byte aligned) from global memory into this CTA's shared memory; the bytes
// complete as transactions on `bar`.
__device__ __forceinline__ void bulk_load_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_addr(dst)),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Named barrier that also ORs a predicate over the participating threads, so a
// group of threads takes one decision together (e.g. "some wait gave up").
__device__ __forceinline__ bool named_barrier_or(uint32_t id, uint32_t threads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}\n"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(threads)
        : "memory");
    return r != 0;
}

// L2 eviction-priority policies for cache hints.
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---------------------------------------------------------------- tcgen05
// TMEM allocation is warp-wide; the allocated base address is written to shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc], kind::f16 (bf16 in, fp32 accumulate).
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// tc_commit on a barrier given by its shared-memory address.
__device__ __forceinline__ void tc_commit_addr(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// Arrives once on `bar` when every tcgen05.mma issued so far by this thread has completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tc_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 lanes x 32 bits, 16 consecutive columns: thread t of the warp receives
// TMEM lane (lane base + t), columns col .. col+15.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// Same shape, 32 consecutive columns.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// ---------------------------------------------------------------- tcgen05, CTA pair
// With .cta_group::2 the two CTAs of a cluster pair act as one MMA unit: A and
// the accumulator are split by rows (128 per CTA), B by columns, each CTA
// holding its share at the same shared-memory offset. TMEM is allocated
// collectively: one warp of each CTA executes the same alloc/dealloc.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// Issued by one thread of the even CTA only; computes the pair's 256-row tile.
__device__ __forceinline__ void tc_mma_f16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrives once on the barrier at the same offset (a shared-memory address) in
// every CTA of `cta_mask` when all prior pair MMAs of this thread have completed.
__device__ __forceinline__ void tc_commit_pair_mc_addr(uint32_t bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar),
        "h"(cta_mask)
        : "memory");
}

// Arrives once on the barrier at the same offset in every CTA of `cta_mask`
// when all prior pair MMAs of this thread have completed.
__device__ __forceinline__ void tc_commit_pair_mc(uint64_t *bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(smem_addr(bar)),
        "h"(cta_mask)
        : "memory");
}

// TMA load into this CTA's shared memory whose completion is signalled on an
// mbarrier that may live in the peer CTA of the pair (shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(const CUtensorMap *m, uint32_t bar_cluster_addr,
                                                 void *dst, int32_t c0, int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster_addr), "r"(c0), "r"(c1)
        : "memory");
}

// ---------------------------------------------------------------- descriptors
// Shared-memory matrix descriptor (tcgen05 "matrix descriptor"):
//   bits  0-13  start address >> 4
//   bits 16-29  leading-dimension byte offset >> 4
//   bits 32-45  stride-dimension byte offset >> 4
//   bits 46-48  fixed 0b001
//   bits 49-51  base offset (0: every swizzle atom used here is 1024-byte aligned)
//   bit  52     leading-dimension offset mode (0: relative)
//   bits 61-63  swizzle mode (2: 128-byte swizzle)
// For a K-major operand with 128-byte swizzle, a row holds 64 bf16 of K, rows
// are 128 bytes apart and groups of 8 rows are `sbo` bytes apart; the leading
// offset is not used. For an MN-major operand with 128-byte swizzle, a row
// holds 64 bf16 of M (or N), consecutive K rows are 128 bytes apart, groups of
// 8 K rows are `sbo` apart and the next 64-wide block along M/N is `lbo` apart.
__device__ __forceinline__ uint64_t make_smem_desc_sw128(uint32_t saddr, uint32_t lbo,
                                                         uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;
    d |= 2ull << 61;
    return d;
}

// Instruction descriptor for tcgen05.mma kind::f16 with bf16 A and B and an
// fp32 accumulator:
//   bits 4-5 D format (1 = f32), bits 7-9 A format (1 = bf16), bits 10-12 B
//   format (1 = bf16), bit 15 A major (0 = K, 1 = MN), bit 16 B major,
//   bits 17-22 N >> 3, bits 24-28 M >> 4.
__host__ __device__ constexpr uint32_t make_idesc_bf16_f32(uint32_t m, uint32_t n, bool a_mn_major,
                                                           bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn_major) << 15) |
           (static_cast<uint32_t>(b_mn_major) << 16) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

// ---------------------------------------------------------------- tcgen05, block-scaled (MX) operands
// Shared-memory matrix descriptor without swizzling: rows of 16 bytes, groups
// of 8 rows `sbo` bytes apart (the leading offset is not used by a matrix
// one 16-byte column wide).
__device__ __forceinline__ uint64_t make_smem_desc_plain(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;
    return d;
}

// Copies a 32-row x 16-byte shared-memory matrix into TMEM: row i lands in
// lane i, columns taddr .. taddr+3 (bytes 4j .. 4j+3 of the row in column
// taddr + j), and the same 32 lanes are written in each of the four lane
// quarters (warpx4). Asynchronous; ordered before later tcgen05.mma of the
// same thread, and tracked by tcgen05.commit like an MMA.
__device__ __forceinline__ void tc_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// D[tmem] (+)= (A scaled) * (B scaled), kind::mxf8f6f4 with one E8M0 scale per
// 32 K elements (scale_vec::1X): FP8 A and B from shared-memory descriptors,
// the scales of A's rows and B's columns in TMEM at sfa / sfb (the byte of
// each 32-bit TMEM cell is chosen by the scale-factor IDs of idesc).
__device__ __forceinline__ void tc_mma_mxf8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}\n" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// CTA-pair forms, issued by one thread of the even CTA. The copy takes the
// same shared-memory offset in both CTAs of the pair and writes each CTA's
// chunk into that CTA's TMEM; the MMA computes the pair's 256-row tile, each
// CTA's 128 rows with the A scales in its own TMEM and the B scales of all N
// columns, which each CTA therefore holds in full.
__device__ __forceinline__ void tc_cp_32x128b_x4_pair(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
__device__ __forceinline__ void tc_mma_mxf8_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                 uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}\n" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= (A scaled) * (B scaled), kind::mxf4nvf4 (packed E2M1 A and B,
// K = 64): with kNv, scale_vec::4X, four scales per row per MMA (one per 16
// elements), the four bytes of each TMEM scale cell; else scale_vec::2X, two
// per row (one per 32 elements), the two bytes from the scale-factor ID on.
// The scale format (E4M3 or E8M0) is bit 23 of idesc. kPair: the CTA-pair
// form, issued by one thread of the even CTA.
template <bool kPair, bool kNv>
__device__ __forceinline__ void tc_mma_fp4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    if constexpr (kPair && kNv)
        asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
                     "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;"
                     "\n\t}\n" ::"r"(d_tmem),
                     "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
                     : "memory");
    else if constexpr (kPair)
        asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
                     "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;"
                     "\n\t}\n" ::"r"(d_tmem),
                     "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
                     : "memory");
    else if constexpr (kNv)
        asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
                     "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;"
                     "\n\t}\n" ::"r"(d_tmem),
                     "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
                     : "memory");
    else
        asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
                     "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;"
                     "\n\t}\n" ::"r"(d_tmem),
                     "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
                     : "memory");
}

// Instruction descriptor of a block-scaled MMA, kind::mxf8f6f4, both operands
// K-major, E8M0 scales:
//   bits 4-5 B scale-factor ID, bits 7-9 A format and 10-12 B format (0 E4M3,
//   1 E5M2), bits 17-22 N >> 3, bit 23 scale type (1 = E8M0), bits 24-28
//   M >> 4, bits 29-30 A scale-factor ID.
__host__ __device__ constexpr uint32_t make_idesc_mxf8(uint32_t m, uint32_t n, uint32_t a_fmt, uint32_t b_fmt) {
    return (a_fmt << 7) | (b_fmt << 10) | ((n >> 3) << 17) | (1u << 23) | ((m >> 4) << 24);
}
// kind::mxf4nvf4: both operands E2M1 (format 1) and K-major; the scale format
// bit is 0 for E4M3 (NVFP4) and 1 for E8M0 (MXFP4).
__host__ __device__ constexpr uint32_t make_idesc_fp4(uint32_t m, uint32_t n, bool e8m0_scales) {
    return (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((e8m0_scales ? 1u : 0u) << 23) | ((m >> 4) << 24);
}
__host__ __device__ constexpr uint32_t idesc_mx_sf_ids(uint32_t a_id, uint32_t b_id) {
    return (b_id << 4) | (a_id << 29);
}

// ---------------------------------------------------------------- conversions
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    // cvt.rn.bf16x2.f32 takes the high half first.
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float bf16lo_to_f32(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t v) {
    return __uint_as_float(v & 0xFFFF0000u);
}

} // namespace tpg
