// Small kernels beside the two GEMM paths:
//  - the K == 0 case, where the product is empty and D = beta * C (zeros when
//    beta == 0, C not read), the BLAS convention for an empty inner dimension;
//  - the watchdog self-test, one CTA that waits on an mbarrier nobody arrives
//    at and must give up after its time limit with an error status, never hang
//    ("Implementing Tensor Parallelism Communication Overlays ...", "Real-world
//    Failure Modes": a stuck wait must be detected and reported, not block
//    forever).
#pragma once

#include "epilogue.cuh"
#include "ptx.cuh"

namespace tpg {

template <bool kOutF32, bool kEpi>
__global__ void __launch_bounds__(256) epilogue_only_kernel(int32_t M, int32_t N, float beta, const void *C,
                                                            int64_t ldc, void *D, int64_t ldd, EpiParams epi) {
    const int64_t total = static_cast<int64_t>(M) * N;
    for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t i = idx / N;
        const int32_t j = static_cast<int32_t>(idx - i * N);
        float c = 0.0f;
        if (beta != 0.0f) {
            if constexpr (kOutF32)
                c = beta * static_cast<const float *>(C)[i * ldc + j];
            else
                c = beta * __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t *>(C)[i * ldc + j]) << 16);
        }
        if constexpr (kEpi) c = epilogue_one<kOutF32>(epi, i, j, c);
        if constexpr (kOutF32)
            static_cast<float *>(D)[i * ldd + j] = c;
        else
            static_cast<uint16_t *>(D)[i * ldd + j] = static_cast<uint16_t>(pack_bf16x2(c, 0.0f) & 0xFFFFu);
    }
}

// One warp; lane 0 waits on a barrier whose phase can never complete. The
// bounded wait gives up after timeout_ns and records kStatusSelftest.
__global__ void watchdog_selftest_kernel(uint32_t *status, uint64_t timeout_ns) {
    __shared__ uint64_t bar;
    __shared__ uint32_t abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0u;
        fence_barrier_init();
    }
    __syncwarp();
    if (threadIdx.x == 0) {
        const WaitCtl ctl{&abort_flag, status, timeout_ns};
        (void)mbar_wait(&bar, 0u, ctl, kStatusSelftest);
    }
    __syncwarp();
}

} // namespace tpg
