// Instantiations of the block-scaled (MX) GEMM kernel: 1-CTA tiles 128 or 192
// columns wide and CTA-pair tiles of 256 x 256, bf16 or fp32 output. The host
// library reaches them through the functions below (launch.cuh).
#include "launch.cuh"

namespace tpg {

namespace {
template <bool kOutF32, int kBN, bool kPair, int kARows = 128>
bool set_limit() {
    return cudaFuncSetAttribute(mx::gemm_mx_kernel<kOutF32, kBN, kPair, kARows>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(mx::Layout<kBN, kPair, kARows>::SMEM_BYTES)) == cudaSuccess;
}
template <bool kOutF32, int kBN, bool kPair, int kARows = 128>
cudaError_t launch_one(const MxLaunch &l) {
    return launch_ex(mx::gemm_mx_kernel<kOutF32, kBN, kPair, kARows>, l.grid, mx::Layout<kBN, kPair, kARows>::THREADS,
                     static_cast<int>(mx::Layout<kBN, kPair, kARows>::SMEM_BYTES), kPair ? 2 : 1, true, l.stream,
                     *l.a, *l.b, *l.sa, *l.sb, *l.c, *l.d, *l.p);
}
} // namespace

cudaError_t mx_launch(const MxLaunch &l) {
    if (l.pair) {
        if (l.tile_n != 256 || l.grid % 2 != 0) return cudaErrorInvalidValue;
        return l.f32 ? launch_one<true, 256, true>(l) : launch_one<false, 256, true>(l);
    }
    if (l.tile_n == 192 && l.a_rows == 32)
        return l.f32 ? launch_one<true, 192, false, 32>(l) : launch_one<false, 192, false, 32>(l);
    if (l.tile_n == 192 && l.a_rows == 64)
        return l.f32 ? launch_one<true, 192, false, 64>(l) : launch_one<false, 192, false, 64>(l);
    if (l.tile_n == 192) return l.f32 ? launch_one<true, 192, false>(l) : launch_one<false, 192, false>(l);
    if (l.tile_n == 128) return l.f32 ? launch_one<true, 128, false>(l) : launch_one<false, 128, false>(l);
    return cudaErrorInvalidValue;
}

bool mx_set_limits() {
    bool ok = set_limit<false, 128, false>();
    ok = set_limit<true, 128, false>() && ok;
    ok = set_limit<false, 192, false>() && ok;
    ok = set_limit<true, 192, false>() && ok;
    ok = set_limit<false, 192, false, 64>() && ok;
    ok = set_limit<true, 192, false, 64>() && ok;
    ok = set_limit<false, 192, false, 32>() && ok;
    ok = set_limit<true, 192, false, 32>() && ok;
    ok = set_limit<false, 256, true>() && ok;
    ok = set_limit<true, 256, true>() && ok;
    return ok;
}

int mx_smem_bytes(int tile_n, bool pair, int a_rows) {
    if (pair) return static_cast<int>(mx::Layout<256, true>::SMEM_BYTES);
    if (a_rows == 32 && tile_n == 192) return static_cast<int>(mx::Layout<192, false, 32>::SMEM_BYTES);
    if (a_rows == 64 && tile_n == 192) return static_cast<int>(mx::Layout<192, false, 64>::SMEM_BYTES);
    return tile_n == 192 ? static_cast<int>(mx::Layout<192, false>::SMEM_BYTES)
                         : static_cast<int>(mx::Layout<128, false>::SMEM_BYTES);
}

int mx_pair_clusters(bool f32, int num_sms) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * (num_sms / 2)), 1, 1);
    cfg.blockDim = dim3(mx::Layout<256, true>::THREADS, 1, 1);
    cfg.dynamicSmemBytes = mx::Layout<256, true>::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    const cudaError_t e = f32 ? cudaOccupancyMaxActiveClusters(&n, mx::gemm_mx_kernel<true, 256, true>, &cfg)
                              : cudaOccupancyMaxActiveClusters(&n, mx::gemm_mx_kernel<false, 256, true>, &cfg);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return -1;
    }
    return n;
}

} // namespace tpg
