// Instantiations of the small-M weight-streaming kernel (bf16 / fp32 output,
// K split 1 or 2, plain or fused epilogue). The host library reaches them
// through the functions below.
#include "launch.cuh"

namespace tpg {

namespace {
template <bool kOutF32, int kSplit, bool kEpi>
bool set_limit() {
    return cudaFuncSetAttribute(stream::gemm_stream_kernel<kOutF32, kSplit, kEpi>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(stream::SMEM_LIMIT)) == cudaSuccess;
}
template <bool kOutF32, int kSplit, bool kEpi>
cudaError_t launch_one(const StreamLaunch &l) {
    return launch_ex(stream::gemm_stream_kernel<kOutF32, kSplit, kEpi>, l.grid, stream::THREADS, l.smem, kSplit,
                     true, l.stream, *l.a, *l.b, *l.p);
}
template <bool kOutF32, bool kEpi>
cudaError_t launch_split(const StreamLaunch &l) {
    return l.split == 2 ? launch_one<kOutF32, 2, kEpi>(l) : launch_one<kOutF32, 1, kEpi>(l);
}
} // namespace

cudaError_t stream_launch(const StreamLaunch &l) {
    if (l.fused) return l.f32 ? launch_split<true, true>(l) : launch_split<false, true>(l);
    return l.f32 ? launch_split<true, false>(l) : launch_split<false, false>(l);
}

bool stream_set_limits() {
    bool ok = set_limit<false, 1, false>();
    ok = set_limit<true, 1, false>() && ok;
    ok = set_limit<false, 2, false>() && ok;
    ok = set_limit<true, 2, false>() && ok;
    ok = set_limit<false, 1, true>() && ok;
    ok = set_limit<true, 1, true>() && ok;
    ok = set_limit<false, 2, true>() && ok;
    ok = set_limit<true, 2, true>() && ok;
    return ok;
}

int stream_split_clusters(bool f32, int num_sms, int smem) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (num_sms / 2), 1, 1);
    cfg.blockDim = dim3(stream::THREADS, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    const cudaError_t e =
        f32 ? cudaOccupancyMaxActiveClusters(&n, stream::gemm_stream_kernel<true, 2, false>, &cfg)
            : cudaOccupancyMaxActiveClusters(&n, stream::gemm_stream_kernel<false, 2, false>, &cfg);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return -1;
    }
    return n;
}

} // namespace tpg
