// Instantiations of the small-M weight-streaming kernel (bf16 / fp32 output,
// K split 1 to 4, plain or fused epilogue). The host library reaches them
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
    switch (l.split) {
    case 1: return launch_one<kOutF32, 1, kEpi>(l);
    case 2: return launch_one<kOutF32, 2, kEpi>(l);
    case 3: return launch_one<kOutF32, 3, kEpi>(l);
    case 4: return launch_one<kOutF32, 4, kEpi>(l);
    default: return cudaErrorInvalidValue;
    }
}

template <bool kOutF32, bool kEpi>
bool set_limits_all() {
    bool ok = set_limit<kOutF32, 1, kEpi>();
    ok = set_limit<kOutF32, 2, kEpi>() && ok;
    ok = set_limit<kOutF32, 3, kEpi>() && ok;
    ok = set_limit<kOutF32, 4, kEpi>() && ok;
    return ok;
}

template <int kSplit>
int clusters_of(bool f32, const cudaLaunchConfig_t &cfg, int *n) {
    return f32 ? static_cast<int>(cudaOccupancyMaxActiveClusters(n, stream::gemm_stream_kernel<true, kSplit, false>, &cfg))
               : static_cast<int>(cudaOccupancyMaxActiveClusters(n, stream::gemm_stream_kernel<false, kSplit, false>, &cfg));
}
} // namespace

cudaError_t stream_launch(const StreamLaunch &l) {
    if (l.fused) return l.f32 ? launch_split<true, true>(l) : launch_split<false, true>(l);
    return l.f32 ? launch_split<true, false>(l) : launch_split<false, false>(l);
}

bool stream_set_limits() {
    bool ok = set_limits_all<false, false>();
    ok = set_limits_all<true, false>() && ok;
    ok = set_limits_all<false, true>() && ok;
    ok = set_limits_all<true, true>() && ok;
    return ok;
}

int stream_split_clusters(bool f32, int num_sms, int smem, int split) {
    if (split < 2 || split > stream::MAX_SPLIT) return -1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(split * (num_sms / split)), 1, 1);
    cfg.blockDim = dim3(stream::THREADS, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(split);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    const int e = split == 2 ? clusters_of<2>(f32, cfg, &n) : split == 3 ? clusters_of<3>(f32, cfg, &n)
                                                                         : clusters_of<4>(f32, cfg, &n);
    if (e != static_cast<int>(cudaSuccess)) {
        (void)cudaGetLastError();
        return -1;
    }
    return n;
}

} // namespace tpg
