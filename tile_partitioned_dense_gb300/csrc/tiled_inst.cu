// Instantiations of the tiled GEMM kernel for one fused-epilogue mode, E =
// TPG_EPI (see launch.cuh): the 1-CTA mode (with and without its K split) and
// the CTA-pair mode, bf16 and fp32 output. Compiled once per mode; the host
// library reaches them through the functions below.
#include "launch.cuh"

#ifndef TPG_EPI
#error "compile with -DTPG_EPI=<0..5>"
#endif
#ifndef TPG_GROUPED
#define TPG_GROUPED 0
#endif
#define TPG_CAT2(a, b) a##b
#define TPG_CAT(a, b) TPG_CAT2(a, b)
#if TPG_GROUPED
#define TPG_NAME(base) TPG_CAT(base, g0)
#else
#define TPG_NAME(base) TPG_CAT(base, TPG_CAT(e, TPG_EPI))
#endif

namespace tpg {

namespace {
constexpr bool kGrouped = TPG_GROUPED != 0;

template <bool kOutF32, bool kPair, bool kKsplit = false>
bool set_limit() {
    return cudaFuncSetAttribute(tiled::gemm_tiled_kernel<kOutF32, kPair, TPG_EPI, kGrouped, kKsplit>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(tiled::Layout<kPair>::SMEM_BYTES)) == cudaSuccess;
}
template <bool kOutF32, bool kPair>
cudaError_t launch_one(const TiledLaunch &l) {
    SegArg<kGrouped> seg{};
    if constexpr (kGrouped) {
        if (!l.groups) return cudaErrorInvalidValue;
        seg = *l.groups;
    }
    // pair mode: clusters of two; 1-CTA mode: the K split (1, 2 or 4) is the cluster
    const bool cluster_ok = kPair ? l.cluster == 2
                                  : (l.cluster == 1 || l.cluster == 2 || l.cluster == 4) && l.cluster == l.p->ksplit;
    if (!cluster_ok) return cudaErrorInvalidValue;
    if constexpr (!kPair && !kGrouped) {
        if (l.cluster > 1)
            return launch_ex(tiled::gemm_tiled_kernel<kOutF32, false, TPG_EPI, false, true>, l.grid, tiled::THREADS,
                             l.smem, l.cluster, true, l.stream, *l.a, *l.b, *l.b1, *l.c, *l.d, *l.p, seg);
    }
    return launch_ex(tiled::gemm_tiled_kernel<kOutF32, kPair, TPG_EPI, kGrouped>, l.grid, tiled::THREADS, l.smem,
                     l.cluster, true, l.stream, *l.a, *l.b, *l.b1, *l.c, *l.d, *l.p, seg);
}
} // namespace

cudaError_t TPG_NAME(tiled_launch_)(const TiledLaunch &l) {
    if (l.pair) return l.f32 ? launch_one<true, true>(l) : launch_one<false, true>(l);
    return l.f32 ? launch_one<true, false>(l) : launch_one<false, false>(l);
}

bool TPG_NAME(tiled_set_limits_)() {
    bool ok = set_limit<false, false>();
    ok = set_limit<true, false>() && ok;
#if !TPG_GROUPED
    ok = set_limit<false, false, true>() && ok;
    ok = set_limit<true, false, true>() && ok;
#endif
    ok = set_limit<false, true>() && ok;
    ok = set_limit<true, true>() && ok;
    return ok;
}

#if TPG_EPI == 0 && !TPG_GROUPED
int tiled_clusters(bool pair, bool f32, int num_sms, int cluster) {
    if (cluster < 1 || (pair && cluster != 2)) return -1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(cluster * (num_sms / cluster)), 1, 1);
    cfg.blockDim = dim3(tiled::THREADS, 1, 1);
    cfg.dynamicSmemBytes = pair ? tiled::Layout<true>::SMEM_BYTES : tiled::Layout<false>::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    cudaError_t e;
    if (pair)
        e = f32 ? cudaOccupancyMaxActiveClusters(&n, tiled::gemm_tiled_kernel<true, true, 0, false>, &cfg)
                : cudaOccupancyMaxActiveClusters(&n, tiled::gemm_tiled_kernel<false, true, 0, false>, &cfg);
    else
        e = f32 ? cudaOccupancyMaxActiveClusters(&n, tiled::gemm_tiled_kernel<true, false, 0, false, true>, &cfg)
                : cudaOccupancyMaxActiveClusters(&n, tiled::gemm_tiled_kernel<false, false, 0, false, true>, &cfg);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return -1;
    }
    return n;
}
#endif

} // namespace tpg
