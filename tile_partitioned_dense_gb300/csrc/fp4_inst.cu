// Instantiations of the block-scaled GEMM kernel for FP4 elements, one format
// per compilation (TPG_FP4 = 1: NVFP4, E4M3 scales per 16 elements; 2: MXFP4,
// E8M0 scales per 32): 256 x 256 and 256 x 192 tiles on CTA pairs, 1-CTA
// 128 x 192 tiles (with 128-, 64- or 32-row A boxes) and 128 x 128 ones, bf16
// or fp32 output. The host library
// reaches them through the functions below (launch.cuh).
#include "launch.cuh"

#ifndef TPG_FP4
#error "compile with -DTPG_FP4=<1 (NVFP4) or 2 (MXFP4)>"
#endif
#define TPG_CAT2(a, b) a##b
#define TPG_CAT(a, b) TPG_CAT2(a, b)
#if TPG_FP4 == 1
#define TPG_NAME(base) TPG_CAT(base, nv)
#else
#define TPG_NAME(base) TPG_CAT(base, mx)
#endif

namespace tpg {

namespace {
constexpr int kFmt = TPG_FP4 == 1 ? mx::kFmtNvf4 : mx::kFmtMxf4;

template <bool kOutF32, int kBN, bool kPair, int kARows = 128>
bool set_limit() {
    return cudaFuncSetAttribute(mx::gemm_mx_kernel<kOutF32, kBN, kPair, kARows, kFmt>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(mx::Layout<kBN, kPair, kARows, kFmt>::SMEM_BYTES)) == cudaSuccess;
}
template <bool kOutF32, int kBN, bool kPair, int kARows = 128>
cudaError_t launch_one(const MxLaunch &l) {
    return launch_ex(mx::gemm_mx_kernel<kOutF32, kBN, kPair, kARows, kFmt>, l.grid,
                     mx::Layout<kBN, kPair, kARows, kFmt>::THREADS,
                     static_cast<int>(mx::Layout<kBN, kPair, kARows, kFmt>::SMEM_BYTES), kPair ? 2 : 1, true,
                     l.stream, *l.a, *l.b, *l.sa, *l.sb, *l.c, *l.d, *l.p);
}
} // namespace

cudaError_t TPG_NAME(fp4_launch_)(const MxLaunch &l) {
    if (l.pair) {
        if (l.grid % 2 != 0) return cudaErrorInvalidValue;
        if (l.tile_n == 256) return l.f32 ? launch_one<true, 256, true>(l) : launch_one<false, 256, true>(l);
        if (l.tile_n == 192) return l.f32 ? launch_one<true, 192, true>(l) : launch_one<false, 192, true>(l);
        return cudaErrorInvalidValue;
    }
    if (l.tile_n == 128) return l.f32 ? launch_one<true, 128, false>(l) : launch_one<false, 128, false>(l);
    if (l.tile_n != 192) return cudaErrorInvalidValue;
    if (l.a_rows == 32) return l.f32 ? launch_one<true, 192, false, 32>(l) : launch_one<false, 192, false, 32>(l);
    if (l.a_rows == 64) return l.f32 ? launch_one<true, 192, false, 64>(l) : launch_one<false, 192, false, 64>(l);
    return l.f32 ? launch_one<true, 192, false>(l) : launch_one<false, 192, false>(l);
}

bool TPG_NAME(fp4_set_limits_)() {
    bool ok = set_limit<false, 128, false>();
    ok = set_limit<true, 128, false>() && ok;
    ok = set_limit<false, 192, false>() && ok;
    ok = set_limit<true, 192, false>() && ok;
    ok = set_limit<false, 192, false, 64>() && ok;
    ok = set_limit<true, 192, false, 64>() && ok;
    ok = set_limit<false, 192, false, 32>() && ok;
    ok = set_limit<true, 192, false, 32>() && ok;
    ok = set_limit<false, 192, true>() && ok;
    ok = set_limit<true, 192, true>() && ok;
    ok = set_limit<false, 256, true>() && ok;
    ok = set_limit<true, 256, true>() && ok;
    return ok;
}

int TPG_NAME(fp4_smem_bytes_)(int tile_n, bool pair, int a_rows) {
    if (pair)
        return tile_n == 256 ? static_cast<int>(mx::Layout<256, true, 128, kFmt>::SMEM_BYTES)
                             : static_cast<int>(mx::Layout<192, true, 128, kFmt>::SMEM_BYTES);
    if (tile_n == 128) return static_cast<int>(mx::Layout<128, false, 128, kFmt>::SMEM_BYTES);
    if (a_rows == 32) return static_cast<int>(mx::Layout<192, false, 32, kFmt>::SMEM_BYTES);
    if (a_rows == 64) return static_cast<int>(mx::Layout<192, false, 64, kFmt>::SMEM_BYTES);
    return static_cast<int>(mx::Layout<192, false, 128, kFmt>::SMEM_BYTES);
}

int TPG_NAME(fp4_pair_clusters_)(bool f32, int num_sms) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * (num_sms / 2)), 1, 1);
    cfg.blockDim = dim3(mx::Layout<256, true, 128, kFmt>::THREADS, 1, 1);
    cfg.dynamicSmemBytes = mx::Layout<256, true, 128, kFmt>::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    const cudaError_t e =
        f32 ? cudaOccupancyMaxActiveClusters(&n, mx::gemm_mx_kernel<true, 256, true, 128, kFmt>, &cfg)
            : cudaOccupancyMaxActiveClusters(&n, mx::gemm_mx_kernel<false, 256, true, 128, kFmt>, &cfg);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return -1;
    }
    return n;
}

} // namespace tpg
