// Instantiations of the block-scaled (MX) GEMM kernel: tiles 128 or 192
// columns wide, bf16 or fp32 output. The host library reaches them through
// mx_launch and mx_set_limits (launch.cuh).
#include "launch.cuh"

namespace tpg {

namespace {
template <bool kOutF32, int kBN>
bool set_limit() {
    return cudaFuncSetAttribute(mx::gemm_mx_kernel<kOutF32, kBN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(mx::Layout<kBN>::SMEM_BYTES)) == cudaSuccess;
}
template <bool kOutF32, int kBN>
cudaError_t launch_one(const MxLaunch &l) {
    return launch_ex(mx::gemm_mx_kernel<kOutF32, kBN>, l.grid, mx::THREADS, static_cast<int>(mx::Layout<kBN>::SMEM_BYTES),
                     1, true, l.stream, *l.a, *l.b, *l.c, *l.d, *l.p);
}
} // namespace

cudaError_t mx_launch(const MxLaunch &l) {
    if (l.tile_n == 192) return l.f32 ? launch_one<true, 192>(l) : launch_one<false, 192>(l);
    if (l.tile_n == 128) return l.f32 ? launch_one<true, 128>(l) : launch_one<false, 128>(l);
    return cudaErrorInvalidValue;
}

bool mx_set_limits() {
    bool ok = set_limit<false, 128>();
    ok = set_limit<true, 128>() && ok;
    ok = set_limit<false, 192>() && ok;
    ok = set_limit<true, 192>() && ok;
    return ok;
}

int mx_smem_bytes(int tile_n) {
    return tile_n == 192 ? static_cast<int>(mx::Layout<192>::SMEM_BYTES) : static_cast<int>(mx::Layout<128>::SMEM_BYTES);
}

} // namespace tpg
