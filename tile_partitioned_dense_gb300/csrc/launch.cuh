// Kernel launch helpers and the interface between the host library
// (tpgemm.cu) and the translation units that instantiate the GEMM kernels
// (tiled_inst.cu, once per fused-epilogue mode, stream_inst.cu, mx_inst.cu and
// fp4_inst.cu, once per FP4 format). Only
// those units name kernel instantiations, so each instantiation is compiled
// once, and the units build in parallel.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "gemm_mx.cuh"
#include "gemm_stream.cuh"
#include "gemm_tiled.cuh"

namespace tpg {

// Launches `kernel`. With pdl, the launch allows programmatic dependent launch:
// the kernel may start its on-chip prologue while the previous kernel in the
// stream finishes, and waits (griddepcontrol.wait) before touching global
// memory; only the GEMM kernels, which do that wait, are launched this way.
// Returns cudaSuccess or the launch error.
template <typename Kernel, typename... Args>
cudaError_t launch_ex(Kernel kernel, int grid, int block, int smem, int cluster, bool pdl, cudaStream_t stream,
                      Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(block), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = static_cast<unsigned>(cluster);
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = n ? attr : nullptr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Fused-epilogue modes of the tiled kernel (its kEpi template argument):
// 0 plain alpha*acc + beta*C; 1 + activation otherwise (bias and aux are
// runtime options inside every fused mode); 5 (tiled::kEpiUnitAlpha) the
// plain epilogue for alpha == 1.
constexpr int kEpiModes = 6;

struct TiledLaunch {
    int grid;
    int smem;
    int cluster; // CTAs per cluster: 2 in pair mode, the K split in 1-CTA mode, else 1
    bool pair;
    bool f32;
    cudaStream_t stream;
    const CUtensorMap *a, *b, *b1, *c, *d; // b: B's 4-D map (or its 3-D one); b1: the 3-D map
    const TiledParams *p;
    const GroupTable *groups; // grouped GEMM only (tiled_launch_g0)
};

struct StreamLaunch {
    int grid;
    int smem;
    int split;
    bool f32;
    bool fused;
    cudaStream_t stream;
    const CUtensorMap *a, *b;
    const StreamParams *p;
};

struct MxLaunch {
    int grid;   // CTAs (twice the pairs in pair mode)
    int tile_n; // 1-CTA tiles: 128 or 192; on pairs 256 (and 192 for FP4)
    bool pair;    // 256-row tiles on CTA pairs
    int a_rows;   // rows of A's box: 128, or 64 / 32 for M <= 64 / 32 on 1-CTA 192-wide tiles
    bool f32;
    cudaStream_t stream;
    const CUtensorMap *a, *b, *sa, *sb, *c, *d;
    const MxParams *p;
};

// mx_inst.cu: the block-scaled (MX) kernel
cudaError_t mx_launch(const MxLaunch &l);
bool mx_set_limits();
int mx_smem_bytes(int tile_n, bool pair, int a_rows);
// co-resident CTA pairs of the MX kernel's pair mode, or -1
int mx_pair_clusters(bool f32, int num_sms);

// fp4_inst.cu, one set per FP4 format: _nv (NVFP4) and _mx (MXFP4)
cudaError_t fp4_launch_nv(const MxLaunch &l);
cudaError_t fp4_launch_mx(const MxLaunch &l);
bool fp4_set_limits_nv();
bool fp4_set_limits_mx();
int fp4_smem_bytes_nv(int tile_n, bool pair, int a_rows);
int fp4_smem_bytes_mx(int tile_n, bool pair, int a_rows);
int fp4_pair_clusters_nv(bool f32, int num_sms);
int fp4_pair_clusters_mx(bool f32, int num_sms);

// tiled_inst.cu, one definition per mode E (compiled with -DTPG_EPI=E).
cudaError_t tiled_launch_e0(const TiledLaunch &l);
cudaError_t tiled_launch_e1(const TiledLaunch &l);
cudaError_t tiled_launch_e2(const TiledLaunch &l);
cudaError_t tiled_launch_e3(const TiledLaunch &l);
cudaError_t tiled_launch_e4(const TiledLaunch &l);
cudaError_t tiled_launch_e5(const TiledLaunch &l);
bool tiled_set_limits_e0();
bool tiled_set_limits_e1();
bool tiled_set_limits_e2();
bool tiled_set_limits_e3();
bool tiled_set_limits_e4();
bool tiled_set_limits_e5();
// grouped GEMM (plain epilogue), from tiled_inst.cu with -DTPG_EPI=0 -DTPG_GROUPED=1
cudaError_t tiled_launch_g0(const TiledLaunch &l);
bool tiled_set_limits_g0();
// co-resident clusters of `cluster` CTAs of the tiled kernel (plain mode; pair
// mode when `pair`, whose clusters are CTA pairs), or -1
int tiled_clusters(bool pair, bool f32, int num_sms, int cluster);

// stream_inst.cu
cudaError_t stream_launch(const StreamLaunch &l);
bool stream_set_limits();
// co-resident clusters of `split` CTAs of the streaming kernel with `smem` bytes each
int stream_split_clusters(bool f32, int num_sms, int smem, int split);

} // namespace tpg
