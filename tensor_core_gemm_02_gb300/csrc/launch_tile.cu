// launch_tile.cu -- instantiations and launcher of the tile kernel: 128 x BN
// tiles on single CTAs (alone, or in clusters of 4 or 8 sharing A by
// multicast), or 256 x (NSUB * BN) tiles on CTA pairs (clusters of two, or of
// four: two pairs sharing A by multicast).
#include <cuda_runtime.h>

#include <mutex>

#include "kernel_tile.cuh"
#include "launch.h"

namespace tcg {

namespace {

// attr must hold two entries
template <int BN, int STAGES, bool PAIR, int NSUB, int MC>
void fill_config(cudaLaunchConfig_t &cfg, cudaLaunchAttribute *attr, int grid, cudaStream_t stream)
{
    using Cfg = TileCfg<BN, STAGES, PAIR, NSUB, MC>;
    cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(Cfg::THREADS, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_ALLOC;
    cfg.stream = stream;
    int n = 0;
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = TCG_PDL;
    ++n;
    if (Cfg::CLUSTER > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = Cfg::CLUSTER;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
}

template <int BN, int STAGES, bool PAIR, int NSUB, int MC>
cudaError_t launch_impl(const GemmMaps &maps, const GemmArgs &args, int grid, cudaStream_t stream)
{
    using Cfg = TileCfg<BN, STAGES, PAIR, NSUB, MC>;
    auto kfn = tile_gemm_kernel<BN, STAGES, PAIR, NSUB, MC>;
    cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(Cfg::SMEM_ALLOC));
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    fill_config<BN, STAGES, PAIR, NSUB, MC>(cfg, attr, grid, stream);
    return cudaLaunchKernelEx(&cfg, kfn, maps.a, maps.b, maps.c, maps.d, args);
}

// How many clusters of this form can be resident at once on the current device
// (SMs that cannot be grouped within their GPC stay idle).  Cached per device.
template <int BN, int STAGES, bool PAIR, int NSUB, int MC>
int max_clusters_impl()
{
    using Cfg = TileCfg<BN, STAGES, PAIR, NSUB, MC>;
    static std::mutex mu;
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (cached[dev] > 0)
        return cached[dev];
    auto kfn = tile_gemm_kernel<BN, STAGES, PAIR, NSUB, MC>;
    if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(Cfg::SMEM_ALLOC)) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    fill_config<BN, STAGES, PAIR, NSUB, MC>(cfg, attr, Cfg::CLUSTER, nullptr);
    cfg.attrs = attr + 1;  // the cluster shape only (the dependent-launch flag is not a query input)
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kfn, &cfg) != cudaSuccess)
        return 0;
    cached[dev] = clusters;
    return clusters;
}

}  // namespace

int tile_stages(int bn, bool pair, int nsub, int mc)
{
    if (pair)
        return (bn != 256 || (mc != 1 && mc != 2 && mc != 4) || (mc == 4 && nsub != 2))
                   ? 0 : (nsub == 2 ? 4 : 6);
    if (nsub != 1)
        return 0;
    if (mc == 4)
        return bn == 256 ? 4 : (bn == 64 ? 8 : 0);
    if (mc == 8)
        return bn == 256 ? 4 : 0;
    if (mc != 1)
        return 0;
    switch (bn) {
    case 256: return 4;
    case 128: return 6;
    case 64: return 8;
    default: return 0;
    }
}

int tile_max_clusters(int bn, bool pair, int nsub, int mc)
{
    if (pair && bn == 256 && mc == 1)
        return nsub == 2 ? max_clusters_impl<256, 4, true, 2, 1>()
                         : max_clusters_impl<256, 6, true, 1, 1>();
    if (pair && bn == 256 && mc == 2)
        return nsub == 2 ? max_clusters_impl<256, 4, true, 2, 2>()
                         : max_clusters_impl<256, 6, true, 1, 2>();
    if (pair && bn == 256 && mc == 4 && nsub == 2)
        return max_clusters_impl<256, 4, true, 2, 4>();
    if (!pair && nsub == 1 && mc == 4) {
        if (bn == 256)
            return max_clusters_impl<256, 4, false, 1, 4>();
        if (bn == 64)
            return max_clusters_impl<64, 8, false, 1, 4>();
    }
    if (!pair && nsub == 1 && mc == 8 && bn == 256)
        return max_clusters_impl<256, 4, false, 1, 8>();
    return 0;
}

cudaError_t launch_tile(int bn, bool pair, int nsub, int mc, const GemmMaps &maps,
                        const GemmArgs &args, int grid, cudaStream_t stream)
{
    if (pair) {
        if (bn != 256 || (mc != 1 && mc != 2 && mc != 4) || (mc == 4 && nsub != 2))
            return cudaErrorInvalidValue;
        if (mc == 4)
            return launch_impl<256, 4, true, 2, 4>(maps, args, grid, stream);
        if (mc == 2)
            return nsub == 2 ? launch_impl<256, 4, true, 2, 2>(maps, args, grid, stream)
                             : launch_impl<256, 6, true, 1, 2>(maps, args, grid, stream);
        return nsub == 2 ? launch_impl<256, 4, true, 2, 1>(maps, args, grid, stream)
                         : launch_impl<256, 6, true, 1, 1>(maps, args, grid, stream);
    }
    if (nsub != 1)
        return cudaErrorInvalidValue;
    if (mc == 4) {
        if (bn == 256)
            return launch_impl<256, 4, false, 1, 4>(maps, args, grid, stream);
        if (bn == 64)
            return launch_impl<64, 8, false, 1, 4>(maps, args, grid, stream);
        return cudaErrorInvalidValue;
    }
    if (mc == 8)
        return bn == 256 ? launch_impl<256, 4, false, 1, 8>(maps, args, grid, stream)
                         : cudaErrorInvalidValue;
    if (mc != 1)
        return cudaErrorInvalidValue;
    switch (bn) {
    case 256: return launch_impl<256, 4, false, 1, 1>(maps, args, grid, stream);
    case 128: return launch_impl<128, 6, false, 1, 1>(maps, args, grid, stream);
    case 64: return launch_impl<64, 8, false, 1, 1>(maps, args, grid, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace tcg
