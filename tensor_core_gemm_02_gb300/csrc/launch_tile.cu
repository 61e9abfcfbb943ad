// launch_tile.cu -- the tile kernel's plain-epilogue instantiations, its
// per-form ring depths and co-residency, and the launch dispatch over
// epilogue modes (the other modes' kernels live in launch_tile_{scatter,
// reduce,seed}.cu).
#include <cuda_runtime.h>

#include <mutex>

#include "launch_tile_impl.cuh"

namespace tcg {

namespace {

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
    auto kfn = tile_gemm_kernel<BN, STAGES, PAIR, NSUB, MC, kModePlain>;
    if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(Cfg::SMEM_ALLOC)) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    tile_fill_config<BN, STAGES, PAIR, NSUB, MC>(cfg, attr, Cfg::CLUSTER, nullptr);
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

cudaError_t launch_tile(int mode, int bn, bool pair, int nsub, int mc, const GemmMaps &maps,
                        const GemmArgs &args, int grid, cudaStream_t stream)
{
    switch (mode) {
    case kModePlain: return launch_tile_mode<kModePlain>(bn, pair, nsub, mc, maps, args, grid, stream);
    case kModeScatter:
        return launch_tile_mode<kModeScatter>(bn, pair, nsub, mc, maps, args, grid, stream);
    case kModeReduce:
        return launch_tile_mode<kModeReduce>(bn, pair, nsub, mc, maps, args, grid, stream);
    case kModeSeed: return launch_tile_mode<kModeSeed>(bn, pair, nsub, mc, maps, args, grid, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace tcg
