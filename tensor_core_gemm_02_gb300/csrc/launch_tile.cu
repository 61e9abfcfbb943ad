// launch_tile.cu -- instantiations and launcher of the tile kernel: 128 x BN
// tiles on single CTAs, or 256 x BN tiles on CTA pairs (cluster of two).
#include <cuda_runtime.h>

#include <mutex>

#include "kernel_tile.cuh"
#include "launch.h"

namespace tcg {

namespace {

template <int BN, int STAGES, bool PAIR, int NSUB>
cudaError_t launch_tile_impl(const GemmMaps &maps, const GemmArgs &args, int grid,
                             cudaStream_t stream)
{
    using Cfg = TileCfg<BN, STAGES, PAIR, NSUB>;
    auto kfn = tile_gemm_kernel<BN, STAGES, PAIR, NSUB>;
    cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(Cfg::SMEM_ALLOC));
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(Cfg::THREADS, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_ALLOC;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (PAIR) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kfn, maps.a, maps.b, maps.c, maps.d, args);
}

// How many CTA pairs of the pair kernel can be resident at once on the current
// device (SMs that cannot be paired within their GPC stay idle).
template <int BN, int STAGES, int NSUB>
int max_pairs_impl()
{
    using Cfg = TileCfg<BN, STAGES, true, NSUB>;
    static std::mutex mu;
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (cached[dev] > 0)
        return cached[dev];
    auto kfn = tile_gemm_kernel<BN, STAGES, true, NSUB>;
    if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(Cfg::SMEM_ALLOC)) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(Cfg::THREADS, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_ALLOC;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kfn, &cfg) != cudaSuccess)
        return 0;
    cached[dev] = clusters;
    return clusters;
}

}  // namespace

int tile_stages(int bn, bool pair, int nsub)
{
    if (pair)
        return bn != 256 ? 0 : (nsub == 2 ? 4 : 6);
    if (nsub != 1)
        return 0;
    switch (bn) {
    case 256: return 4;
    case 128: return 6;
    case 64: return 8;
    default: return 0;
    }
}

int tile_max_pairs(int bn, int nsub)
{
    if (bn != 256)
        return 0;
    return nsub == 2 ? max_pairs_impl<256, 4, 2>() : max_pairs_impl<256, 6, 1>();
}

cudaError_t launch_tile(int bn, bool pair, int nsub, const GemmMaps &maps, const GemmArgs &args,
                        int grid, cudaStream_t stream)
{
    if (pair) {
        if (bn != 256)
            return cudaErrorInvalidValue;
        return nsub == 2 ? launch_tile_impl<256, 4, true, 2>(maps, args, grid, stream)
                         : launch_tile_impl<256, 6, true, 1>(maps, args, grid, stream);
    }
    if (nsub != 1)
        return cudaErrorInvalidValue;
    switch (bn) {
    case 256: return launch_tile_impl<256, 4, false, 1>(maps, args, grid, stream);
    case 128: return launch_tile_impl<128, 6, false, 1>(maps, args, grid, stream);
    case 64: return launch_tile_impl<64, 8, false, 1>(maps, args, grid, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace tcg
