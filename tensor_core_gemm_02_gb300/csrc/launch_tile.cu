// launch_tile.cu -- instantiations and launcher of the 128 x BN tile kernel.
#include <cuda_runtime.h>

#include "kernel_tile.cuh"
#include "launch.h"

namespace tcg {

template <int BN, int STAGES>
static cudaError_t launch_tile_impl(const GemmMaps &maps, const GemmArgs &args, int grid,
                                    cudaStream_t stream)
{
    using Cfg = TileCfg<BN, STAGES>;
    auto kfn = tile_gemm_kernel<BN, STAGES>;
    cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(Cfg::SMEM_ALLOC));
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(Cfg::THREADS, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_ALLOC;
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, kfn, maps.a, maps.b, maps.c, maps.d, args);
}

int tile_stages(int bn)
{
    switch (bn) {
    case 256: return 4;
    case 128: return 6;
    case 64: return 8;
    default: return 0;
    }
}

cudaError_t launch_tile(int bn, const GemmMaps &maps, const GemmArgs &args, int grid,
                        cudaStream_t stream)
{
    switch (bn) {
    case 256: return launch_tile_impl<256, 4>(maps, args, grid, stream);
    case 128: return launch_tile_impl<128, 6>(maps, args, grid, stream);
    case 64: return launch_tile_impl<64, 8>(maps, args, grid, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace tcg
