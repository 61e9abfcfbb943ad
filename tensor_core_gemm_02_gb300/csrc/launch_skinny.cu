// launch_skinny.cu -- instantiations and launcher of the swap-AB stream-K kernel.
#include <cuda_runtime.h>

#include "kernel_skinny.cuh"
#include "launch.h"

namespace tcg {

template <int MP, int STAGES>
static cudaError_t launch_skinny_impl(const GemmMaps &maps, const GemmArgs &args, int grid,
                                      cudaStream_t stream)
{
    using Cfg = SkinnyCfg<MP, STAGES>;
    auto kfn = skinny_gemm_kernel<MP, STAGES>;
    cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(Cfg::SMEM_ALLOC));
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(Cfg::THREADS, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_ALLOC;
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, kfn, maps.a, maps.b, args);
}

int skinny_stages(int mp)
{
    switch (mp) {
    case 16: return 11;
    case 32: return 10;
    case 64: return 8;
    default: return 0;
    }
}

cudaError_t launch_skinny(int mp, const GemmMaps &maps, const GemmArgs &args, int grid,
                          cudaStream_t stream)
{
    switch (mp) {
    case 16: return launch_skinny_impl<16, 11>(maps, args, grid, stream);
    case 32: return launch_skinny_impl<32, 10>(maps, args, grid, stream);
    case 64: return launch_skinny_impl<64, 8>(maps, args, grid, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace tcg
