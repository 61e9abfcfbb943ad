// launch_skinny.cu -- instantiations and launcher of the swap-AB stream-K kernel
// (bf16/f16 B, FP4 B with block scales converted into tensor memory, or both
// operands FP4 on the block-scaled MMA).
#include <cuda_runtime.h>

#include "kernel_skinny.cuh"
#include "launch.h"

// K extent of one pipeline stage is 64 * TCG_SKINNY_KBOX elements.
#ifndef TCG_SKINNY_KBOX
#define TCG_SKINNY_KBOX 1
#endif

namespace tcg {

namespace {

template <int MP, bool W4, bool MX = false>
cudaError_t launch_skinny_impl(const GemmMaps &maps, const GemmArgs &args, int grid,
                               cudaStream_t stream)
{
    constexpr int KBOX = W4 ? 4 : (MX ? 1 : TCG_SKINNY_KBOX);
    using Cfg = SkinnyCfg<MP, KBOX, W4, MX>;
    auto kfn = skinny_gemm_kernel<MP, KBOX, W4, MX>;
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
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = TCG_PDL;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kfn, maps.a, maps.b, maps.c, maps.sfa, args);
}

}  // namespace

int skinny_kstage() { return 64 * TCG_SKINNY_KBOX; }
int skinny_w4_kstage() { return SkinnyCfg<16, 4, true>::KSTAGE; }

int skinny_stages(int mp)
{
    switch (mp) {
    case 16: return SkinnyCfg<16, TCG_SKINNY_KBOX>::STAGES;
    case 32: return SkinnyCfg<32, TCG_SKINNY_KBOX>::STAGES;
    case 64: return SkinnyCfg<64, TCG_SKINNY_KBOX>::STAGES;
    default: return 0;
    }
}

cudaError_t launch_skinny(int mp, const GemmMaps &maps, const GemmArgs &args, int grid,
                          cudaStream_t stream)
{
    switch (mp) {
    case 16: return launch_skinny_impl<16, false>(maps, args, grid, stream);
    case 32: return launch_skinny_impl<32, false>(maps, args, grid, stream);
    case 64: return launch_skinny_impl<64, false>(maps, args, grid, stream);
    default: return cudaErrorInvalidValue;
    }
}

int skinny_w4_stages(int mp)
{
    switch (mp) {
    case 16: return SkinnyCfg<16, 4, true>::STAGES;
    case 32: return SkinnyCfg<32, 4, true>::STAGES;
    case 64: return SkinnyCfg<64, 4, true>::STAGES;
    default: return 0;
    }
}

cudaError_t launch_skinny_w4(int mp, const GemmMaps &maps, const GemmArgs &args, int grid,
                             cudaStream_t stream)
{
    switch (mp) {
    case 16: return launch_skinny_impl<16, true>(maps, args, grid, stream);
    case 32: return launch_skinny_impl<32, true>(maps, args, grid, stream);
    case 64: return launch_skinny_impl<64, true>(maps, args, grid, stream);
    default: return cudaErrorInvalidValue;
    }
}

int skinny_mx_kstage() { return SkinnyCfg<16, 1, false, true>::KSTAGE; }

int skinny_mx_stages(int mp)
{
    switch (mp) {
    case 16: return SkinnyCfg<16, 1, false, true>::STAGES;
    case 32: return SkinnyCfg<32, 1, false, true>::STAGES;
    case 64: return SkinnyCfg<64, 1, false, true>::STAGES;
    default: return 0;
    }
}

cudaError_t launch_skinny_mx(int mp, const GemmMaps &maps, const GemmArgs &args, int grid,
                             cudaStream_t stream)
{
    switch (mp) {
    case 16: return launch_skinny_impl<16, false, true>(maps, args, grid, stream);
    case 32: return launch_skinny_impl<32, false, true>(maps, args, grid, stream);
    case 64: return launch_skinny_impl<64, false, true>(maps, args, grid, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace tcg
