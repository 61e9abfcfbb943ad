// launch_tiny.cu -- launcher of the warp-level tiny-GEMM kernel.
#include <cuda_runtime.h>

#include "kernel_tiny.cuh"
#include "launch.h"

namespace tcg {

int tiny_warps_per_cta() { return kTinyWarps; }

cudaError_t launch_tiny(const void *A, int64_t lda, const void *B, int64_t ldb,
                        const GemmArgs &args, int grid, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(32 * kTinyWarps, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = TCG_PDL;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tiny_gemm_kernel, static_cast<const unsigned short *>(A), lda,
                              static_cast<const unsigned short *>(B), ldb, args);
}

}  // namespace tcg
