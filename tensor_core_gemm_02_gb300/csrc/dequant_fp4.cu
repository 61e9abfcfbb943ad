// dequant_fp4.cu -- FP4 E2M1 codes with UE8M0 block scales -> bf16 rows, for
// the M > 64 path of gemm_bf16_e2m1 (which then runs the bf16 tile kernel).
// Memory-bound: each thread turns 8 codes (4 bytes) into 8 bf16 (16 bytes).
#include <cuda_runtime.h>

#include "common.cuh"
#include "fp4.cuh"
#include "launch.h"

namespace tcg {

__global__ void __launch_bounds__(256)
    dequant_fp4_kernel(const uint8_t *codes, int64_t ldq, const uint8_t *scales, int64_t lds,
                       int32_t N, int32_t K, uint16_t *out, int64_t ldo)
{
    grid_dependency_wait();
    if (threadIdx.x == 0)
        grid_launch_dependents();
    const int32_t groups = K / 8;  // 8 codes per thread
    const int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (g >= static_cast<int64_t>(N) * groups)
        return;
    const int32_t n = static_cast<int32_t>(g / groups);
    const int32_t k0 = static_cast<int32_t>(g - static_cast<int64_t>(n) * groups) * 8;
    const uint32_t w = *reinterpret_cast<const uint32_t *>(codes + n * ldq + k0 / 2);
    const uint32_t sc2 = ue8m0_to_bf16x2(scales[static_cast<int64_t>(k0 / 32) * lds + n]);
    uint4 v;
    e2m1x4_to_bf16(w & 0xFFFFu, sc2, v.x, v.y);
    e2m1x4_to_bf16(w >> 16, sc2, v.z, v.w);
    *reinterpret_cast<uint4 *>(out + n * ldo + k0) = v;
}

cudaError_t launch_dequant_fp4(const uint8_t *codes, int64_t ldq, const uint8_t *scales,
                               int64_t lds, int32_t N, int32_t K, uint16_t *out, int64_t ldo,
                               cudaStream_t stream)
{
    const int64_t threads = static_cast<int64_t>(N) * (K / 8);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((threads + 255) / 256), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = TCG_PDL;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, dequant_fp4_kernel, codes, ldq, scales, lds, N, K, out, ldo);
}

}  // namespace tcg
