// dequant_fp4.cu -- FP4 E2M1 codes with UE8M0 block scales -> bf16 rows, for
// the M > 64 path of gemm_bf16_e2m1 (which then runs the bf16 tile kernel).
// Memory-bound: 4 bytes of codes and 1/32 byte of scale in for every 16
// bytes of bf16 out.
#include <cuda_runtime.h>

#include "common.cuh"
#include "fp4.cuh"
#include "launch.h"

namespace tcg {

// Thread (row n, scale block b) turns the 32 codes of one UE8M0 block (16
// bytes, one 16-byte load) into 32 bf16 (64 bytes, four 16-byte stores).  A
// block of 256 threads covers 32 rows x 8 scale blocks: the eight threads of
// a row read one 128-byte run of codes and write one 512-byte run of bf16,
// and a warp's scale bytes come from 8 scale rows, 4 bytes each.
__global__ void __launch_bounds__(256)
    dequant_fp4_kernel(const uint8_t *codes, int64_t ldq, const uint8_t *scales, int64_t lds,
                       int32_t N, int32_t K, uint16_t *out, int64_t ldo)
{
    grid_dependency_wait();
    if (threadIdx.x == 0)
        grid_launch_dependents();
    const int32_t n = static_cast<int32_t>(blockIdx.x) * 32 + static_cast<int32_t>(threadIdx.x / 8u);
    const int32_t b = static_cast<int32_t>(blockIdx.y) * 8 + static_cast<int32_t>(threadIdx.x % 8u);
    if (n >= N || b >= K / 32)
        return;
    const uint4 w = *reinterpret_cast<const uint4 *>(codes + static_cast<int64_t>(n) * ldq + 16 * b);
    const uint32_t sc2 = ue8m0_to_bf16x2(scales[static_cast<int64_t>(b) * lds + n]);
    uint4 *dst = reinterpret_cast<uint4 *>(out + static_cast<int64_t>(n) * ldo + 32 * b);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t p[4];
        e2m1x8_to_bf16(ws[i], sc2, p);  // codes 8i .. 8i+7 of the block
        dst[i] = make_uint4(p[0], p[1], p[2], p[3]);
    }
}

cudaError_t launch_dequant_fp4(const uint8_t *codes, int64_t ldq, const uint8_t *scales,
                               int64_t lds, int32_t N, int32_t K, uint16_t *out, int64_t ldo,
                               cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    // rows along x (up to 2^31 - 1 blocks), scale blocks along y (K / 256 of them)
    cfg.gridDim = dim3(static_cast<unsigned>((N + 31) / 32), static_cast<unsigned>((K / 32 + 7) / 8), 1);
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
