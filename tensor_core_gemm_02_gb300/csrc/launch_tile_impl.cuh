// launch_tile_impl.cuh -- launch helpers and the form dispatch of the tile
// kernel, for one epilogue mode.  Each mode's kernels are instantiated in a
// translation unit of their own (launch_tile*.cu), compiled in parallel.
//
// Forms: 128 x BN tiles on single CTAs (alone, or in clusters of 4 or 8 sharing
// A by multicast), or 256 x (NSUB * BN) tiles on CTA pairs (clusters of two, or
// two / four pairs sharing A by multicast).
#pragma once

#include <cuda_runtime.h>

#include "kernel_tile.cuh"
#include "launch.h"

namespace tcg {

// attr must hold two entries
template <int BN, int STAGES, bool PAIR, int NSUB, int MC, int MX = 0>
inline void tile_fill_config(cudaLaunchConfig_t &cfg, cudaLaunchAttribute *attr, int grid,
                             cudaStream_t stream)
{
    using Cfg = TileCfg<BN, STAGES, PAIR, NSUB, MC, MX>;
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

template <int BN, int STAGES, bool PAIR, int NSUB, int MC, int MODE, int MX = 0>
cudaError_t tile_launch_impl(const GemmMaps &maps, const GemmArgs &args, int grid,
                             cudaStream_t stream)
{
    using Cfg = TileCfg<BN, STAGES, PAIR, NSUB, MC, MX>;
    auto kfn = tile_gemm_kernel<BN, STAGES, PAIR, NSUB, MC, MODE, MX>;
    cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(Cfg::SMEM_ALLOC));
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    tile_fill_config<BN, STAGES, PAIR, NSUB, MC, MX>(cfg, attr, grid, stream);
    return cudaLaunchKernelEx(&cfg, kfn, maps.a, maps.b, maps.c, maps.d, maps.sfa, maps.sfb, args);
}

// Every form of the tile kernel, for epilogue mode MODE.
template <int MODE>
cudaError_t launch_tile_mode(int bn, bool pair, int nsub, int mc, const GemmMaps &maps,
                             const GemmArgs &args, int grid, cudaStream_t stream)
{
    if (pair) {
        if (bn != 256)
            return cudaErrorInvalidValue;
        if (mc == 4)
            return nsub == 2 ? tile_launch_impl<256, 4, true, 2, 4, MODE>(maps, args, grid, stream)
                             : cudaErrorInvalidValue;
        if (mc == 2)
            return nsub == 2 ? tile_launch_impl<256, 4, true, 2, 2, MODE>(maps, args, grid, stream)
                             : tile_launch_impl<256, 6, true, 1, 2, MODE>(maps, args, grid, stream);
        if (mc != 1)
            return cudaErrorInvalidValue;
        return nsub == 2 ? tile_launch_impl<256, 4, true, 2, 1, MODE>(maps, args, grid, stream)
                         : tile_launch_impl<256, 6, true, 1, 1, MODE>(maps, args, grid, stream);
    }
    if (nsub != 1)
        return cudaErrorInvalidValue;
    if (mc == 4) {
        if (bn == 256)
            return tile_launch_impl<256, 4, false, 1, 4, MODE>(maps, args, grid, stream);
        if (bn == 64)
            return tile_launch_impl<64, 8, false, 1, 4, MODE>(maps, args, grid, stream);
        return cudaErrorInvalidValue;
    }
    if (mc == 8)
        return bn == 256 ? tile_launch_impl<256, 4, false, 1, 8, MODE>(maps, args, grid, stream)
                         : cudaErrorInvalidValue;
    if (mc != 1)
        return cudaErrorInvalidValue;
    switch (bn) {
    case 256: return tile_launch_impl<256, 4, false, 1, 1, MODE>(maps, args, grid, stream);
    case 128: return tile_launch_impl<128, 6, false, 1, 1, MODE>(maps, args, grid, stream);
    case 64: return tile_launch_impl<64, 8, false, 1, 1, MODE>(maps, args, grid, stream);
    default: return cudaErrorInvalidValue;
    }
}

// (defined, one mode each, in launch_tile.cu and launch_tile_{scatter,reduce,seed}.cu)
extern template cudaError_t launch_tile_mode<kModeScatter>(int, bool, int, int, const GemmMaps &,
                                                           const GemmArgs &, int, cudaStream_t);
extern template cudaError_t launch_tile_mode<kModeReduce>(int, bool, int, int, const GemmMaps &,
                                                          const GemmArgs &, int, cudaStream_t);
extern template cudaError_t launch_tile_mode<kModeSeed>(int, bool, int, int, const GemmMaps &,
                                                        const GemmArgs &, int, cudaStream_t);

}  // namespace tcg
