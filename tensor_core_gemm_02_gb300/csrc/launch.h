// launch.h -- host-side interface between the C ABI (api.cu) and the kernel
// launchers (launch_*.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace tcg {

struct GemmMaps {
    CUtensorMap a;  // A tiles, or the gather table (box of one row)
    CUtensorMap b;  // B tiles
    CUtensorMap c;  // C boxes (float32), unused when C is not read
    CUtensorMap d;  // D boxes
};

int tile_stages(int bn);
cudaError_t launch_tile(int bn, const GemmMaps &maps, const GemmArgs &args, int grid,
                        cudaStream_t stream);

}  // namespace tcg
