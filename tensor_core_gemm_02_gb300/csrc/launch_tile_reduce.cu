// launch_tile_reduce.cu -- the tile kernel's instantiations for the reduce epilogue
// mode (a translation unit of its own, so the modes compile in parallel).
#include "launch_tile_impl.cuh"

namespace tcg {

template cudaError_t launch_tile_mode<kModeReduce>(int, bool, int, int, const GemmMaps &, const GemmArgs &,
                                          int, cudaStream_t);

}  // namespace tcg
