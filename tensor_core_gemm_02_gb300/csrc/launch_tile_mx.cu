// launch_tile_mx.cu -- the tile kernel's instantiations for FP4 E2M1 operands
// with block scales (a translation unit of its own, compiled in parallel).
// Ring depths: as many stages of codes, scale rows and rearranged scale tiles
// as fit beside the epilogue buffers (3 for 256-wide tiles, 5 for 128-wide).
#include "launch_tile_impl.cuh"

namespace tcg {

int tile_mx_stages(int mx, int bn)
{
    if (mx != 1 && mx != 2)
        return 0;
    return bn == 256 ? 3 : (bn == 128 ? 5 : 0);
}

int tile_mx_kstage(int mx)
{
    return mx == 1 ? TileCfg<256, 3, false, 1, 1, 1>::BK : TileCfg<256, 3, false, 1, 1, 2>::BK;
}

cudaError_t launch_tile_mx(int mx, int bn, const GemmMaps &maps, const GemmArgs &args, int grid,
                           cudaStream_t stream)
{
    if (mx == 1) {
        if (bn == 256)
            return tile_launch_impl<256, 3, false, 1, 1, kModePlain, 1>(maps, args, grid, stream);
        if (bn == 128)
            return tile_launch_impl<128, 5, false, 1, 1, kModePlain, 1>(maps, args, grid, stream);
    } else if (mx == 2) {
        if (bn == 256)
            return tile_launch_impl<256, 3, false, 1, 1, kModePlain, 2>(maps, args, grid, stream);
        if (bn == 128)
            return tile_launch_impl<128, 5, false, 1, 1, kModePlain, 2>(maps, args, grid, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace tcg
