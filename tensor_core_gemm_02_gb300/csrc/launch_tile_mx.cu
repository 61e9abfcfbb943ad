// launch_tile_mx.cu -- the tile kernel's instantiations for FP4 E2M1 operands
// with block scales (a translation unit of its own, compiled in parallel).
// Ring depths: as many stages of codes, scale rows and rearranged scale tiles
// as fit beside the epilogue buffers: single CTAs 3 (256-wide tiles) or 5
// (128-wide), CTA pairs (256 x 256 tiles, each CTA loading half of B's rows) 5.
#include <mutex>

#include "launch_tile_impl.cuh"

namespace tcg {

int tile_mx_stages(int mx, int bn, bool pair)
{
    if (mx != 1 && mx != 2)
        return 0;
    if (pair)
        return bn == 256 ? 5 : 0;
    return bn == 256 ? 3 : (bn == 128 ? 5 : 0);
}

int tile_mx_kstage(int mx)
{
    return mx == 1 ? TileCfg<256, 3, false, 1, 1, 1>::BK : TileCfg<256, 3, false, 1, 1, 2>::BK;
}

namespace {

// CTA pairs of the FP4 pair form that can be resident at once (cached per device).
template <int MX>
int max_pairs_impl()
{
    using Cfg = TileCfg<256, 5, true, 1, 1, MX>;
    static std::mutex mu;
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (cached[dev] > 0)
        return cached[dev];
    auto kfn = tile_gemm_kernel<256, 5, true, 1, 1, kModePlain, MX>;
    if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(Cfg::SMEM_ALLOC)) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    tile_fill_config<256, 5, true, 1, 1, MX>(cfg, attr, Cfg::CLUSTER, nullptr);
    cfg.attrs = attr + 1;  // the cluster shape only
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kfn, &cfg) != cudaSuccess)
        return 0;
    cached[dev] = clusters;
    return clusters;
}

}  // namespace

int tile_mx_max_pairs(int mx)
{
    return mx == 1 ? max_pairs_impl<1>() : (mx == 2 ? max_pairs_impl<2>() : 0);
}

cudaError_t launch_tile_mx(int mx, int bn, bool pair, const GemmMaps &maps, const GemmArgs &args,
                           int grid, cudaStream_t stream)
{
    if (pair) {
        if (bn != 256)
            return cudaErrorInvalidValue;
        if (mx == 1)
            return tile_launch_impl<256, 5, true, 1, 1, kModePlain, 1>(maps, args, grid, stream);
        if (mx == 2)
            return tile_launch_impl<256, 5, true, 1, 1, kModePlain, 2>(maps, args, grid, stream);
        return cudaErrorInvalidValue;
    }
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
