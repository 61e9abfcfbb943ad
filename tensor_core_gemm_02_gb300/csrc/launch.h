// launch.h -- host-side interface between the C ABI (api.cu) and the kernel
// launchers (launch_*.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

// Launch with programmatic dependent launch allowed (1) or not (0): a GEMM
// may then start its set-up while the previous kernel in the stream ends.
#ifndef TCG_PDL
#define TCG_PDL 1
#endif
// skinny kernel, FP4 B: whole waves of tiles go to CTAs whole (0: every tile shared)
#ifndef TCG_SKINNY_WHOLE
#define TCG_SKINNY_WHOLE 1
#endif

namespace tcg {

struct GemmMaps {
    CUtensorMap a;    // A tiles, or the gather table (box of one row); FP4: A's codes
    CUtensorMap b;    // B tiles; FP4: B's codes
    CUtensorMap c;    // C boxes (float32), unused when C is not read
    CUtensorMap d;    // D boxes
    CUtensorMap sfa;  // FP4 operands: A's block scales (K/32 rows of M bytes)
    CUtensorMap sfb;  // FP4 operands: B's block scales (K/32 rows of N bytes)
};

// Tile kernel forms: 128 x bn tiles on single CTAs (mc = 1), or on clusters of
// mc = 4 CTAs sharing each A box by multicast; 256 x (nsub * bn) tiles on CTA
// pairs with tcgen05 cta_group::2.  grid counts CTAs.
int tile_stages(int bn, bool pair, int nsub, int mc);
// clusters (pairs, or groups of mc) of a form that can be resident at once on
// the current device; 0 if unknown
int tile_max_clusters(int bn, bool pair, int nsub, int mc);
// mode: 0 plain epilogue, 1 scattered rows, 2 reduce-add into D, 3 seeded
// accumulators (kModePlain ... kModeSeed)
cudaError_t launch_tile(int mode, int bn, bool pair, int nsub, int mc, const GemmMaps &maps,
                        const GemmArgs &args, int grid, cudaStream_t stream);

// The tile kernel with FP4 E2M1 operands and UE8M0 block scales (plain
// epilogue): single CTAs with 128 x bn tiles (bn 128 or 256), or CTA pairs with
// 256 x 256 tiles (pair = true, bn 256).  mx 1: codes packed two per byte,
// kind::mxf4; mx 2: codes in the 16U4_ALIGN16B image, kind::mxf8f6f4.
// maps.a / maps.b: the codes (128-byte boxes of 128 / bn rows -- pairs: bn / 2
// -- with 128-byte swizzle); maps.sfa / maps.sfb: the scales (uint8 boxes of
// 128 / bn columns by K_stage / 32 rows).  tile_mx_kstage: K elements per
// stage; tile_mx_max_pairs: pairs that can be resident at once (0 if unknown).
int tile_mx_stages(int mx, int bn, bool pair);
int tile_mx_kstage(int mx);
int tile_mx_max_pairs(int mx);
inline int tile_max_pairs_or(int mx, int fallback)
{
    const int r = tile_mx_max_pairs(mx);
    return r > 0 ? r : fallback;
}
cudaError_t launch_tile_mx(int mx, int bn, bool pair, const GemmMaps &maps, const GemmArgs &args,
                           int grid, cudaStream_t stream);

// Warp-level tiny-GEMM kernel: one 16 x 8 block of D per warp.
int tiny_warps_per_cta();
cudaError_t launch_tiny(const void *A, int64_t lda, const void *B, int64_t ldb,
                        const GemmArgs &args, int grid, cudaStream_t stream);

int skinny_stages(int mp);
// The same kernel with FP4 B: maps.b = the codes (uint8, 128-byte boxes of
// 128 rows, 128-byte swizzle), maps.c = the block scales (uint8, 128 x 8
// boxes); bf16 A.
int skinny_w4_stages(int mp);
int skinny_w4_kstage();  // K elements per stage (and per stream-K unit) of the FP4 form
// FP4 codes (N rows of K/2 bytes, ldq apart) and scales (K/32 rows of N bytes,
// lds apart) -> bf16 N x K rows, ldo elements apart; K a multiple of 32.
cudaError_t launch_dequant_fp4(const uint8_t *codes, int64_t ldq, const uint8_t *scales,
                               int64_t lds, int32_t N, int32_t K, uint16_t *out, int64_t ldo,
                               cudaStream_t stream);
cudaError_t launch_skinny_w4(int mp, const GemmMaps &maps, const GemmArgs &args, int grid,
                             cudaStream_t stream);
int skinny_kstage();  // K elements per pipeline stage (and per stream-K unit)
// Both operands FP4 (packed codes, UE8M0 scales per 32), M <= 64: maps.a / maps.b
// the codes of A / B (uint8, 128-byte boxes of mp / 128 rows, 128-byte
// swizzle), maps.c / maps.sfa the scales of B / A (uint8 boxes of 128 / mp
// columns by K_stage / 32 rows); block-scaled MMA kind::mxf4.
int skinny_mx_kstage();
int skinny_mx_stages(int mp);
cudaError_t launch_skinny_mx(int mp, const GemmMaps &maps, const GemmArgs &args, int grid,
                             cudaStream_t stream);
cudaError_t launch_skinny(int mp, const GemmMaps &maps, const GemmArgs &args, int grid,
                          cudaStream_t stream);

// Stream-K split of the skinny kernel: the CTA that owns linear k-block x
// when W blocks are shared by G CTAs as [W g / G, W (g+1) / G).
inline int64_t skinny_owner_host(int64_t x, int64_t W, int64_t G) { return ((x + 1) * G - 1) / W; }

// Tiles of the skinny kernel shared block by block when T tiles run on G
// CTAs.  bf16 / f16 B: all of them.  FP4 B: the T mod G left over after
// whole waves (each CTA takes floor(T / G) tiles whole), plus one wave more
// when fewer than G / 4 are left over, so that no tile is cut into more than
// about five parts.  The shared tiles are tiles 0 .. S-1; T - S is always a
// multiple of G.
inline int64_t skinny_sk_tiles(int64_t T, int64_t G, bool w4)
{
    if (!w4 || !TCG_SKINNY_WHOLE)
        return T;
    const int64_t waves = T / G;
    int64_t S = T - waves * G;
    if (S != 0 && waves > 0 && 4 * S < G)
        S += G;
    return S;
}

// Most CTAs that contribute to one shared tile (workspace slots per tile)
// when `tiles` tiles of nkb K blocks are shared by G CTAs.
inline int32_t skinny_max_parts(int64_t tiles, int64_t nkb, int64_t G)
{
    if (tiles == 0)
        return 1;
    const int64_t W = tiles * nkb;
    if (tiles > 65536) {
        // shares are at least W / G blocks long, so a tile of nkb blocks holds at
        // most (nkb - 1) / (W / G) + 1 share boundaries
        const int64_t shortest = W / G;
        return static_cast<int32_t>((nkb - 1) / shortest + 2);
    }
    int64_t most = 1;
    for (int64_t t = 0; t < tiles; ++t) {
        const int64_t parts = skinny_owner_host((t + 1) * nkb - 1, W, G) -
                              skinny_owner_host(t * nkb, W, G) + 1;
        most = parts > most ? parts : most;
    }
    return static_cast<int32_t>(most);
}

}  // namespace tcg
