// api_e2m1.cu -- gemm_e2m1: both operands FP4 E2M1 with UE8M0 block scales,
// on the tensor cores' block-scaled MMAs (include/tcgemm.h has the contract).
//
// The codes come in by TMA either as plain bytes (two codes per byte; the
// MMA kind::mxf4 reads them packed, at twice the rate of the next form) or
// with the 16U4_ALIGN16B descriptor format, which places every sixteen codes
// in the low eight bytes of a sixteen-byte shared block ("cp.async.bulk.tensor"
// page, section "Interleave and packed FP4": inner dimension a multiple of
// 128, inner box 128, 32-byte aligned origins and strides, the barrier counting
// payload bytes), the image the MMA kind::mxf8f6f4 reads.  The scales are
// loaded as they lie (K/32 rows of M or N bytes), rearranged in shared memory
// and copied into tensor memory, where the MMAs read them.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>

#include "host_internal.h"

// Whether the automatic plan picks CTA pairs for FP4 operands.  Measured
// (8192^3, packed codes): pairs 450 us, single CTAs 291 us -- the pairs' scale
// path (each CTA's scale warp, the peer's arrival at the leader, the copies
// into both CTAs' tensor memory) holds every stage back -- so single CTAs
// (0); pairs stay available to gemm_debug_force_tile.
#ifndef TCG_MX_AUTO_PAIRS
#define TCG_MX_AUTO_PAIRS 0
#endif

namespace tcg {
namespace host {

namespace {

constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

struct E2m1Problem {
    int64_t M, N, K;
    const uint8_t *Aq;
    int64_t ldaq;
    const uint8_t *As;
    int64_t ldas;
    const uint8_t *Bq;
    int64_t ldbq;
    const uint8_t *Bs;
    int64_t ldbs;
    const float *C;
    int64_t ldc;
    void *D;
    int64_t ldd;
    int out;
    float alpha, beta;
    int image;  // 0: packed codes (kind::mxf4); 1: the 16U4_ALIGN16B image (kind::mxf8f6f4)
    cudaStream_t stream;
};

bool aligned32(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

gemm_status validate_e2m1(const E2m1Problem &p, bool *empty)
{
    *empty = false;
    if (p.M < 0 || p.N < 0 || p.K < 0)
        return GEMM_ERR_INVALID_ARG;
    if (p.out != GEMM_OUT_F32 && p.out != GEMM_OUT_BF16 && p.out != GEMM_OUT_F16)
        return GEMM_ERR_INVALID_ARG;
    if (p.image != 0 && p.image != 1)
        return GEMM_ERR_INVALID_ARG;
    if (p.M > kMaxDim || p.N > kMaxDim || p.K > kMaxDim)
        return GEMM_ERR_UNSUPPORTED;
    if (p.K % 32 != 0 || (p.image == 1 && p.K % 128 != 0))
        return GEMM_ERR_UNSUPPORTED;  // whole scale blocks; the 16U4 image: K a multiple of 128
    if (p.M == 0 || p.N == 0) {
        *empty = true;
        return GEMM_OK;
    }
    const bool c_used = p.C != nullptr && p.beta != 0.0f;
    if (!p.D)
        return GEMM_ERR_INVALID_ARG;
    if (p.ldd < p.N || (c_used && p.ldc < p.N))
        return GEMM_ERR_INVALID_ARG;
    if (p.ldd > kMaxDim || p.ldc > kMaxDim)
        return GEMM_ERR_UNSUPPORTED;
    if (p.K > 0) {
        if (!p.Aq || !p.Bq || !p.As || !p.Bs)
            return GEMM_ERR_INVALID_ARG;
        if (p.ldaq < p.K / 2 || p.ldbq < p.K / 2 || p.ldas < p.M || p.ldbs < p.N)
            return GEMM_ERR_INVALID_ARG;
        if (p.ldaq > kMaxDim || p.ldbq > kMaxDim || p.ldas > kMaxDim || p.ldbs > kMaxDim)
            return GEMM_ERR_UNSUPPORTED;
        const int64_t pitch = p.image == 1 ? 32 : 16;
        const bool base_ok = p.image == 1 ? (aligned32(p.Aq) && aligned32(p.Bq))
                                          : (aligned16(p.Aq) && aligned16(p.Bq));
        if (!base_ok || p.ldaq % pitch || p.ldbq % pitch)
            return GEMM_ERR_ALIGNMENT;
    }
    if (c_used && (reinterpret_cast<uintptr_t>(p.C) & 3u))
        return GEMM_ERR_ALIGNMENT;
    if (reinterpret_cast<uintptr_t>(p.D) & static_cast<uintptr_t>(out_size(p.out) - 1))
        return GEMM_ERR_ALIGNMENT;
    const uint64_t d_span = span_bytes(p.M, p.N, p.ldd, out_size(p.out));
    if (p.K > 0 &&
        (overlap(p.D, d_span, p.Aq, span_bytes(p.M, p.K / 2, p.ldaq, 1)) ||
         overlap(p.D, d_span, p.Bq, span_bytes(p.N, p.K / 2, p.ldbq, 1)) ||
         overlap(p.D, d_span, p.As, span_bytes(p.K / 32, p.M, p.ldas, 1)) ||
         overlap(p.D, d_span, p.Bs, span_bytes(p.K / 32, p.N, p.ldbs, 1))))
        return GEMM_ERR_ALIAS;
    if (c_used && overlap(p.D, d_span, p.C, span_bytes(p.M, p.N, p.ldc, 4))) {
        const bool exact_in_place = static_cast<const void *>(p.C) == p.D &&
                                    p.out == GEMM_OUT_F32 && p.ldc == p.ldd;
        if (!exact_in_place)
            return GEMM_ERR_ALIAS;
    }
    return GEMM_OK;
}

// Scales with an unaligned base or a pitch that is not a multiple of 16 bytes
// are first copied into a padded per-stream buffer (TMA needs both).
gemm_status tma_scales(const DeviceInfo *dev, cudaStream_t stream, int use, const uint8_t *s,
                       int64_t ld, int64_t cols, int64_t rows, const uint8_t **out, int64_t *ld_out)
{
    if (aligned16(s) && ld % 16 == 0) {
        *out = s;
        *ld_out = ld;
        return GEMM_OK;
    }
    const int64_t pitch = (cols + 15) / 16 * 16;
    void *buf = nullptr;
    gemm_status st = get_dequant_buffer(dev->index, stream, use, static_cast<size_t>(pitch) * rows, &buf);
    if (st != GEMM_OK)
        return st;
    if (cudaMemcpy2DAsync(buf, pitch, s, ld, cols, rows, cudaMemcpyDeviceToDevice, stream) !=
        cudaSuccess)
        return GEMM_ERR_CUDA;
    *out = static_cast<const uint8_t *>(buf);
    *ld_out = pitch;
    return GEMM_OK;
}

// Few rows of A, packed codes: the swap-AB stream-K skinny kernel with
// block-scaled MMAs (128 rows of B on the MMA's M side, the padded rows of A on
// its N side, the K blocks of all tiles shared out over the SMs).
gemm_status run_e2m1_skinny(const E2m1Problem &p, const gemm_plan &plan, const DeviceInfo *dev)
{
    const int mp = plan.bm;
    GemmMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    const uint8_t *as = nullptr, *bs = nullptr;
    int64_t ldas = 0, ldbs = 0;
    gemm_status st;
    if ((st = tma_scales(dev, p.stream, kBufScalesA, p.As, p.ldas, p.M, p.K / 32, &as, &ldas)) != GEMM_OK ||
        (st = tma_scales(dev, p.stream, kBufScalesB, p.Bs, p.ldbs, p.N, p.K / 32, &bs, &ldbs)) != GEMM_OK)
        return st;
    const uint32_t sf_rows = static_cast<uint32_t>(tcg::skinny_mx_kstage() / 32);
    if (!encode_2d(&maps.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.Aq, p.K / 2, p.M, p.ldaq, 128,
                   static_cast<uint32_t>(mp), CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&maps.b, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.Bq, p.K / 2, p.N, p.ldbq, 128, 128,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&maps.c, CU_TENSOR_MAP_DATA_TYPE_UINT8, bs, p.N, p.K / 32, ldbs, 128, sf_rows,
                   CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_2d(&maps.sfa, CU_TENSOR_MAP_DATA_TYPE_UINT8, as, p.M, p.K / 32, ldas,
                   static_cast<uint32_t>(mp), sf_rows, CU_TENSOR_MAP_SWIZZLE_NONE))
        return GEMM_ERR_CUDA;
    Problem q{};  // (the fields fill_common reads)
    q.M = p.M;
    q.N = p.N;
    q.K = p.K;
    q.C = p.C;
    q.ldc = p.ldc;
    q.D = p.D;
    q.ldd = p.ldd;
    q.out = p.out;
    q.alpha = p.alpha;
    q.beta = p.beta;
    GemmArgs a;
    std::memset(&a, 0, sizeof(a));
    fill_common(a, q, dev);
    a.num_m_blocks = 1;
    a.num_n_blocks = static_cast<int32_t>(plan.tiles);
    a.num_k_blocks = static_cast<int32_t>(ceil_div(p.K, tcg::skinny_mx_kstage()));
    a.num_tiles = static_cast<int32_t>(plan.tiles);
    a.sk_tiles = static_cast<int32_t>(plan.tiles);  // every tile shared block by block
    a.group_m = 1;
    a.splits = plan.splits;
    if (plan.splits > 1) {
        Workspace w;
        const size_t bytes = static_cast<size_t>(plan.tiles) * plan.splits * 128 * mp * sizeof(float);
        if ((st = get_workspace(dev->index, p.stream, bytes, static_cast<size_t>(plan.tiles), &w)) !=
            GEMM_OK)
            return st;
        a.workspace = w.partials;
        a.counters = w.counters;
    }
    const cudaError_t e = tcg::launch_skinny_mx(mp, maps, a, plan.grid, p.stream);
    return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

gemm_status run_e2m1(const E2m1Problem &p)
{
    bool empty = false;
    gemm_status st = validate_e2m1(p, &empty);
    if (st != GEMM_OK || empty)
        return st;
    DeviceInfo *dev = nullptr;
    if ((st = device_info(&dev)) != GEMM_OK)
        return st;
    const gemm_plan plan = e2m1_plan(p.M, p.N, p.K, p.image, dev->sm_count);
    if (plan.kernel == 15)
        return run_e2m1_skinny(p, plan, dev);
    const int mx = (plan.kernel == 11 || plan.kernel == 13) ? 1 : 2;
    const bool pair = plan.kernel >= 13;
    const int bn = plan.bn;
    int grid = plan.grid;
    if (pair) {
        // never more pairs than can be resident together
        const int resident = tcg::tile_max_pairs_or(mx, dev->sm_count / 2);
        const int64_t pairs = plan.tiles < resident ? plan.tiles : resident;
        grid = static_cast<int>(2 * pairs);
    }
    const bool c_used = p.C != nullptr && p.beta != 0.0f;

    GemmMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    const int kstage = tcg::tile_mx_kstage(mx);
    if (p.K > 0) {
        const uint8_t *as = nullptr, *bs = nullptr;
        int64_t ldas = 0, ldbs = 0;
        if ((st = tma_scales(dev, p.stream, kBufScalesA, p.As, p.ldas, p.M, p.K / 32, &as, &ldas)) !=
                GEMM_OK ||
            (st = tma_scales(dev, p.stream, kBufScalesB, p.Bs, p.ldbs, p.N, p.K / 32, &bs, &ldbs)) !=
                GEMM_OK)
            return st;
        // codes: 128-byte rows of 128 (A) or bn (B) rows, 128-byte swizzle; packed
        // codes as bytes (K / 2 per row), the 16U4 image in elements (K per row)
        const CUtensorMapDataType code_t =
            mx == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B;
        const uint64_t inner = mx == 1 ? static_cast<uint64_t>(p.K / 2) : static_cast<uint64_t>(p.K);
        const uint32_t sf_rows = static_cast<uint32_t>(kstage / 32);
        if (!encode_2d(&maps.a, code_t, p.Aq, inner, p.M, p.ldaq, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_2d(&maps.b, code_t, p.Bq, inner, p.N, p.ldbq, 128,
                       static_cast<uint32_t>(pair ? bn / 2 : bn), CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_2d(&maps.sfa, CU_TENSOR_MAP_DATA_TYPE_UINT8, as, p.M, p.K / 32, ldas, 128, sf_rows,
                       CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !encode_2d(&maps.sfb, CU_TENSOR_MAP_DATA_TYPE_UINT8, bs, p.N, p.K / 32, ldbs,
                       static_cast<uint32_t>(bn), sf_rows, CU_TENSOR_MAP_SWIZZLE_NONE))
            return GEMM_ERR_CUDA;
    }
    // C and D: 32 x 32 boxes, as the other tile forms
    const bool c_tma = c_used && aligned16(p.C) && (p.ldc * 4) % 16 == 0;
    const bool d_tma = aligned16(p.D) && (p.ldd * out_size(p.out)) % 16 == 0;
    if (c_tma && !encode_2d(&maps.c, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p.C, p.N, p.M, p.ldc * 4, 32,
                            32, CU_TENSOR_MAP_SWIZZLE_128B))
        return GEMM_ERR_CUDA;
    if (d_tma) {
        const CUtensorMapDataType dt = p.out == GEMM_OUT_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                       : p.out == GEMM_OUT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                                : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
        const CUtensorMapSwizzle sw =
            p.out == GEMM_OUT_F32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
        if (!encode_2d(&maps.d, dt, p.D, p.N, p.M, p.ldd * out_size(p.out), 32, 32, sw))
            return GEMM_ERR_CUDA;
    }

    Problem q{};  // (the fields fill_common reads)
    q.M = p.M;
    q.N = p.N;
    q.K = p.K;
    q.C = p.C;
    q.ldc = p.ldc;
    q.D = p.D;
    q.ldd = p.ldd;
    q.out = p.out;
    q.alpha = p.alpha;
    q.beta = p.beta;
    GemmArgs a;
    std::memset(&a, 0, sizeof(a));
    fill_common(a, q, dev);
    a.num_m_blocks = static_cast<int32_t>(ceil_div(p.M, pair ? 256 : 128));
    a.num_n_blocks = static_cast<int32_t>(ceil_div(p.N, bn));
    a.num_k_blocks = static_cast<int32_t>(ceil_div(p.K, kstage));
    a.num_tiles = a.num_m_blocks * a.num_n_blocks;
    a.group_m = a.num_m_blocks < 16 ? a.num_m_blocks : 16;
    a.splits = 1;
    a.c_tma = c_tma ? 1 : 0;
    a.d_tma = d_tma ? 1 : 0;
    a.d_tail_direct = (p.N * out_size(p.out)) % 16 != 0 ? 1 : 0;
    const cudaError_t e = tcg::launch_tile_mx(mx, bn, pair, maps, a, grid, p.stream);
    return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

}  // namespace

// Forms: M <= 64 with packed codes: the skinny kernel (kernel 15).  Otherwise
// CTA pairs with 256 x 256 tiles (each SM moves 2/3 of the operand bytes
// per MMA that a single CTA with a 128 x 256 tile moves, which FP4 operands,
// four times the MMA rate of 16-bit ones on the same bytes, need) when M > 128
// and there are at least as many pair tiles as half the pairs; otherwise single
// CTAs, 128 x bn with the width that takes fewer waves (cost waves x (bn + 32),
// as for the other single-CTA forms), 256 on a tie.  A forced form applies.
gemm_plan e2m1_plan(int64_t M, int64_t N, int64_t K, int image, int sm_count)
{
    gemm_plan p;
    std::memset(&p, 0, sizeof(p));
    if (M == 0 || N == 0)
        return p;
    int fk = 0, fbn = 0;
    forced_tile(&fk, &fbn);
    // M <= 64 with packed codes (and K > 0): the skinny kernel, unless a tile
    // form is forced; forced (kernel 15) wherever it can run.  Measured
    // (microseconds, skinny / tile, C, fp32 out, graph replay over operand
    // copies): 16 x 4096^2 8.1 / 12.0, 32 x 28672 x 4096 17.3 / 21.7,
    // 33 x 28672 x 4096 20.9 / 23.8, 64 x 28672 x 4096 18.4 / 21.3, 64 x 4096^2
    // 9.9 / 12.2, 48 x 8192^2 14.8 / 19.3, 64 x 2048 x 8192 12.2 / 18.6,
    // 64 x 1024^2 5.3 / 6.7.
    const bool skinny_ok = image == 0 && M <= 64 && K > 0;
    if (skinny_ok && (fk == 15 || !(fk >= 11 && fk <= 14))) {
        const int mp = M <= 16 ? 16 : (M <= 32 ? 32 : 64);
        const int64_t tiles = ceil_div(N, 128);
        const int64_t nkb = ceil_div(K, tcg::skinny_mx_kstage());
        // at least kSkinnyMinBlocks K blocks (of 256 elements) per CTA
        constexpr int64_t kSkinnyMinBlocks = 4;
        const int64_t want = ceil_div(tiles * nkb, kSkinnyMinBlocks);
        const int64_t G = want < sm_count ? want : sm_count;
        p.kernel = 15;
        p.bm = mp;
        p.bn = 128;
        p.stages = tcg::skinny_mx_stages(mp);
        p.tiles = tiles;
        p.splits = tcg::skinny_max_parts(tiles, nkb, G);
        p.grid = static_cast<int32_t>(G);
        return p;
    }
    const int mx = image == 0 ? 1 : 2;
    const int pairs = sm_count / 2;
    bool pair = false;
    int bn = 256;
    if (fk >= 11 && fk <= 14) {
        pair = fk >= 13;
        bn = fbn;
    } else {
        const int64_t pair_tiles = ceil_div(M, 256) * ceil_div(N, 256);
        pair = TCG_MX_AUTO_PAIRS && M > 128 && pairs > 0 && 2 * pair_tiles >= pairs;
        if (!pair) {
            const int64_t w256 = ceil_div(ceil_div(M, 128) * ceil_div(N, 256), sm_count);
            const int64_t w128 = ceil_div(ceil_div(M, 128) * ceil_div(N, 128), sm_count);
            if (w128 * (128 + 32) < w256 * (256 + 32))
                bn = 128;
        }
    }
    p.kernel = (image == 0 ? 11 : 12) + (pair ? 2 : 0);
    p.bm = pair ? 256 : 128;
    p.bn = bn;
    p.stages = tcg::tile_mx_stages(mx, bn, pair);
    p.tiles = ceil_div(M, p.bm) * ceil_div(N, bn);
    p.splits = 1;
    const int64_t sets = pair ? pairs : sm_count;
    p.grid = static_cast<int32_t>((pair ? 2 : 1) * (p.tiles < sets ? p.tiles : sets));
    (void)K;
    return p;
}

}  // namespace host
}  // namespace tcg

extern "C" gemm_status gemm_e2m1(int64_t M, int64_t N, int64_t K, const uint8_t *Aq, int64_t ldaq,
                                 const uint8_t *As, int64_t ldas, const uint8_t *Bq, int64_t ldbq,
                                 const uint8_t *Bs, int64_t ldbs, const float *C, int64_t ldc,
                                 void *D, int64_t ldd, int out, float alpha, float beta, int image,
                                 void *stream)
{
    using namespace tcg::host;
    const E2m1Problem p{M,  N,   K,   Aq,  ldaq, As,    ldas, Bq,    ldbq,  Bs,
                        ldbs, C, ldc, D,   ldd,  out,   alpha, beta, image, static_cast<cudaStream_t>(stream)};
    return run_e2m1(p);
}
