// kernel_skinny.cuh -- swap-AB stream-K tcgen05 GEMM for M <= 64.
//
// With few rows of A the product is bound by streaming B from HBM.  The
// kernel computes D^T = B * A^T instead: 128 rows of B sit on the MMA's M
// side and the (padded) MP <= 64 rows of A on its N side, so every B byte
// feeds a 128 x MP x 16 MMA.  This relabels operands instead of moving data
// ("mma.sync" page, section "Accumulation, transpose and alpha/beta": a
// transpose is a change of view, not an exchange of values).
//
// Work split (stream-K, FP4 B with whole tiles): of the T 128-row tiles of
// B, the first S (args.sk_tiles) are shared block by block -- their (tile,
// k-block) pairs form one list of W = S nkb and CTA g takes the contiguous
// share [W g / G, W (g+1) / G) -- and the other T - S, a multiple of G, go
// whole, tile S + g + G j to CTA g.  A shared tile touched by several CTAs
// gets one partial sum from each; each writes its partial to the workspace,
// and the last to arrive (an atomic counter per tile) adds them in a fixed
// order, applies the epilogue and resets the counter.  No CTA waits for
// another.  A CTA runs its tail piece first, its whole tiles next and its head
// piece last (FP4 B: both pieces first), so that the hand-ins overlap the
// whole tiles' MMAs and the last piece finishes its tile from registers.
// (bf16 / f16 B shares every tile, S = T: with whole tiles its HBM stream
// measured 10-20% slower, FP4 B, bound by the decode, 3-12% faster.)
//
//   warp 0     producer: per stage, KBOX TMA boxes of B (128 x 64) and of A
//              (MP x 64) at consecutive K, so each row of B is read in
//              KBOX * 128-byte runs (FP4 B: the codes, 128 rows x 128 bytes,
//              and the stage's scale rows)
//   warps 1..I MMA issuers (I = ISSUERS: 4 for MP = 16, 2 for FP4 B and for
//              both operands FP4 with MP = 32 / 64, else 1): tcgen05.mma M=128
//              N=MP K=16 (both FP4: block-scaled, K=64), each issuer into two
//              TMEM accumulators of its own (FP4 B: A operand from TMEM)
//   next 4     epilogue (8 for MP = 64 except FP4 B, two per TMEM lane
//              quarter, 32 columns each): tcgen05.ld (the issuers' partial sums added in
//              order), partial or final fma.rn(alpha, acc, beta*C) with
//              coalesced plain loads/stores (lanes walk along N); with
//              scattered rows, row m of the result lands in row idx[m] of D;
//              in the accumulating form every part is added into D with
//              float32 atomic adds instead (no workspace, no last arriver)
//   the rest   (FP4 B) converters: E2M1 codes and UE8M0 scales to bf16 rows
//              in tensor memory (tcgen05.st), the MMA's A operand; or (both
//              operands FP4, MX) one scale warp: the stage's scale rows of B
//              and A rearranged into the tiles tcgen05.cp copies into tensor
//              memory, where the block-scaled MMA (kind::mxf4) reads them
#pragma once

#include "common.cuh"
#include "fp4.cuh"


// Accumulator buffers of the bf16 / f16 form (at most 512 / MP).
#ifndef TCG_SKINNY_MX_ISSUERS16
#define TCG_SKINNY_MX_ISSUERS16 4
#endif
#ifndef TCG_SKINNY_MX_ISSUERS32
#define TCG_SKINNY_MX_ISSUERS32 2
#endif
#ifndef TCG_SKINNY_BF16_ISSUERS16
#define TCG_SKINNY_BF16_ISSUERS16 4
#endif
#ifndef TCG_SKINNY_NACC
#define TCG_SKINNY_NACC 2
#endif


namespace tcg {

// A tensor-memory allocation: a power of two of at least 32 columns.
__host__ __device__ constexpr uint32_t tmem_cols_for(uint32_t cols)
{
    return cols <= 32u ? 32u : (cols <= 64u ? 64u : (cols <= 128u ? 128u : (cols <= 256u ? 256u : 512u)));
}

template <int MP_, int KBOX_, bool W4_ = false, bool MX_ = false>
struct SkinnyCfg {
    static constexpr int MP = MP_;      // padded rows of A = MMA N
    static constexpr int BN = 128;      // rows of B per tile = MMA M
    // MX: A and B both FP4 E2M1, codes packed two per byte, with UE8M0 scales
    // per 32 elements: a 128-byte box holds 256 elements of a row, and the MMA
    // is the block-scaled kind::mxf4 (K = 64 per instruction)
    static constexpr bool MX = MX_;
    static constexpr int BK = MX ? 256 : 64;  // K of one 128-byte swizzled box
    static constexpr int KBOX = KBOX_;  // boxes per stage: each row of B is read KBOX*128 B at a time
    static constexpr int KSTAGE = BK * KBOX;
    // W4: B arrives as FP4 codes (two per byte) with one UE8M0 scale per 32
    // elements, KBOX = 4 blocks of 64 per stage so each row of codes is read
    // in 128-byte runs (32-byte runs leave HBM mostly idle); converter warps
    // turn the codes into bf16 in tensor memory, where the MMA takes its A
    // operand from (row r of B in TMEM lane r, two elements per column)
    static constexpr bool W4 = W4_;
    static constexpr uint32_t RAW_B = W4 ? BN * BK / 2 * KBOX : 0;  // 128 rows x 128 bytes of codes
    // scale rows (32-element blocks) of a stage: B's 128 columns, (MX) A's MP
    static constexpr int SF_KB = (W4 || MX) ? KSTAGE / 32 : 0;
    static constexpr uint32_t SCALE_B = SF_KB * BN;
    static constexpr uint32_t SCALE_A = MX ? SF_KB * MP : 0;
    // (MX) the stage's scales rearranged for tcgen05.cp 32x128b.warpx4: 512-byte
    // tiles of 128 rows x four 32-element blocks (row l + 32 q, block b at byte
    // 16 l + 4 q + b) -- B's two 128-element chunks, then A's (rows >= MP zero)
    static constexpr int SF_TILES = MX ? 2 * (KSTAGE / 128) : 0;
    static constexpr uint32_t SF_CP = SF_TILES * 512;

    // MMA-issuing warps.  One thread issues a tcgen05.mma about every 117
    // cycles whatever its N, so at N = MP a lone issuer, not the tensor pipe,
    // sets the rate; issuers in separate warps add up (with A in TMEM; A
    // from shared memory saturates its reads first).  FP4 B: issuer e takes
    // the blocks j = e (mod ISSUERS) of every stage; bf16 / f16 B with MP = 16:
    // four issuers, issuer e the K step e of each box (16 x 28672 x 4096:
    // 41.2 -> 39.9 us; for MP = 32 / 64 more issuers measured slower).  Each
    // issuer has accumulators of its own, and the epilogue adds the partial
    // sums in issuer order.
    // Both operands FP4 (MX): a stage is four block-scaled MMAs; issuer e takes
    // MX_PER of them (consecutive, so one 128-element chunk of scales), copying
    // that chunk's scale tiles into TMEM columns of its own.
    static constexpr int ISSUERS =
        W4 ? (MP <= 16 ? 4 : 2)
           : (MX ? (MP <= 16 ? TCG_SKINNY_MX_ISSUERS16 : (MP <= 32 ? TCG_SKINNY_MX_ISSUERS32 : 2))
                 : (MP <= 16 ? TCG_SKINNY_BF16_ISSUERS16 : 1));
    static constexpr int MX_PER = MX ? 4 / ISSUERS : 0;
    // Epilogue warps: four (one per TMEM lane quarter), or eight with MP = 64
    // (bf16 / f16 B and both operands FP4), two per quarter, each finishing 32
    // of the 64 columns, which halves a thread's chain of loads and stores.
    static constexpr int EPI_SPLIT = (!W4 && MP == 64) ? 2 : 1;
    static constexpr int EPI_WARPS = 4 * EPI_SPLIT;
    static constexpr int EPI_WARP0 = 1 + ISSUERS;
    static constexpr int CONV_WARP0 = EPI_WARP0 + EPI_WARPS;  // then the converters
    // Accumulator buffers: the MMA fills one while the epilogue drains the
    // other.  (Four for bf16 B measured the same as two; FP4 B needs the rest
    // of tensor memory for converted weights.)
    static constexpr int NACC = W4 ? 2 : TCG_SKINNY_NACC;
    static constexpr uint32_t ACC_COLS = static_cast<uint32_t>(NACC * ISSUERS * MP);
    static constexpr uint32_t TMEM_COLS = (W4 || MX) ? 512u : tmem_cols_for(ACC_COLS);
    // TMEM columns: accumulator (buffer b, issuer e) at (b ISSUERS + e) MP,
    // then whole-stage converted sets (two elements per column) from the
    // next multiple of 128 to the end of the allocation
    static constexpr uint32_t CSET_COL0 = (ACC_COLS + 127u) / 128u * 128u;
    static constexpr uint32_t CSET_COLS = KSTAGE / 2;
    static constexpr int CSETS = W4 ? static_cast<int>((TMEM_COLS - CSET_COL0) / CSET_COLS) : 0;
    // Converter warps: CONV_PER_Q for each quarter of TMEM lanes (a warp
    // reaches only quarter warp % 4), each taking KBOX / CONV_PER_Q blocks of
    // every stage for its 32 rows.  All of them convert every stage and move
    // through the sets together, so none sits waiting for the MMA while a set
    // is free, and the decode (ALU-bound) keeps the SM busy; two per quarter
    // for MP > 16 (the chunked epilogue's registers, four issuers' worth of
    // TMEM accumulators not fitting; four there measured slower with spills).
    static constexpr int CONV_PER_Q = W4 ? (MP <= 16 ? 4 : 2) : 0;
    static constexpr int CONV_WARPS = 4 * CONV_PER_Q;
    static constexpr int SCALE_WARPS = MX ? 1 : 0;  // (MX) after the epilogue
    static constexpr int THREADS = 32 * CONV_WARP0 + 32 * (CONV_WARPS + SCALE_WARPS);

    static constexpr uint32_t B_BOX = BN * 128;  // 128 rows of one 128-byte box
    static constexpr uint32_t A_BOX = MP * 128;
    static constexpr uint32_t B_BYTES = W4 ? 0 : KBOX * B_BOX;
    static constexpr uint32_t A_BYTES = KBOX * A_BOX;
    static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES + RAW_B + SCALE_B + SCALE_A;  // TMA
    // as many stages as fit in about 200 KB of shared memory (at most 16)
    static constexpr uint32_t RING_BUDGET = 204800u;
    static constexpr uint32_t STAGE_SMEM = STAGE_BYTES + SF_CP;
    static constexpr int STAGES = (RING_BUDGET / STAGE_SMEM) < 16 ? (RING_BUDGET / STAGE_SMEM) : 16;
    static constexpr uint32_t OFF_B = 0;
    static constexpr uint32_t OFF_A = OFF_B + STAGES * B_BYTES;
    static constexpr uint32_t OFF_RAW = OFF_A + STAGES * A_BYTES;
    static constexpr uint32_t OFF_SC = OFF_RAW + STAGES * RAW_B;
    static constexpr uint32_t OFF_SCA = OFF_SC + STAGES * SCALE_B;
    static constexpr uint32_t OFF_SFC = OFF_SCA + STAGES * SCALE_A;
    static constexpr uint32_t OFF_BAR = (OFF_SFC + STAGES * SF_CP + 7u) & ~7u;
    // (MX: one more per stage, the scale warp's hand-over to the MMA thread)
    static constexpr uint32_t NUM_BARS = 2 * STAGES + 2 * NACC + 2 * CSETS + (MX ? STAGES : 0);
    // (MX) scale columns of stage s, issuer e: SF_COL0 + (s ISSUERS + e) 8 (B's
    // chunk, then A's, four columns each)
    static constexpr uint32_t SF_COL0 = ACC_COLS;
    static constexpr uint32_t SF_COLS = MX ? ISSUERS * 8 : 0;  // a stage's
    static constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr uint32_t OFF_ROWS = OFF_MISC + 16;  // MP destination rows (scattered rows)
    static constexpr uint32_t SMEM_BYTES = OFF_ROWS + MP * 4;
    static constexpr uint32_t SMEM_ALLOC = SMEM_BYTES + 1024;

    static_assert(!W4 || KBOX == 4, "W4 stages hold 128-byte runs of codes");
    static_assert(!W4 || (KBOX % CONV_PER_Q == 0 && CSETS >= 2), "converters split a stage's blocks");
    static_assert(W4 ? KBOX % ISSUERS == 0 : (MX ? (ISSUERS == 2 || ISSUERS == 4) : (BK / 16) % ISSUERS == 0),
                  "issuers split a stage's blocks (MX: each within one chunk of scales; bf16 / "
                  "f16 B: each box's K steps)");
    static_assert(OFF_RAW % 1024 == 0 && RAW_B % 128 == 0, "TMA destinations stay aligned");
    static_assert(MP % 16 == 0 && MP >= 16 && MP <= 64, "MMA N for M = 128 is a multiple of 16");
    static_assert((TMEM_COLS & (TMEM_COLS - 1)) == 0, "TMEM allocation is a power of two");
    static_assert(ACC_COLS <= TMEM_COLS && NACC >= 2, "accumulators fit the allocation");
    static_assert(!W4 || CSET_COL0 + CSETS * CSET_COLS <= TMEM_COLS,
                  "accumulators and converted sets fit the allocation");
    static_assert(A_BOX % 1024 == 0 && B_BOX % 1024 == 0, "box images stay 1024-aligned");
    static_assert(STAGES >= 2, "at least double buffering");
    static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
    static_assert(!(W4 && MX) && (!MX || (KBOX == 1 && SF_COL0 + STAGES * SF_COLS <= TMEM_COLS)),
                  "both-FP4 stages: one box per operand, scale tiles in TMEM");
    static_assert(OFF_SFC % 16 == 0 && OFF_SCA % 16 == 0, "scale images 16-byte aligned");
};

// The CTA that owns linear k-block x when W blocks are split over G CTAs as
// [W g / G, W (g+1) / G).
__device__ __forceinline__ int32_t skinny_owner(int64_t x, int64_t W, int64_t G)
{
    return static_cast<int32_t>(((x + 1) * G - 1) / W);
}

// Named barrier 1 among the epilogue's N threads.
template <int N>
__device__ __forceinline__ void epi_bar_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(N) : "memory");
}

// Row of C and D for row m of A: m itself, or (scattered rows) the entry
// that the epilogue staged in shared memory; -1 when nothing is written.
__device__ __forceinline__ int32_t skinny_row(const GemmArgs &a, const int32_t *drow, int m)
{
    if (a.scatter)
        return drow[m];
    return m < a.M ? m : -1;
}

// The epilogue works on chunks of CH rows of A (m0 .. m0 + CH - 1) of one
// column n of D, so its registers do not grow with MP.

// c[m] = C[r][n] for the chunk's rows (0 where nothing is written or C is
// absent).  The loads are left in flight: beta is applied where the values
// are used (skinny_beta_c), so a warp that fetches C early does not stall on it.
//
// One epilogue warp per TMEM lane quarter runs these, so each is a straight
// run of independent loads or stores: the per-call conditions are tested
// once, and row m is a fixed stride from row 0 (scattered rows excepted).
template <int CH>
__device__ __forceinline__ void skinny_load_c(const GemmArgs &a, const int32_t *drow, int32_t n,
                                              int m0, float (&c)[CH])
{
#pragma unroll
    for (int m = 0; m < CH; ++m)
        c[m] = 0.f;
    if (!a.has_c || n >= a.N)
        return;
    if (a.scatter) {
#pragma unroll
        for (int m = 0; m < CH; ++m) {
            const int32_t r = drow[m0 + m];
            if (r >= 0)
                c[m] = a.C[static_cast<int64_t>(r) * a.ldc + n];
        }
        return;
    }
    const float *p = a.C + static_cast<int64_t>(m0) * a.ldc + n;
    const int32_t rows = a.M - m0;  // rows m < rows exist
#pragma unroll
    for (int m = 0; m < CH; ++m)
        if (m < rows)
            c[m] = p[static_cast<int64_t>(m) * a.ldc];
}

// cb[m] = mul.rn(beta, c[m])
template <int CH>
__device__ __forceinline__ void skinny_beta_c(const GemmArgs &a, const float (&c)[CH], float (&cb)[CH])
{
#pragma unroll
    for (int m = 0; m < CH; ++m)
        cb[m] = mul_rn(a.beta, c[m]);
}

// Final values: D[r][n] = fma.rn(alpha, v[m], cb[m]) with r = skinny_row(m)
// (or D = mul.rn(alpha, v[m]) without C).
template <typename T, int CH, typename Cvt>
__device__ __forceinline__ void skinny_store_rows(const GemmArgs &a, const int32_t *drow, int32_t n,
                                                  int m0, const float (&d)[CH], Cvt cvt)
{
    T *D = static_cast<T *>(a.D);
    if (a.scatter) {
#pragma unroll
        for (int m = 0; m < CH; ++m) {
            const int32_t r = drow[m0 + m];
            if (r >= 0)
                D[static_cast<int64_t>(r) * a.ldd + n] = cvt(d[m]);
        }
        return;
    }
    T *p = D + static_cast<int64_t>(m0) * a.ldd + n;
    const int32_t rows = a.M - m0;
#pragma unroll
    for (int m = 0; m < CH; ++m)
        if (m < rows)
            p[static_cast<int64_t>(m) * a.ldd] = cvt(d[m]);
}

template <int CH>
__device__ __forceinline__ void skinny_store(const GemmArgs &a, const int32_t *drow, int32_t n,
                                             int m0, const float (&v)[CH], const float (&cb)[CH])
{
    if (n >= a.N)
        return;
    float d[CH];
    if (a.has_c) {
#pragma unroll
        for (int m = 0; m < CH; ++m)
            d[m] = fma_rn(a.alpha, v[m], cb[m]);
    } else {
#pragma unroll
        for (int m = 0; m < CH; ++m)
            d[m] = mul_rn(a.alpha, v[m]);
    }
    if (a.out_kind == kOutF32)
        skinny_store_rows<float>(a, drow, n, m0, d, [](float x) { return x; });
    else if (a.out_kind == kOutBF16)
        skinny_store_rows<unsigned short>(a, drow, n, m0, d, [](float x) { return f32_to_bf16_rn(x); });
    else
        skinny_store_rows<unsigned short>(a, drow, n, m0, d, [](float x) { return f32_to_f16_rn(x); });
}

// Accumulating form: add mul.rn(alpha, v[m]) into D[r][n] (float32 atomic
// adds, so the parts of a split tile need no workspace and no ordering).
template <int CH>
__device__ __forceinline__ void skinny_add(const GemmArgs &a, const int32_t *drow, int32_t n,
                                           int m0, const float (&v)[CH])
{
    if (n >= a.N)
        return;
    float d[CH];
#pragma unroll
    for (int m = 0; m < CH; ++m)
        d[m] = mul_rn(a.alpha, v[m]);
    float *D = static_cast<float *>(a.D);
    if (a.scatter) {
#pragma unroll
        for (int m = 0; m < CH; ++m) {
            const int32_t r = drow[m0 + m];
            if (r >= 0)
                atomicAdd(D + static_cast<int64_t>(r) * a.ldd + n, d[m]);
        }
        return;
    }
    float *p = D + static_cast<int64_t>(m0) * a.ldd + n;
    const int32_t rows = a.M - m0;
#pragma unroll
    for (int m = 0; m < CH; ++m)
        if (m < rows)
            atomicAdd(p + static_cast<int64_t>(m) * a.ldd, d[m]);
}

template <int MP, int KBOX, bool W4, bool MX = false>
__global__ void __launch_bounds__(SkinnyCfg<MP, KBOX, W4, MX>::THREADS, 1)
    skinny_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmS,
                       const __grid_constant__ CUtensorMap tmSA, const GemmArgs args)
{
    using Cfg = SkinnyCfg<MP, KBOX, W4, MX>;
    constexpr int STAGES = Cfg::STAGES;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);

    const uint32_t warp = __shfl_sync(0xffffffffu, threadIdx.x / 32u, 0);
    const uint32_t lane = threadIdx.x % 32u;

    const uint32_t bar0 = base + Cfg::OFF_BAR;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    constexpr int NACC = Cfg::NACC;
    auto accf_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
    auto acce_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + NACC + b); };
    auto cfull_bar = [&](int c) { return bar0 + 8u * (2 * STAGES + 2 * NACC + c); };  // per converted set
    auto cempty_bar = [&](int c) { return bar0 + 8u * (2 * STAGES + 2 * NACC + Cfg::CSETS + c); };
    // (MX) stage s's scales are rearranged for tcgen05.cp
    auto sfr_bar = [&](int st) { return bar0 + 8u * (2 * STAGES + 2 * NACC + 2 * Cfg::CSETS + st); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + Cfg::OFF_MISC);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(gbase + Cfg::OFF_MISC + 4);
    volatile uint32_t *arrival = reinterpret_cast<volatile uint32_t *>(gbase + Cfg::OFF_MISC + 8);
    // (the last piece's early read of its tile's counter: a slot of its own, as
    // slower epilogue warps may still be reading `arrival` of the piece before)
    volatile uint32_t *seen = reinterpret_cast<volatile uint32_t *>(gbase + Cfg::OFF_MISC + 12);

    const int64_t nkb = args.num_k_blocks;
    const int64_t S = args.sk_tiles;
    const int64_t W = S * nkb;  // shared K blocks
    const int64_t G = gridDim.x;
    const int64_t my_start = W * blockIdx.x / G;
    const int64_t my_end = W * (blockIdx.x + 1) / G;
    const int64_t sk_n = my_end - my_start;
    // whole tiles S + blockIdx.x + G j (T - S is a multiple of G)
    const int64_t n_steps = sk_n + (args.num_tiles - S) / G * nkb;
    // The share [my_start, my_end) is the tail of one tile, whole tiles, and the
    // head of another.  The tail piece goes first.  Where the epilogue can
    // finish a tile from registers (kHeadLast: not FP4 B), the head piece goes
    // last: the next CTA handed in its part of that tile with its own first
    // piece, so this CTA finishes the tile without writing its part, and the
    // tail piece's hand-in (its tile is finished by the previous CTA) overlaps
    // the whole tiles' MMAs.  FP4 B runs both pieces first, then the whole
    // tiles, so that its reductions (through the workspace) do not end the
    // kernel.  Step i (0 <= i < n_steps) is linear K block order(i) (tile
    // order(i) / nkb); pieces stay contiguous.
    const int64_t b1 = (my_start + nkb - 1) / nkb * nkb;  // first tile boundary
    const int64_t b2 = my_end / nkb * nkb;                 // last tile boundary
    const bool crosses = b1 < my_end;
    const int64_t len_a = crosses ? b1 - my_start : sk_n;  // tail piece
    const int64_t len_b = crosses ? my_end - b2 : 0;       // head piece
    constexpr bool kHeadLast = !W4;
    const int64_t ms = kHeadLast ? len_a : len_a + len_b;  // first step of the share's whole tiles
    const int64_t os = sk_n - len_b + (kHeadLast ? 0 : len_b);  // ... of the own tiles
    const int64_t oe = n_steps - (kHeadLast ? len_b : 0);  // end of the own tiles
    const int64_t hs = kHeadLast ? oe : len_a;             // first step of the head piece
    auto order = [&](int64_t i) -> int64_t {
        if (i < len_a)
            return my_start + i;
        if (i >= hs && i < hs + len_b)
            return b2 + (i - hs);
        if (i >= ms && i < os)
            return b1 + (i - ms);
        const int64_t d = i - os;
        return (S + blockIdx.x + G * (d / nkb)) * nkb + d % nkb;
    };
    // end, in steps, of the piece that step i belongs to: the tail piece, the
    // head piece, or a whole tile of nkb steps (those of the share, which
    // start on a tile boundary, and the CTA's own)
    auto piece_end = [&](int64_t i) -> int64_t {
        if (i < len_a)
            return len_a;
        if (i >= hs && i < hs + len_b)
            return hs + len_b;
        const int64_t w0 = i < os ? ms : os;
        return w0 + ((i - w0) / nkb + 1) * nkb;
    };

    // (tile, K block) of successive steps without divisions: one thread's
    // 64-bit divisions cost hundreds of cycles, and the producer's time per
    // step bounds the stream.  The divisions of order() are taken only where
    // a run of consecutive K blocks starts (the tail piece, the share's whole
    // tiles, the own tiles, the head piece); inside the own tiles the next
    // tile is G further on.
    struct Cursor {
        int64_t i;
        int32_t t, kb;
    };
    // (by value: a cursor whose address is taken lives on the stack)
    auto cursor_at = [&](int64_t i) -> Cursor {
        const int64_t q = order(i);
        const int32_t t = static_cast<int32_t>(q / nkb);
        return Cursor{i, t, static_cast<int32_t>(q - static_cast<int64_t>(t) * nkb)};
    };
    auto cursor_next = [&](Cursor c) -> Cursor {
        ++c.i;
        if (c.i == len_a || c.i == ms || c.i == os || c.i == oe || c.i == hs || c.i == hs + len_b)
            return c.i < n_steps ? cursor_at(c.i) : c;
        if (++c.kb == nkb) {
            c.kb = 0;
            c.t += c.i > os && c.i < oe ? static_cast<int32_t>(G) : 1;
        }
        return c;
    };

    // stage st <- B and A boxes of K block kb of tile t, counted on full_bar(st)
    auto issue_stage = [&](int st, int32_t t, int32_t kb, uint32_t extra) {
        mbar_arrive_expect_tx(full_bar(st), Cfg::STAGE_BYTES + extra);
        if constexpr (MX) {
            // one 128-byte box of codes of B (128 rows) and of A (MP rows), x in
            // bytes; the stage's scale rows of B (128 columns) and of A (MP)
            tma_load_2d(base + Cfg::OFF_B + st * Cfg::B_BYTES, &tmB, full_bar(st), kb * 128,
                        t * Cfg::BN);
            tma_load_2d(base + Cfg::OFF_A + st * Cfg::A_BYTES, &tmA, full_bar(st), kb * 128, 0);
            tma_load_2d(base + Cfg::OFF_SC + st * Cfg::SCALE_B, &tmS, full_bar(st), t * Cfg::BN,
                        kb * Cfg::SF_KB);
            tma_load_2d(base + Cfg::OFF_SCA + st * Cfg::SCALE_A, &tmSA, full_bar(st), 0,
                        kb * Cfg::SF_KB);
        } else if constexpr (W4) {
            // 128 rows x 128 bytes of codes (128-byte swizzle), the stage's
            // eight scale rows, and KBOX boxes of A
            tma_load_2d(base + Cfg::OFF_RAW + st * Cfg::RAW_B, &tmB, full_bar(st),
                        kb * (Cfg::KSTAGE / 2), t * Cfg::BN);
            tma_load_2d(base + Cfg::OFF_SC + st * Cfg::SCALE_B, &tmS, full_bar(st), t * Cfg::BN,
                        kb * (Cfg::KSTAGE / 32));
            for (int j = 0; j < KBOX; ++j)
                tma_load_2d(base + Cfg::OFF_A + st * Cfg::A_BYTES + j * Cfg::A_BOX, &tmA,
                            full_bar(st), kb * Cfg::KSTAGE + j * Cfg::BK, 0);
        } else {
            for (int j = 0; j < KBOX; ++j) {
                const int32_t k0 = kb * Cfg::KSTAGE + j * Cfg::BK;
                tma_load_2d(base + Cfg::OFF_B + st * Cfg::B_BYTES + j * Cfg::B_BOX, &tmB,
                            full_bar(st), k0, t * Cfg::BN);
                tma_load_2d(base + Cfg::OFF_A + st * Cfg::A_BYTES + j * Cfg::A_BOX, &tmA,
                            full_bar(st), k0, 0);
            }
        }
    };

    int pre = 0;  // stages the producer issued before the set-up barrier
    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            // the MMA, and (W4) each warp of the converter group that takes the stage
            mbar_init(empty_bar(s), W4 ? Cfg::ISSUERS + Cfg::CONV_WARPS : Cfg::ISSUERS);
        }
        for (int c = 0; c < Cfg::CSETS; ++c) {
            mbar_init(cfull_bar(c), Cfg::CONV_WARPS);
            mbar_init(cempty_bar(c), Cfg::ISSUERS);
        }
        if (MX)
            for (int st = 0; st < STAGES; ++st)
                mbar_init(sfr_bar(st), 1);
        for (int b = 0; b < NACC; ++b) {
            mbar_init(accf_bar(b), Cfg::ISSUERS);
            mbar_init(acce_bar(b), Cfg::EPI_WARPS);
        }
        *abort_flag = 0u;
        fence_mbar_init();
        fence_proxy_async_smem();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if (W4 || MX)
            tma_prefetch_desc(&tmS);
        if (MX)
            tma_prefetch_desc(&tmSA);
        // inputs are read only once the previous kernel in the stream is done
        grid_dependency_wait();
        // the ring is empty: start the B stream now instead of after the
        // tensor-memory allocation and the set-up barrier
        Cursor c = cursor_at(0);
        for (int64_t i = 0; i < n_steps && pre < STAGES; ++i, ++pre) {
            issue_stage(pre, c.t, c.kb, pre == 0 ? args.extra_tx : 0u);
            c = cursor_next(c);
        }
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), Cfg::TMEM_COLS);
        tmem_relinquish();
    }
    grid_dependency_wait();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    if (threadIdx.x == 0)
        grid_launch_dependents();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        pre = __shfl_sync(0xffffffffu, pre, 0);
        int s = 0;
        uint32_t ph = 0;
        int pending = 0;
        bool alive = true;
        Cursor c{0, 0, 0};
        for (int64_t i = 0; i < n_steps; ++i) {
            if (i >= pre) {
                c = i == pre ? cursor_at(i) : cursor_next(c);
                if (!warp_wait_bounded(empty_bar(s), ph ^ 1u, abort_flag, args.status,
                                       args.timeout_ns, kWhereProducerEmpty)) {
                    alive = false;
                    break;
                }
                if (lane == 0)
                    issue_stage(s, c.t, c.kb, 0u);
                __syncwarp();
            }
            pending = min(pending + 1, STAGES);
            if (++s == STAGES) {
                s = 0;
                ph ^= 1u;
            }
        }
        if (!alive && lane == 0) {
            int ds = s;
            uint32_t dph = ph;
            for (int i = 0; i < pending; ++i) {
                if (--ds < 0) {
                    ds = STAGES - 1;
                    dph ^= 1u;
                }
                wait_drain(full_bar(ds), dph, 10000000ull);
            }
        }
        __syncwarp();
    } else if (warp < static_cast<uint32_t>(Cfg::EPI_WARP0)) {
        // ------------------------------------------------------------ MMA issuers
        const int e = static_cast<int>(warp) - 1;  // this warp's share of each stage's blocks
        if (lane == 0) {
            const uint32_t idesc = idesc_f16_f32acc(args.ab_bf16 != 0, Cfg::BN, MP);
            int s = 0;
            uint32_t ph = 0;
            int ab = 0;
            uint32_t aph = 0;
            int cset = 0;  // converted set (W4)
            uint32_t cph = 0;
            bool alive = true;
            for (int64_t i = 0; i < n_steps && alive;) {
                const int64_t i1 = piece_end(i);  // this piece: steps i .. i1 - 1
                if (!wait_bounded<W4>(acce_bar(ab), aph ^ 1u, abort_flag, args.status,
                                      args.timeout_ns, kWhereMmaAccEmpty))
                    break;
                tc_fence_after_sync();
                const uint32_t d_tmem =
                    tmem_base + static_cast<uint32_t>((ab * Cfg::ISSUERS + e) * MP);
                for (int64_t st = i; st < i1; ++st) {
                    if (!wait_bounded<W4 || MX>(full_bar(s), ph, abort_flag, args.status,
                                                args.timeout_ns, kWhereMmaFull)) {
                        alive = false;
                        break;
                    }
                    if (W4 && !wait_bounded<true>(cfull_bar(cset), cph, abort_flag, args.status,
                                            args.timeout_ns, kWhereMmaFull)) {
                        alive = false;  // (the stage's blocks, as bf16 in converted set cset)
                        break;
                    }
                    if (MX && !wait_bounded<true>(sfr_bar(s), ph, abort_flag, args.status,
                                                  args.timeout_ns, kWhereMmaFull)) {
                        alive = false;  // (the stage's scales, rearranged by the scale warp)
                        break;
                    }
                    tc_fence_after_sync();
                    if constexpr (MX) {
                        // this issuer's MMAs k0 .. k0 + MX_PER - 1 of the stage's four
                        // block-scaled ones (M = 128 rows of B, N = MP rows of A, K = 64
                        // each, 32 bytes along the 128-byte rows), all in 128-element
                        // chunk k0 / 2: that chunk's scale tiles of B and A into the
                        // issuer's TMEM columns first; MMA k reads scale bytes 2 (k % 2)
                        // and up
                        const int k0 = e * Cfg::MX_PER;
                        const uint32_t chunk = static_cast<uint32_t>(k0 / 2);
                        const uint32_t sfc = base + Cfg::OFF_SFC + s * Cfg::SF_CP;
                        const uint32_t sfcol =
                            tmem_base + Cfg::SF_COL0 + static_cast<uint32_t>((s * Cfg::ISSUERS + e) * 8);
                        tc_cp_32x128b_warpx4(sfcol, sdesc_rows16(sfc + 512u * chunk));
                        tc_cp_32x128b_warpx4(sfcol + 4u,
                                             sdesc_rows16(sfc + 512u * (Cfg::SF_TILES / 2 + chunk)));
                        const uint64_t bd = sdesc_k_sw128(base + Cfg::OFF_B + s * Cfg::B_BYTES);
                        const uint64_t ad = sdesc_k_sw128(base + Cfg::OFF_A + s * Cfg::A_BYTES);
#pragma unroll
                        for (int kk = 0; kk < Cfg::MX_PER; ++kk) {
                            const int k = k0 + kk;
                            const uint32_t sfid = static_cast<uint32_t>((k % 2) * 2);
                            tc_mma_mxf4(d_tmem, bd + 2u * k, ad + 2u * k,
                                        idesc_mx(1u, Cfg::BN, MP, sfid, sfid), sfcol, sfcol + 4u,
                                        (st != i || kk != 0) ? 1u : 0u);
                        }
                    }
#pragma unroll
                    for (int j = 0; j < (MX ? 0 : KBOX); ++j) {
                        if (W4 && j % Cfg::ISSUERS != e)
                            continue;
                        const uint64_t ad =
                            sdesc_k_sw128(base + Cfg::OFF_A + s * Cfg::A_BYTES + j * Cfg::A_BOX);
                        if constexpr (W4) {
                            // converted rows of B in TMEM: 8 columns per K step of 16
                            const uint32_t bt = tmem_base + Cfg::CSET_COL0 +
                                                Cfg::CSET_COLS * static_cast<uint32_t>(cset) +
                                                static_cast<uint32_t>(j * (Cfg::BK / 2));
#pragma unroll
                            for (int k = 0; k < Cfg::BK / 16; ++k)
                                tc_mma_f16_tmem_a(d_tmem, bt + 8u * k, ad + 2u * k, idesc,
                                                  (st != i || j != e || k != 0) ? 1u : 0u);
                        } else {
                            const uint64_t bd = sdesc_k_sw128(base + Cfg::OFF_B + s * Cfg::B_BYTES +
                                                              j * Cfg::B_BOX);
                            // (several issuers: issuer e takes K steps e KPER .. of each box)
                            constexpr int KPER = (Cfg::BK / 16) / Cfg::ISSUERS;
#pragma unroll
                            for (int kk = 0; kk < KPER; ++kk) {
                                const int k = e * KPER + kk;
                                tc_mma_f16(d_tmem, bd + 2u * k, ad + 2u * k, idesc,
                                           (st != i || j != 0 || kk != 0) ? 1u : 0u);
                            }
                        }
                    }
                    tc_commit(empty_bar(s));
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                    if (W4) {
                        tc_commit(cempty_bar(cset));
                        if (++cset == Cfg::CSETS) {
                            cset = 0;
                            cph ^= 1u;
                        }
                    }
                }
                if (!alive)
                    break;
                tc_commit(accf_bar(ab));
                if (++ab == NACC) {
                    ab = 0;
                    aph ^= 1u;
                }
                i = i1;
            }
        }
        __syncwarp();
    } else if (warp < static_cast<uint32_t>(Cfg::CONV_WARP0)) {
        // ------------------------------------------------------------ epilogue
        const uint32_t q = warp & 3u;
        const bool leader = warp == static_cast<uint32_t>(Cfg::EPI_WARP0) && lane == 0;
        const int32_t n_local = 32 * static_cast<int32_t>(q) + static_cast<int32_t>(lane);
        // this warp's columns of the MP: [mb, mb + MPH)
        constexpr int MPH = MP / Cfg::EPI_SPLIT;
        const int mb = static_cast<int>((warp - static_cast<uint32_t>(Cfg::EPI_WARP0)) / 4u) * MPH;
        constexpr int EPI_THREADS = 32 * Cfg::EPI_WARPS;
        // scattered rows: D row of each row of A, read once (after the set-up
        // barrier, so after the previous kernel in the stream has finished)
        int32_t *drow = reinterpret_cast<int32_t *>(gbase + Cfg::OFF_ROWS);
        if (args.scatter) {
            const int32_t e = static_cast<int32_t>(threadIdx.x) - 32 * Cfg::EPI_WARP0;  // epilogue thread
            if (e < MP) {
                int32_t r = -1;
                if (e < args.M) {
                    r = args.idx[e];
                    if (r < 0 || r >= args.d_rows) {
                        record_error(args.status, kStatusIndex, 0);
                        r = -1;
                    }
                }
                drow[e] = r;
            }
            epi_bar_sync<EPI_THREADS>();
        }
        int ab = 0;
        uint32_t aph = 0;
        for (int64_t i = 0; i < n_steps;) {
            const int32_t t = static_cast<int32_t>(order(i) / nkb);
            i = piece_end(i);
            const int32_t n = t * Cfg::BN + n_local;
            // FP4 weights with MP > 16 finish the MP rows of A in chunks of 16,
            // so the epilogue's registers stay those of MP = 16 and leave room
            // for the converter warps; otherwise one chunk of the warp's MPH
            // rows.  beta * C is fetched while the MMAs still run: into
            // registers when there is one chunk, else its lines into L2.
            constexpr int CH = (W4 && MP > 16) ? 16 : MPH;
            constexpr int NCH = MPH / CH;
            float c0[CH];  // (one chunk) C, still in flight
            if constexpr (NCH == 1) {
                skinny_load_c<CH>(args, drow, n, mb, c0);
            } else if (args.has_c && n < args.N) {
#pragma unroll 4
                for (int m = mb; m < mb + MPH; ++m) {
                    const int32_t r = skinny_row(args, drow, m);
                    if (r >= 0)
                        prefetch_l2(args.C + static_cast<int64_t>(r) * args.ldc + n);
                }
            }
            auto chunk_cb = [&](int g, float (&cb)[CH]) {  // beta * C of chunk g
                if constexpr (NCH == 1) {
                    skinny_beta_c<CH>(args, c0, cb);
                } else {
                    float c[CH];
                    skinny_load_c<CH>(args, drow, n, mb + CH * g, c);
                    skinny_beta_c<CH>(args, c, cb);
                }
            };
            const bool shared_tile = t < S;
            const int32_t c_lo =
                shared_tile ? skinny_owner(static_cast<int64_t>(t) * nkb, W, G) : static_cast<int32_t>(blockIdx.x);
            const int32_t c_hi =
                shared_tile ? skinny_owner(static_cast<int64_t>(t + 1) * nkb - 1, W, G) : c_lo;
            const int32_t parts = args.reduce ? 1 : c_hi - c_lo + 1;
            // a split tile's partial sums: slot (t, blockIdx.x - c_lo) of the workspace
            const int32_t my_slot = static_cast<int32_t>(blockIdx.x) - c_lo;
            float *slot0 = args.workspace + static_cast<int64_t>(t) * args.splits * (Cfg::BN * MP);
            float *mine = slot0 + static_cast<int64_t>(my_slot) * (Cfg::BN * MP);
            // The CTA's last piece, of a split tile whose other parts are all
            // in already (the usual case: the CTAs sharing the tile started
            // with it): this CTA is the last to arrive whatever happens, so it
            // skips writing its part, the fences and the counter, and adds its
            // part from registers below.  (An earlier piece rarely finds the
            // others in, and the extra load there measured slower.  bf16 / f16
            // B only, at most 32 columns a thread: keeping the part in
            // registers spills beside FP4 B's converter warps, and FP4 B ends
            // on whole tiles.)
            // Its counter is read before the wait for this CTA's own sums, and
            // (a tile of two parts, 16 columns a thread: 32 more registers
            // spill beside 32 columns) the other CTA's part with it, so neither
            // round trip follows the last MMA.
            constexpr bool kKeep = !W4 && MPH <= 32 && NCH == 1;
            constexpr bool kPreOther = kKeep && CH <= 16;
            bool last_known = false;
            float other[kPreOther ? CH : 1];  // (kPreOther, two parts) the other CTA's part
            bool have_other = false;
            if (kKeep && parts > 1 && i == n_steps) {
                if (leader) {
                    const uint32_t in = ld_acquire_gpu(args.counters + t);
                    *seen = in;
                }
                epi_bar_sync<EPI_THREADS>();
                last_known = *seen == static_cast<uint32_t>(parts - 1);
                if constexpr (kPreOther) {
                    if (last_known && parts == 2) {
                        const float *src = slot0 + static_cast<int64_t>(1 - my_slot) * (Cfg::BN * MP);
#pragma unroll
                        for (int m = 0; m < CH; ++m)
                            other[m] = __ldcg(src + (mb + m) * Cfg::BN + n_local);
                        have_other = true;
                    }
                }
            }
            // (inline: the loads of C and of the other part stay in flight)
            const bool ok = warp_wait_bounded_inline(accf_bar(ab), aph, abort_flag, args.status,
                                                     args.timeout_ns, kWhereEpiAccFull);
            // all epilogue warps agree before the named barriers below
            epi_bar_sync<EPI_THREADS>();
            if (!ok || *abort_flag)
                break;
            tc_fence_after_sync();
            float v[CH];  // this chunk's sums (with one chunk: the CTA's whole part)
#pragma unroll 1
            for (int g = 0; g < NCH; ++g) {
                // the issuers' partial sums of this chunk, added in issuer order:
                // with several issuers (not FP4 B, whose converter warps leave
                // few registers) all loads first and one wait, else one 16-column
                // load and wait at a time
                auto tmem_col = [&](int e, int h) {
                    return tmem_base + ((32u * q) << 16) +
                           static_cast<uint32_t>((ab * Cfg::ISSUERS + e) * MP + mb + CH * g + 16 * h);
                };
                if constexpr (Cfg::ISSUERS > 1 && !W4) {
                    uint32_t r[Cfg::ISSUERS][CH / 16][16];
#pragma unroll
                    for (int e = 0; e < Cfg::ISSUERS; ++e)
#pragma unroll
                        for (int h = 0; h < CH / 16; ++h)
                            tc_ld_32x32b_x16(tmem_col(e, h), r[e][h]);
#pragma unroll
                    for (int e = 0; e < Cfg::ISSUERS; ++e)
#pragma unroll
                        for (int h = 0; h < CH / 16; ++h)
                            tc_wait_ld(r[e][h]);  // (the first waits; the rest tie the registers)
#pragma unroll
                    for (int e = 0; e < Cfg::ISSUERS; ++e)
#pragma unroll
                        for (int h = 0; h < CH / 16; ++h)
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                v[16 * h + i] = e == 0 ? __uint_as_float(r[e][h][i])
                                                       : v[16 * h + i] + __uint_as_float(r[e][h][i]);
                } else {
#pragma unroll
                    for (int e = 0; e < Cfg::ISSUERS; ++e) {
#pragma unroll
                        for (int h = 0; h < CH / 16; ++h) {
                            uint32_t r[16];
                            tc_ld_32x32b_x16(tmem_col(e, h), r);
                            tc_wait_ld(r);
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                v[16 * h + i] = e == 0 ? __uint_as_float(r[i])
                                                       : v[16 * h + i] + __uint_as_float(r[i]);
                        }
                    }
                }
                if (args.reduce) {
                    skinny_add<CH>(args, drow, n, mb + CH * g, v);  // every part adds itself into D
                } else if (parts == 1) {
                    float cb[CH];
                    chunk_cb(g, cb);
                    skinny_store<CH>(args, drow, n, mb + CH * g, v, cb);
                } else if (!last_known) {
#pragma unroll
                    for (int m = 0; m < CH; ++m)
                        __stcg(mine + (mb + CH * g + m) * Cfg::BN + n_local, v[m]);
                }
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(acce_bar(ab));
            if (++ab == NACC) {
                ab = 0;
                aph ^= 1u;
            }
            if (parts == 1)
                continue;
            if (!last_known) {
                // The CTA barrier orders every thread's partial before the
                // leader's device-scope fence and counter increment; for the
                // last CTA to arrive, the leader's second fence orders the
                // other CTAs' parts before the reads below (the barrier after
                // it passes that on).  (With the other parts seen in beforehand,
                // the acquire load above and its barrier did the same.)
                epi_bar_sync<EPI_THREADS>();
                if (leader) {
                    __threadfence();
                    const uint32_t before = atomicAdd(args.counters + t, 1u);
                    if (before == static_cast<uint32_t>(parts - 1))
                        __threadfence();
                    *arrival = before;
                }
                epi_bar_sync<EPI_THREADS>();
                if (*arrival != static_cast<uint32_t>(parts - 1))
                    continue;  // another CTA still has to add its part
            }
            // last to arrive: add the parts in slot order (this CTA's own part
            // from registers where it keeps it -- the bits it wrote or would
            // have written -- else read back), then finish the tile
#pragma unroll 1
            for (int g = 0; g < NCH; ++g) {
                float sum[CH];
#pragma unroll
                for (int m = 0; m < CH; ++m)
                    sum[m] = 0.f;
                for (int p = 0; p < parts; ++p) {
                    const float *src = slot0 + static_cast<int64_t>(p) * (Cfg::BN * MP);
                    float part[CH];
                    if (kKeep && p == my_slot) {
#pragma unroll
                        for (int m = 0; m < CH; ++m)
                            part[m] = v[m];
                    } else if (kPreOther && have_other) {
#pragma unroll
                        for (int m = 0; m < CH; ++m)
                            part[m] = other[kPreOther ? m : 0];
                    } else {
#pragma unroll
                        for (int m = 0; m < CH; ++m)
                            part[m] = __ldcg(src + (mb + CH * g + m) * Cfg::BN + n_local);
                    }
#pragma unroll
                    for (int m = 0; m < CH; ++m)
                        sum[m] += part[m];
                }
                float cb[CH];
                chunk_cb(g, cb);
                skinny_store<CH>(args, drow, n, mb + CH * g, sum, cb);
            }
            if (leader)
                args.counters[t] = 0u;  // ready for the next call
        }
    } else if constexpr (W4) {
        // ------------------------------------------------------------ converters
        // Every converter warp takes every stage of this CTA's share: lane l of
        // warp w turns row 32 (w % 4) + l of its run of blocks (32 bytes of
        // codes and two scales each) into bf16 and stores it in that TMEM lane
        // of the stage's converted set.
        constexpr uint32_t kRun = static_cast<uint32_t>(KBOX / Cfg::CONV_PER_Q);
        const uint32_t cw = warp - static_cast<uint32_t>(Cfg::CONV_WARP0);
        const uint32_t quarter = warp & 3u;
        const uint32_t row = 32u * quarter + lane;
        const uint32_t j0 = (cw / 4u) * kRun;
        const uint32_t t_lane = tmem_base + ((32u * quarter) << 16);
        int s = 0;
        uint32_t ph = 0;
        int cset = 0;
        uint32_t cph = 0;
        for (int64_t q = 0; q < n_steps; ++q) {
            if (!warp_wait_bounded<true>(full_bar(s), ph, abort_flag, args.status, args.timeout_ns,
                                   kWhereMmaFull))
                break;
            if (!warp_wait_bounded<true>(cempty_bar(cset), cph ^ 1u, abort_flag, args.status,
                                   args.timeout_ns, kWhereProducerEmpty))
                break;
            tc_fence_after_sync();  // the stores below come after the MMA's reads of the set
            const uint32_t src = base + Cfg::OFF_RAW + s * Cfg::RAW_B + row * 128u;
            const uint32_t sc = base + Cfg::OFF_SC + s * Cfg::SCALE_B + row;
            const uint32_t tcol = t_lane + Cfg::CSET_COL0 + Cfg::CSET_COLS * static_cast<uint32_t>(cset);
#pragma unroll 1
            for (uint32_t j = j0; j < j0 + kRun; ++j) {
                // block j: the row's 16-byte chunks 2j, 2j+1 of the 128-byte swizzled image
                uint32_t w[8];
                ld_shared_v4(src + (((2u * j) ^ (row & 7u)) << 4), w[0], w[1], w[2], w[3]);
                ld_shared_v4(src + (((2u * j + 1u) ^ (row & 7u)) << 4), w[4], w[5], w[6], w[7]);
                uint32_t v[32];  // the block's 64 elements, two per column, in K order
                // scale blocks 2j and 2j+1 (words 0-3 and 4-7): the first word of
                // each through the byte tables, the other three as bit fields (the
                // mix keeps the ALU and FMA pipes both busy); one warp vote for the
                // block picks the field form with or without its second factor
                const uint32_t s_lo = ld_shared_u8(sc + 2u * j * 128u);
                const uint32_t s_hi = ld_shared_u8(sc + (2u * j + 1u) * 128u);
                uint32_t fa[2], fb[2];
                const bool two_lo = e2m1_field_scales(s_lo, fa[0], fb[0]);
                const bool two_hi = e2m1_field_scales(s_hi, fa[1], fb[1]);
                {
                    uint32_t p[4];
                    e2m1x8_to_bf16(w[0], ue8m0_to_bf16x2(s_lo), p);
#pragma unroll
                    for (uint32_t e = 0; e < 4; ++e)
                        v[e] = p[e];
                    e2m1x8_to_bf16(w[4], ue8m0_to_bf16x2(s_hi), p);
#pragma unroll
                    for (uint32_t e = 0; e < 4; ++e)
                        v[16 + e] = p[e];
                }
                if (__any_sync(0xffffffffu, two_lo || two_hi)) {
#pragma unroll
                    for (uint32_t k = 1; k < 8; ++k) {
                        if (k == 4)
                            continue;
                        uint32_t p[4];
                        e2m1x8_to_bf16_fields<true>(w[k], fa[k / 4], fb[k / 4], p);
#pragma unroll
                        for (uint32_t e = 0; e < 4; ++e)
                            v[4 * k + e] = p[e];
                    }
                } else {
#pragma unroll
                    for (uint32_t k = 1; k < 8; ++k) {
                        if (k == 4)
                            continue;
                        uint32_t p[4];
                        e2m1x8_to_bf16_fields<false>(w[k], fa[k / 4], fb[k / 4], p);
#pragma unroll
                        for (uint32_t e = 0; e < 4; ++e)
                            v[4 * k + e] = p[e];
                    }
                }
                tc_st_32x32b_x32(tcol + 32u * j, v);
            }
            tc_wait_st();
            tc_fence_before_sync();  // the MMA reads the set once every converter has arrived
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(cfull_bar(cset));
                mbar_arrive(empty_bar(s));
            }
            if (++s == STAGES) {
                s = 0;
                ph ^= 1u;
            }
            if (++cset == Cfg::CSETS) {
                cset = 0;
                cph ^= 1u;
            }
        }
    } else if constexpr (MX) {
        // ------------------------------------------------------------ scale warp
        // Per stage: the scale rows as loaded (row b: one byte per row of B, then
        // one per row of A) into the tiles tcgen05.cp takes -- lane l loads the
        // 32-bit words of rows 4l .. 4l+3 for four blocks, transposes the 4 x 4
        // bytes so each word holds one row's four blocks, and stores row r's word
        // at 16 (r % 32) + 4 (r / 32) of the tile (rows of A past MP zero) --
        // then hands the stage to the MMA thread (tcgen05.cp reads through the
        // async proxy, hence the fence).
        int s = 0;
        uint32_t ph = 0;
        for (int64_t q = 0; q < n_steps; ++q) {
            if (!warp_wait_bounded<true>(full_bar(s), ph, abort_flag, args.status, args.timeout_ns,
                                         kWhereMmaFull))
                break;
            const uint8_t *srcb = gbase + Cfg::OFF_SC + s * Cfg::SCALE_B;
            const uint8_t *srca = gbase + Cfg::OFF_SCA + s * Cfg::SCALE_A;
            uint8_t *dst = gbase + Cfg::OFF_SFC + s * Cfg::SF_CP;
#pragma unroll
            for (int ti = 0; ti < Cfg::SF_TILES; ++ti) {
                const bool b_tile = ti < Cfg::SF_TILES / 2;
                const int c = ti % (Cfg::SF_TILES / 2);
                const uint32_t pitch = b_tile ? static_cast<uint32_t>(Cfg::BN) : static_cast<uint32_t>(MP);
                const uint8_t *src = (b_tile ? srcb : srca) + 4u * c * pitch + 4u * lane;
                const bool have = b_tile || 4u * lane < static_cast<uint32_t>(MP);
                uint32_t w[4];
#pragma unroll
                for (int b = 0; b < 4; ++b)
                    w[b] = have ? *reinterpret_cast<const uint32_t *>(src + b * pitch) : 0u;
                const uint32_t t0 = __byte_perm(w[0], w[1], 0x5140);
                const uint32_t t1 = __byte_perm(w[0], w[1], 0x7362);
                const uint32_t t2 = __byte_perm(w[2], w[3], 0x5140);
                const uint32_t t3 = __byte_perm(w[2], w[3], 0x7362);
                const uint32_t o[4] = {__byte_perm(t0, t2, 0x5410), __byte_perm(t0, t2, 0x7632),
                                       __byte_perm(t1, t3, 0x5410), __byte_perm(t1, t3, 0x7632)};
                uint8_t *tile = dst + 512u * ti + 4u * (lane / 8u);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    *reinterpret_cast<uint32_t *>(tile + 16u * ((4u * lane + i) % 32u)) = o[i];
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(sfr_bar(s));
            if (++s == STAGES) {
                s = 0;
                ph ^= 1u;
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
}

}  // namespace tcg
