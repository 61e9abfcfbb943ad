// kernel_tile.cuh -- persistent warp-specialised tcgen05 GEMM, 128 x BN tiles.
//
//   warp 0      producer: TMA loads of A (tiled, or tile::gather4 rows of a
//               table) and B boxes into a STAGES-deep shared ring, each stage
//               completing on an mbarrier armed with its byte count
//               ("cp.async.bulk.tensor" page, sections "Example: two explicit
//               8x16 boxes" and "Gather4 and scatter4").
//   warp 1      MMA issuer: one thread issues tcgen05.mma (M=128, N=BN, K=16)
//               into one of two TMEM accumulators; the first K step starts
//               from zero and later ones accumulate ("mma.sync" page, section
//               "Accumulation, transpose and alpha/beta": only the first K
//               issue reads the start value).  tcgen05.commit frees stages.
//               (Single CTAs with BN <= 128: warp 6 is a second issuer taking
//               every other K block into an accumulator of its own.)
//   warps 2-5   epilogue: TMEM -> registers (tcgen05.ld; the two issuers'
//               partial sums added), optional C box via
//               TMA, D = fma.rn(alpha, acc, beta*C) ("fma" page), convert,
//               swizzled shared image, TMA store ("cp.async.bulk.tensor"
//               page, section "Stores, reductions, and completion").  With
//               scattered rows, C comes in by tile::gather4 and D goes out by
//               tile::scatter4 at the rows idx[m] (section "Gather4 and
//               scatter4").  In the accumulating form the box is added into
//               D by a TMA reduce-add instead of stored.
//
// PAIR = true runs the same roles on a CTA pair (ranks 2p, 2p+1 of a cluster) sharing
// one tcgen05.mma.cta_group::2 of M = 256: each CTA loads its own 128 rows of
// A and its own half of the BN rows of B, both report their bytes to the
// leader CTA's stage barrier, the leader's MMA thread issues for both, and
// commits arrive in both CTAs.  Each CTA drains its own 128 accumulator rows.
// Per SM this moves 2/3 of the operand bytes of the single-CTA form.  With
// MC = 2 as well, two pairs (a cluster of four) compute neighbouring tiles of
// one block row and each CTA loads half of its A rows, multicasting them to the
// CTA with the same role in the other pair: half the A loads (or gather4
// issues) per CTA at the pair form's bytes per flop.
//
// Two accumulators let the epilogue of tile i overlap the mainloop of tile
// i+1.  NSUB = 2 (a 2*BN-wide tile made of two MMA halves) has room for one
// accumulator only; its halves are handed over separately and the MMA order
// at tile boundaries lets the drain of one half overlap MMAs of the other.  Every wait is bounded (common.cuh); on a timeout all roles leave
// their loops, the copies in flight are drained, TMEM is freed and the
// kernel returns with the error recorded.
#pragma once

#include "common.cuh"

// Evict-first L2 policy on the epilogue's C loads and D stores (0 or 1;
// measured 1-3% faster on the 8192^3 and 8192 x 28672 x 4096 workloads).
#ifndef TCG_EPI_EVICT_FIRST
#define TCG_EPI_EVICT_FIRST 1
#endif

namespace tcg {

template <int BN_, int STAGES_, bool PAIR_ = false, int NSUB_ = 1, int MC_ = 1, int MX_ = 0>
struct TileCfg {
    static constexpr bool PAIR = PAIR_;
    // MX: operand kind.  0 = f16/bf16 (tcgen05 kind::f16); 1 = FP4 E2M1 codes
    // packed two per byte (kind::mxf4); 2 = FP4 codes in the 16U4_ALIGN16B TMA
    // image, sixteen codes in the low 8 bytes of each 16-byte block
    // (kind::mxf8f6f4).  The FP4 kinds carry UE8M0 block scales (one per 32
    // elements along K) through shared memory into TMEM.  Single CTAs, or CTA
    // pairs (each CTA holds the scales of its own rows of A and of all of B's).
    static constexpr int MX = MX_;
    // MC > 1: MC CTAs (or MC pairs) work on MC neighbouring tiles of one
    // block row; each loads 1/MC of the shared A box and multicasts it to the
    // others, so per CTA the A traffic (or the number of gather4 issues) drops
    // by MC.
    static constexpr int MC = MC_;
    static constexpr int CLUSTER = (PAIR ? 2 : 1) * MC;
    // NSUB = 2: the tile is two BN-wide halves side by side (two MMAs per K
    // step into one 2*BN-column accumulator), so each row of A feeds twice the
    // work; without a second accumulator the epilogue no longer overlaps.
    static constexpr int NSUB = NSUB_;
    static constexpr int BM = 128;                  // rows of A (and D) per CTA
    static constexpr int TILE_M = PAIR ? 256 : 128;  // rows per output tile
    static constexpr int BN = BN_;       // N of one MMA
    static constexpr int TILE_N = BN * NSUB;
    // Accumulators: two (the epilogue of one tile overlaps the next tile's
    // MMAs), except for two-half tiles and for FP4 tiles 256 wide, whose block
    // scales need TMEM columns beside the one 256-column accumulator.
    static constexpr int NUM_ACC = (NSUB == 1 && !(MX != 0 && BN == 256)) ? 2 : 1;
    static constexpr int BN_LOCAL = PAIR ? BN / 2 : BN;  // rows of B per half each CTA loads
    // K elements per stage: one 128-byte swizzle row of each operand row
    // (64 x 16-bit, 256 packed FP4 codes, or 128 codes in the 16U4 image)
    static constexpr int BK = MX == 0 ? 64 : (MX == 1 ? 256 : 128);
    static constexpr int MMA_K = MX == 0 ? 16 : (MX == 1 ? 64 : 32);  // K of one MMA (32 bytes)
    static constexpr int STAGES = STAGES_;
    static constexpr uint32_t ROW_BYTES = 128;
    static constexpr uint32_t A_BYTES = BM * ROW_BYTES;
    static constexpr int A_SLICE_ROWS = BM / MC;  // rows of A this CTA loads for the cluster
    static constexpr uint32_t A_SLICE_BYTES = A_BYTES / MC;
    static constexpr uint32_t B_SUB_BYTES = BN_LOCAL * ROW_BYTES;
    static constexpr uint32_t B_BYTES = NSUB * B_SUB_BYTES;
    static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
    // Block scales of a stage (FP4): SF_KB rows of 32-element blocks, as TMA
    // loads them from the K/32 x rows scale matrices (BM bytes for A, TILE_N
    // for B per row), then rearranged by the scale warp into 512-byte tiles
    // (128 rows x 4 blocks: row l + 32 q of the tile, block b at byte
    // 16 l + 4 q + b) that tcgen05.cp copies into 4 TMEM columns each: the A
    // tiles (one per 128-element K chunk), then per chunk the B row tiles.
    static constexpr int SF_KB = MX ? BK / 32 : 0;
    static constexpr int SF_CHUNKS = MX ? BK / 128 : 0;
    static constexpr int SF_B_ROWTILES = MX ? (TILE_N + 127) / 128 : 0;
    static constexpr int SF_TILES = SF_CHUNKS * (1 + SF_B_ROWTILES);
    static constexpr uint32_t SF_STAGE_BYTES = SF_KB * (BM + TILE_N);
    static constexpr uint32_t SF_CP_BYTES = SF_TILES * 512;
    static constexpr uint32_t SF_COLS = SF_TILES * 4;  // TMEM columns per stage
    // bytes one CTA's code loads report per stage: codes in the 16U4 image count
    // their payload, not the padding ("cp.async.bulk.tensor" page, section
    // "Interleave and packed FP4"); the scale rows complete on a barrier of
    // their own (SF_STAGE_BYTES)
    static constexpr uint32_t STAGE_TX = MX == 2 ? STAGE_BYTES / 2 : STAGE_BYTES;
    static constexpr uint32_t EPI_BUF = 32 * 128;  // 32 rows x 128 B
    static constexpr uint32_t OFF_A = 0;
    static constexpr uint32_t OFF_B = STAGES * A_BYTES;
    static constexpr uint32_t OFF_SFS = STAGES * STAGE_BYTES;             // scales as loaded
    static constexpr uint32_t OFF_SFC = OFF_SFS + STAGES * SF_STAGE_BYTES;  // rearranged
    static constexpr uint32_t OFF_EPI = OFF_SFC + STAGES * SF_CP_BYTES;
    static constexpr uint32_t OFF_BAR = OFF_EPI + 8 * EPI_BUF;  // 4 warps x 2 buffers
    static constexpr uint32_t NUM_BARS = 2 * STAGES + 4 + 8 + (MX ? 2 * STAGES : 0);
    static constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16;
    static constexpr uint32_t SMEM_ALLOC = SMEM_BYTES + 1024;  // slack to align the base
    // MMA issuers.  One thread issues a tcgen05.mma about every 117 cycles
    // whatever its N, while a 128 x BN x 16 MMA takes the tensor pipe about
    // BN / 2 cycles: at BN <= 128 a lone issuer, not the tensor pipe, sets
    // the rate.  Those single-CTA forms get a second issuing warp (warp 6)
    // that takes every other K block into an accumulator of its own; the
    // epilogue adds the two.  (Pairs and wider tiles are tensor-bound.)
    static constexpr int ISS = (!PAIR && MC == 1 && NSUB == 1 && BN <= 128 && MX == 0) ? 2 : 1;
    static constexpr uint32_t ACC_COLS = NUM_ACC * TILE_N * ISS;  // fp32 accumulators
    static constexpr uint32_t SF_COL0 = ACC_COLS;                 // first scale column (FP4)
    static constexpr uint32_t TMEM_COLS = MX ? 512u : ACC_COLS;
    // warp 6: the second MMA issuer, or (FP4) the scale warp
    static constexpr int THREADS = 192 + 32 * (ISS - 1) + (MX ? 32 : 0);
    static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "tile width");
    static_assert(NSUB == 1 || NSUB == 2, "one or two halves");
    static_assert(MC == 1 || (!PAIR && (MC == 2 || MC == 4 || MC == 8)) ||
                      (PAIR && (MC == 2 || MC == 4)),
                  "A multicast over 2, 4 or 8 single CTAs, or over two or four pairs");
    static_assert(!PAIR || (BN % 32 == 0 && BN_LOCAL % 8 == 0), "pair splits B in 8-row groups");
    static_assert(TMEM_COLS >= 32 && TMEM_COLS <= 512 && (TMEM_COLS & (TMEM_COLS - 1)) == 0,
                  "TMEM allocation must be a power of two in [32, 512]");
    static_assert(MX == 0 || (MC == 1 && NSUB == 1 && (BN == 256 || (BN == 128 && !PAIR))),
                  "FP4 operands: single CTAs with tiles 128 or 256 wide, or pairs with 256 x 256 tiles");
    static_assert(MX == 0 || SF_COL0 + STAGES * SF_COLS <= 512, "TMEM for the block scales");
};

// Byte offset of 16-byte chunk `chunk` of row `row` in a swizzled box image
// whose rows are `row_bytes` long (128: 128-byte swizzle, 64: 64-byte).  The
// image base is aligned to the swizzle period.
__device__ __forceinline__ uint32_t swz_off(uint32_t row, uint32_t chunk, uint32_t row_bytes)
{
    const uint32_t lin = row * row_bytes + chunk * 16u;
    const uint32_t mask = row_bytes / 16u - 1u;  // 7 or 3
    return lin ^ (((lin >> 7) & mask) << 4);
}

// Epilogue modes, a template parameter so that each kernel carries only its own:
// the fma.rn epilogue with optional C, rows scattered through idx, reduce-add
// into D, and accumulators seeded with C.
enum : int { kModePlain = 0, kModeScatter = 1, kModeReduce = 2, kModeSeed = 3 };

template <int BN, int STAGES, bool PAIR, int NSUB, int MC, int MODE, int MX = 0>
__global__ void __launch_bounds__(TileCfg<BN, STAGES, PAIR, NSUB, MC, MX>::THREADS, 1)
    tile_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmC,
                     const __grid_constant__ CUtensorMap tmD,
                     const __grid_constant__ CUtensorMap tmSFA,
                     const __grid_constant__ CUtensorMap tmSFB, const GemmArgs args)
{
    using Cfg = TileCfg<BN, STAGES, PAIR, NSUB, MC, MX>;
    constexpr int CL = Cfg::CLUSTER;
    // issuers in use: one for seeded accumulators (C is the start value of the
    // one chain of K steps, as the pages' recurrence has it)
    constexpr int kIss = MODE == kModeSeed ? 1 : Cfg::ISS;
    constexpr uint16_t kAllCtas = static_cast<uint16_t>((1u << CL) - 1u);
    constexpr int TILE_N = Cfg::TILE_N;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);

    const uint32_t warp = __shfl_sync(0xffffffffu, threadIdx.x / 32u, 0);
    const uint32_t lane = threadIdx.x % 32u;

    const uint32_t bar0 = base + Cfg::OFF_BAR;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto accf_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
    auto acce_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
    auto c_bar = [&](int q, int j) { return bar0 + 8u * (2 * STAGES + 4 + 2 * q + j); };
    // (FP4) stage s's scale rows have landed in this CTA / have been rearranged
    // for tcgen05.cp (in the leader: by the scale warps of both CTAs of a pair)
    auto sf_full_bar = [&](int st) { return bar0 + 8u * (2 * STAGES + 12 + st); };
    auto sf_bar = [&](int st) { return bar0 + 8u * (3 * STAGES + 12 + st); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + Cfg::OFF_MISC);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(gbase + Cfg::OFF_MISC + 4);

    // cluster bookkeeping: pairs (ranks 2p, 2p+1; the even rank leads), MC
    // CTAs or pairs sharing A, or one CTA
    const uint32_t rank = CL > 1 ? cluster_ctarank() : 0u;
    const uint32_t role = PAIR ? (rank & 1u) : 0u;        // place within the pair
    const uint32_t share = PAIR ? (rank >> 1) : rank;     // which of the MC sharers of A
    const uint32_t pair_base = rank & ~1u;
    const bool leader = !PAIR || role == 0u;
    const int32_t cta_set = static_cast<int32_t>(blockIdx.x) / CL;
    const int32_t cta_sets = static_cast<int32_t>(gridDim.x) / CL;
    // CTAs that receive this CTA's slice of A: all of the cluster, or (pairs)
    // the CTAs with the same role in every pair
    constexpr uint16_t kSameRole = PAIR ? static_cast<uint16_t>(0x5555u & kAllCtas) : kAllCtas;
    const uint16_t a_mask = static_cast<uint16_t>(kSameRole << role);
    // this pair's two CTAs, as a multicast mask
    const uint16_t pair_mask = static_cast<uint16_t>(3u << pair_base);
    // the leader's copy of a barrier, as a shared::cluster address
    auto lead = [&](uint32_t bar) { return PAIR ? mapa_shared(bar, pair_base) : bar; };
    // raise the abort flag here and (pair) in the peer CTA
    auto raise_abort = [&]() {
        *abort_flag = 1u;
        if (PAIR)
            st_shared_cluster_u32(mapa_shared(smem_u32(const_cast<uint32_t *>(abort_flag)), rank ^ 1u), 1u);
    };

    // Single CTAs loading plain boxes (and, FP4, the stage's scale rows): the
    // first tile's first stages are issued right after the barriers exist,
    // before the tensor-memory allocation and the set-up barrier (one-wave
    // problems spend a good part of their time reaching the first full stage).
    // `pre` stages; the producer skips them.
    constexpr bool kPrefill = !PAIR && MC == 1;
    int pre = 0;
    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), MC);  // MC > 1: every CTA's MMA frees the shared A slices
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), kIss);  // each issuer's last MMAs of the tile
            mbar_init(acce_bar(b), PAIR ? 8 : 4);  // one arrival per epilogue warp (of both CTAs)
        }
        for (int q = 0; q < 4; ++q)
            for (int j = 0; j < 2; ++j)
                mbar_init(c_bar(q, j), 1);
        if (MX)
            for (int st = 0; st < STAGES; ++st) {
                mbar_init(sf_full_bar(st), 1);
                mbar_init(sf_bar(st), PAIR ? 2 : 1);
            }
        *abort_flag = 0u;
        fence_mbar_init();
        fence_proxy_async_smem();
        if (args.num_k_blocks > 0) {  // with K == 0 the A/B descriptors are left empty
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            if (MX) {
                tma_prefetch_desc(&tmSFA);
                tma_prefetch_desc(&tmSFB);
            }
        }
        if (args.has_c && args.c_tma)
            tma_prefetch_desc(&tmC);
        if (args.d_tma)
            tma_prefetch_desc(&tmD);
        if constexpr (kPrefill) {
            if (!args.gather && args.num_k_blocks > 0 && cta_set < args.num_tiles) {
                // (inputs are read only once the previous kernel in the stream is done)
                if (!args.co_tail)
                    grid_dependency_wait();
                int32_t mb, nb;
                tile_coords(cta_set, args, mb, nb);
                const int32_t m0 = mb * Cfg::TILE_M, nb0 = nb * TILE_N;
                const int32_t n = min(STAGES, args.num_k_blocks);
                for (; pre < n; ++pre) {
                    const int32_t k0 = MX ? pre * 128 : pre * Cfg::BK;
                    if (MX) {
                        const uint32_t sfs = base + Cfg::OFF_SFS + pre * Cfg::SF_STAGE_BYTES;
                        mbar_arrive_expect_tx(sf_full_bar(pre), Cfg::SF_STAGE_BYTES);
                        tma_load_2d(sfs, &tmSFA, sf_full_bar(pre), m0, pre * Cfg::SF_KB);
                        tma_load_2d(sfs + Cfg::SF_KB * Cfg::BM, &tmSFB, sf_full_bar(pre), nb * TILE_N,
                                    pre * Cfg::SF_KB);
                    }
                    mbar_arrive_expect_tx(full_bar(pre), Cfg::STAGE_TX + (pre == 0 ? args.extra_tx : 0u));
                    tma_load_2d(base + Cfg::OFF_A + pre * Cfg::A_BYTES, &tmA, full_bar(pre), k0, m0);
                    for (int j = 0; j < NSUB; ++j)
                        tma_load_2d(base + Cfg::OFF_B + pre * Cfg::B_BYTES + j * Cfg::B_SUB_BYTES, &tmB,
                                    full_bar(pre), k0, nb0 + j * BN);
                }
            }
        }
    }
    if (warp == 1) {
        if (PAIR) {
            tmem_alloc_pair(smem_u32(tmem_slot), Cfg::TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(tmem_slot), Cfg::TMEM_COLS);
            tmem_relinquish();
        }
    }
    // set-up above touched only shared and tensor memory; inputs and outputs
    // are used only after the previous kernel in the stream has finished (a
    // co-launched tail skips this: the kernel it runs beside let it launch
    // only after passing this same wait, and writes other rows of D)
    if (!args.co_tail)
        grid_dependency_wait();
    tc_fence_before_sync();
    if (CL > 1)
        cluster_sync_all();  // the peers' barriers exist before anything targets them
    else
        __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    if (threadIdx.x == 0)
        grid_launch_dependents();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        int s = 0;
        uint32_t ph = 0;
        int pending = 0;  // stages issued and not yet seen consumed (for teardown)
        bool first = true;
        bool alive = true;
        int pre_left = __shfl_sync(0xffffffffu, pre, 0);  // prefilled stages of the first tile
        for (int32_t t = cta_set; t < args.num_tiles && alive; t += cta_sets) {
            int32_t mb, nb;
            tile_coords(t, args, mb, nb);
            if (MC > 1)
                nb = nb * MC + static_cast<int32_t>(share);  // this CTA's tile of the cluster's row
            const int32_t m0 = mb * Cfg::TILE_M + static_cast<int32_t>(role) * Cfg::BM;
            const int32_t nb0 = nb * TILE_N + static_cast<int32_t>(role) * Cfg::BN_LOCAL;
            // rows of A this CTA fetches: all 128, or (MC > 1) its slice for the sharers
            const int32_t a_row0 = m0 + (MC > 1 ? static_cast<int32_t>(share) * Cfg::A_SLICE_ROWS : 0);
            const uint32_t a_off = MC > 1 ? share * Cfg::A_SLICE_BYTES : 0u;
            const bool gather_lane = static_cast<int>(lane) < Cfg::A_SLICE_ROWS / 4;
            int32_t rows[4] = {0, 0, 0, 0};
            if (args.gather && gather_lane) {
                // lane l fetches rows 4l .. 4l+3 of the slice, four per gather4
                for (int r = 0; r < 4; ++r) {
                    const int32_t m = a_row0 + 4 * (int32_t)lane + r;
                    int32_t v = 0;
                    if (m < args.M) {
                        v = args.idx[m];
                        if (v < 0 || v >= args.table_rows) {
                            record_error(args.status, kStatusIndex, 0);
                            v = 0;  // fetch a valid row; the epilogue zeroes this one
                        }
                    }
                    rows[r] = v;
                }
            }
            for (int32_t kb = 0; kb < args.num_k_blocks; ++kb) {
                if (pre_left > 0) {  // issued before the set-up barrier
                    --pre_left;
                    first = false;
                    pending = min(pending + 1, STAGES);
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                    continue;
                }
                if (!warp_wait_bounded<true>(empty_bar(s), ph ^ 1u, abort_flag, args.status,
                                       args.timeout_ns, kWhereProducerEmpty)) {
                    alive = false;
                    break;
                }
                if (lane == 0 && leader) {
                    // the leader's barrier counts the bytes of both CTAs of a pair
                    const uint32_t bytes = (PAIR ? 2u : 1u) * Cfg::STAGE_TX + (first ? args.extra_tx : 0u);
                    mbar_arrive_expect_tx(full_bar(s), bytes);
                }
                first = false;
                __syncwarp();
                // inner coordinate: K elements (16-bit codes and the 16U4 image) or
                // bytes (packed FP4 codes); FP4 rows of a stage are 128 of either
                const int32_t k0 = MX ? kb * 128 : kb * Cfg::BK;
                const uint32_t sa = base + Cfg::OFF_A + s * Cfg::A_BYTES;
                const uint32_t sb = base + Cfg::OFF_B + s * Cfg::B_BYTES;
                if (MX && lane == 0) {
                    // FP4: the stage's SF_KB rows of block scales, this CTA's rows of A
                    // and all of the tile's rows of B, on this CTA's own barrier
                    const uint32_t sfs = base + Cfg::OFF_SFS + s * Cfg::SF_STAGE_BYTES;
                    mbar_arrive_expect_tx(sf_full_bar(s), Cfg::SF_STAGE_BYTES);
                    tma_load_2d(sfs, &tmSFA, sf_full_bar(s), m0, kb * Cfg::SF_KB);
                    tma_load_2d(sfs + Cfg::SF_KB * Cfg::BM, &tmSFB, sf_full_bar(s), nb * TILE_N,
                                kb * Cfg::SF_KB);
                }
                if (PAIR) {
                    const uint32_t fb = lead(full_bar(s));
                    if (MC > 1) {
                        if (args.gather) {
                            if (gather_lane)
                                tma_gather4_pair_multicast(sa + a_off + lane * 512u, &tmA, fb, k0,
                                                           rows[0], rows[1], rows[2], rows[3], a_mask);
                        } else if (lane == 0) {
                            tma_load_2d_pair_multicast(sa + a_off, &tmA, fb, k0, a_row0, a_mask);
                        }
                    } else if (args.gather) {
                        tma_gather4_pair(sa + lane * 512u, &tmA, fb, k0, rows[0], rows[1], rows[2],
                                         rows[3]);
                    } else if (lane == 0) {
                        tma_load_2d_pair(sa, &tmA, fb, k0, m0);
                    }
                    if (lane == 0)
                        for (int j = 0; j < NSUB; ++j)
                            tma_load_2d_pair(sb + j * Cfg::B_SUB_BYTES, &tmB, fb, k0, nb0 + j * BN);
                } else if (MC > 1) {
                    if (args.gather) {
                        if (gather_lane)
                            tma_gather4_multicast(sa + a_off + lane * 512u, &tmA, full_bar(s), k0,
                                                  rows[0], rows[1], rows[2], rows[3], a_mask);
                    } else if (lane == 0) {
                        tma_load_2d_multicast(sa + a_off, &tmA, full_bar(s), k0, a_row0, a_mask);
                    }
                    if (lane == 0)
                        tma_load_2d(sb, &tmB, full_bar(s), k0, nb0);
                } else {
                    if (args.gather)
                        tma_gather4(sa + lane * 512u, &tmA, full_bar(s), k0, rows[0], rows[1],
                                    rows[2], rows[3]);
                    else if (lane == 0)
                        tma_load_2d(sa, &tmA, full_bar(s), k0, m0);
                    if (lane == 0)
                        for (int j = 0; j < NSUB; ++j)
                            tma_load_2d(sb + j * Cfg::B_SUB_BYTES, &tmB, full_bar(s), k0, nb0 + j * BN);
                }
                pending = min(pending + 1, STAGES);
                if (++s == STAGES) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        if (!alive && leader) {
            // Drain: every issued stage's bytes land before shared memory is
            // released (for a pair the leader's barriers count both CTAs' bytes,
            // and the peer leaves only after the final cluster barrier).  The
            // waits are bounded again; a stage whose expected count can never
            // be met (the test hook) simply times out here.
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
        if (MX && !alive && lane == 0) {
            // (FP4) each CTA's scale rows land on its own barriers: drain those too
            int ds = s;
            uint32_t dph = ph;
            for (int i = 0; i < pending; ++i) {
                if (--ds < 0) {
                    ds = STAGES - 1;
                    dph ^= 1u;
                }
                wait_drain(sf_full_bar(ds), dph, 10000000ull);
            }
        }
    } else if (warp == 1 || (Cfg::ISS == 2 && warp == 6)) {
        // ------------------------------------------------------------ MMA issuers
        const int e = warp == 1 ? 0 : 1;  // issuer e takes the K blocks kb = e (mod kIss)
        if (lane == 0 && leader && e < kIss) {
            const uint32_t idesc = idesc_f16_f32acc(args.ab_bf16 != 0, Cfg::TILE_M, BN);
            const int32_t nkb = args.num_k_blocks;
            int s = 0;
            uint32_t ph = 0;
            int ab = 0;
            uint32_t aph = 0;
            bool alive = true;
            // K block kb of MMA half j on stage st into the accumulator at d_tmem
            // seeded accumulators (C written to TMEM by the epilogue) are
            // accumulated onto from the first K step on
            constexpr bool seeded = MODE == kModeSeed;
            auto issue_half = [&](int st, int32_t kb, int j, uint32_t d_tmem) {
                const uint64_t ad = sdesc_k_sw128(base + Cfg::OFF_A + st * Cfg::A_BYTES);
                const uint64_t bd =
                    sdesc_k_sw128(base + Cfg::OFF_B + st * Cfg::B_BYTES + j * Cfg::B_SUB_BYTES);
                const uint32_t dj = d_tmem + static_cast<uint32_t>(j * BN);
                if constexpr (MX != 0) {
                    // the stage's scale tiles into its TMEM columns, then four
                    // block-scaled MMAs of 32 bytes of K each; MMA k reads the
                    // scales of its 128-element chunk, the byte(s) its scale ids pick
                    const uint32_t sfc = base + Cfg::OFF_SFC + st * Cfg::SF_CP_BYTES;
                    const uint32_t sfcol = tmem_base + Cfg::SF_COL0 + st * Cfg::SF_COLS;
#pragma unroll
                    for (int ti = 0; ti < Cfg::SF_TILES; ++ti) {
                        if (PAIR)
                            tc_cp_32x128b_warpx4_pair(sfcol + 4u * ti, sdesc_rows16(sfc + 512u * ti));
                        else
                            tc_cp_32x128b_warpx4(sfcol + 4u * ti, sdesc_rows16(sfc + 512u * ti));
                    }
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        constexpr uint32_t kFmt = MX == 1 ? 1u : 5u;  // E2M1 in each kind's coding
                        const uint32_t chunk = (k * Cfg::MMA_K) / 128;
                        const uint32_t sfid = ((k * Cfg::MMA_K) % 128) / 32;
                        const uint32_t id = idesc_mx(kFmt, Cfg::TILE_M, BN, sfid, sfid);
                        const uint32_t sfa = sfcol + 4u * chunk;
                        const uint32_t sfb = sfcol + 4u * Cfg::SF_CHUNKS + 4u * Cfg::SF_B_ROWTILES * chunk;
                        const uint32_t acc = (kb | k) != 0 ? 1u : 0u;
                        if (MX == 1 && PAIR)
                            tc_mma_mxf4_pair(dj, ad + 2u * k, bd + 2u * k, id, sfa, sfb, acc);
                        else if (MX == 1)
                            tc_mma_mxf4(dj, ad + 2u * k, bd + 2u * k, id, sfa, sfb, acc);
                        else if (PAIR)
                            tc_mma_mxf8f6f4_pair(dj, ad + 2u * k, bd + 2u * k, id, sfa, sfb, acc);
                        else
                            tc_mma_mxf8f6f4(dj, ad + 2u * k, bd + 2u * k, id, sfa, sfb, acc);
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < Cfg::BK / 16; ++k) {  // +32 B per K=16 step
                        // (the first K step of this issuer's chain starts from zero)
                        if (PAIR)
                            tc_mma_f16_pair(dj, ad + 2u * k, bd + 2u * k, idesc,
                                            (seeded || ((kb / kIss) | k) != 0) ? 1u : 0u);
                        else
                            tc_mma_f16(dj, ad + 2u * k, bd + 2u * k, idesc,
                                       (seeded || ((kb / kIss) | k) != 0) ? 1u : 0u);
                    }
                }
            };
            // arrive on `bar` (both CTAs of a pair) once the MMAs issued so far finish
            auto commit_to = [&](uint32_t bar) {
                if (PAIR)
                    tc_commit_pair_multicast(bar, pair_mask);
                else
                    tc_commit(bar);
            };
            // a stage whose A slices came from the whole cluster is free only
            // once every CTA (every pair) of the cluster has consumed it
            auto free_stage = [&](int st) {
                if (MC > 1 && PAIR)
                    tc_commit_pair_multicast(empty_bar(st), kAllCtas);
                else if (MC > 1)
                    tc_commit_multicast(empty_bar(st), kAllCtas);
                else
                    commit_to(empty_bar(st));
            };
            // wait until stage s holds K block data; false if the kernel is aborting
            auto next_full = [&](int &st) {
                if (!wait_bounded<true>(full_bar(s), ph, abort_flag, args.status, args.timeout_ns,
                                  kWhereMmaFull))
                    return false;
                // (FP4: and for the scale warp(s) to have rearranged the stage's
                // scales; a pair's peer wrote its own, hence the cluster scope)
                if (MX && !(PAIR ? (mbar_probe_cluster(sf_bar(s), ph) ||
                                    wait_bounded_cluster(sf_bar(s), ph, abort_flag, args.status,
                                                         args.timeout_ns, kWhereMmaFull))
                                 : wait_bounded<true>(sf_bar(s), ph, abort_flag, args.status,
                                                      args.timeout_ns, kWhereMmaFull)))
                    return false;
                tc_fence_after_sync();
                st = s;
                if (++s == STAGES) {
                    s = 0;
                    ph ^= 1u;
                }
                return true;
            };
            auto wait_acc_free = [&](int b) {
                // (seeded: the epilogue's first arrival is the seed, so the first
                // use waits for it instead of passing on a fresh barrier)
                if (!wait_bounded<true>(acce_bar(b), seeded ? aph : aph ^ 1u, abort_flag, args.status,
                                  args.timeout_ns,
                                  kWhereMmaAccEmpty))
                    return false;
                tc_fence_after_sync();
                return true;
            };
            for (int32_t t = cta_set; t < args.num_tiles && alive; t += cta_sets) {
                if constexpr (NSUB == 1) {
                    if (!wait_acc_free(ab))
                        break;
                    const uint32_t d_tmem =
                        tmem_base + static_cast<uint32_t>((ab * kIss + e) * TILE_N);
                    for (int32_t kb = 0; kb < nkb; ++kb) {
                        if (kIss > 1 && kb % kIss != e) {
                            if (++s == STAGES) {  // the other issuer's stage
                                s = 0;
                                ph ^= 1u;
                            }
                            continue;
                        }
                        int st;
                        if (!next_full(st)) {
                            alive = false;
                            break;
                        }
                        issue_half(st, kb, 0, d_tmem);
                        free_stage(st);  // frees the stage (in both CTAs of a pair)
                    }
                    if (!alive)
                        break;
                    if (nkb <= e && !PAIR)
                        mbar_arrive(accf_bar(ab));  // nothing to multiply here
                    else
                        commit_to(accf_bar(ab));
                } else {
                    // Two halves of one accumulator, handed to the epilogue and back
                    // separately (barrier index = half).  At the start of a tile the
                    // half-1 MMAs of the first kFirst K blocks wait until the epilogue
                    // has drained half 1 of the previous tile; at the end, half 0 of
                    // the last kLast K blocks goes first so half 0 can be drained
                    // while half 1 finishes.  Both overlap drain time with MMA work.
                    constexpr int kFirst = STAGES / 2, kLast = STAGES / 2;
                    const uint32_t d_tmem = tmem_base;
                    const int32_t f = nkb < kFirst ? nkb : kFirst;
                    const int32_t l = (nkb - kLast) > f ? (nkb - kLast) : f;
                    int held[kFirst > kLast ? kFirst : kLast];
                    if (!wait_acc_free(0))
                        break;
                    for (int32_t kb = 0; kb < f && alive; ++kb) {
                        alive = next_full(held[kb]);
                        if (alive)
                            issue_half(held[kb], kb, 0, d_tmem);
                    }
                    if (!alive)
                        break;
                    if (f == nkb)
                        commit_to(accf_bar(0));  // all of half 0 is issued
                    if (!wait_acc_free(1))
                        break;
                    for (int32_t kb = 0; kb < f; ++kb) {
                        issue_half(held[kb], kb, 1, d_tmem);
                        free_stage(held[kb]);
                    }
                    for (int32_t kb = f; kb < l && alive; ++kb) {
                        int st;
                        alive = next_full(st);
                        if (alive) {
                            issue_half(st, kb, 0, d_tmem);
                            issue_half(st, kb, 1, d_tmem);
                            free_stage(st);
                        }
                    }
                    if (!alive)
                        break;
                    if (l < nkb) {
                        for (int32_t kb = l; kb < nkb && alive; ++kb) {
                            alive = next_full(held[kb - l]);
                            if (alive)
                                issue_half(held[kb - l], kb, 0, d_tmem);
                        }
                        if (!alive)
                            break;
                        commit_to(accf_bar(0));
                        for (int32_t kb = l; kb < nkb; ++kb) {
                            issue_half(held[kb - l], kb, 1, d_tmem);
                            free_stage(held[kb - l]);
                        }
                    } else if (f < nkb) {
                        commit_to(accf_bar(0));
                    }
                    commit_to(accf_bar(1));
                }
                if (++ab == Cfg::NUM_ACC) {
                    ab = 0;
                    aph ^= 1u;
                }
            }
        }
        __syncwarp();
    } else if (MX != 0 && warp == 6) {
        // ------------------------------------------------------------ scale warp
        // For every stage: wait for its loads, rearrange the scale rows as loaded
        // (row b of the stage: one byte per row of A, then of B) into 512-byte
        // tiles (row l + 32 q, block b at byte 16 l + 4 q + b) and hand them to
        // the MMA thread (tcgen05.cp reads them through the async proxy, hence
        // the fence).  Per tile, lane l loads the 32-bit words of rows 4l .. 4l+3
        // for its four blocks, transposes the 4 x 4 bytes so that each word
        // holds one row's four blocks, and stores row r's word at 16 (r % 32) +
        // 4 (r / 32).
        if constexpr (MX != 0) {
            int s = 0;
            uint32_t ph = 0;
            bool alive = true;
            for (int32_t t = cta_set; t < args.num_tiles && alive; t += cta_sets) {
                for (int32_t kb = 0; kb < args.num_k_blocks; ++kb) {
                    if (!warp_wait_bounded<true>(sf_full_bar(s), ph, abort_flag, args.status,
                                                 args.timeout_ns, kWhereMmaFull)) {
                        alive = false;
                        break;
                    }
                    const uint8_t *src = gbase + Cfg::OFF_SFS + s * Cfg::SF_STAGE_BYTES;
                    uint8_t *dst = gbase + Cfg::OFF_SFC + s * Cfg::SF_CP_BYTES;
                    uint32_t w[Cfg::SF_TILES][4];
#pragma unroll
                    for (int ti = 0; ti < Cfg::SF_TILES; ++ti) {
                        const bool a_tile = ti < Cfg::SF_CHUNKS;
                        const int c = a_tile ? ti : (ti - Cfg::SF_CHUNKS) / Cfg::SF_B_ROWTILES;
                        const int rt = a_tile ? 0 : (ti - Cfg::SF_CHUNKS) % Cfg::SF_B_ROWTILES;
                        const uint32_t pitch = a_tile ? Cfg::BM : Cfg::TILE_N;
                        const uint8_t *rows = src + (a_tile ? 0u : Cfg::SF_KB * Cfg::BM) + 128u * rt +
                                              4u * c * pitch + 4u * lane;
#pragma unroll
                        for (int b = 0; b < 4; ++b)
                            w[ti][b] = *reinterpret_cast<const uint32_t *>(rows + b * pitch);
                    }
#pragma unroll
                    for (int ti = 0; ti < Cfg::SF_TILES; ++ti) {
                        // w[b] byte i = block b of row 4 lane + i  ->  o[i] byte b
                        const uint32_t t0 = __byte_perm(w[ti][0], w[ti][1], 0x5140);
                        const uint32_t t1 = __byte_perm(w[ti][0], w[ti][1], 0x7362);
                        const uint32_t t2 = __byte_perm(w[ti][2], w[ti][3], 0x5140);
                        const uint32_t t3 = __byte_perm(w[ti][2], w[ti][3], 0x7362);
                        const uint32_t o[4] = {__byte_perm(t0, t2, 0x5410), __byte_perm(t0, t2, 0x7632),
                                               __byte_perm(t1, t3, 0x5410), __byte_perm(t1, t3, 0x7632)};
                        uint8_t *tile = dst + 512u * ti + 4u * (lane / 8u);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            *reinterpret_cast<uint32_t *>(tile + 16u * ((4u * lane + i) % 32u)) = o[i];
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if (PAIR && !leader)
                            mbar_arrive_cluster(lead(sf_bar(s)));
                        else
                            mbar_arrive(sf_bar(s));
                    }
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const uint32_t q = warp & 3u;  // TMEM lane quarter this warp may read
        const uint32_t buf0 = base + Cfg::OFF_EPI + q * 2u * Cfg::EPI_BUF;
        const bool has_c = args.has_c != 0;
        const bool c_tma = has_c && args.c_tma != 0;
        constexpr bool scatter = MODE == kModeScatter;
        constexpr bool reduce = MODE == kModeReduce;  // D += alpha * acc (float32 D, no C)
        constexpr bool seed = MODE == kModeSeed;      // accumulators start from C
        const bool acc_zero = !seed && args.num_k_blocks == 0;
        const int out_kind = args.out_kind;
        // A 32 x 32 box goes out from lane 0; scattered rows go out as eight
        // tile::scatter4 copies of four rows, lane g moving rows 4g .. 4g+3
        // (bulk groups belong to the issuing thread, so each waits for its own).
        const bool bulk_lane = lane < (scatter ? 8u : 1u);
        // C and D are touched once: their lines go first out of L2, so the A
        // and B panels that neighbouring tiles share stay resident
        const uint64_t epi_policy = l2_policy_evict_first();
        // The accumulator comes and goes back in units: the whole tile
        // (NSUB = 1, barrier index = ab) or each BN-wide half (NSUB = 2,
        // barrier index = half), so the MMA can refill half 0 while half 1
        // is still being drained.
        constexpr int kUnitChunks = (NSUB == 2 ? BN : TILE_N) / 32;
        // hand accumulator unit `unit` back to the MMA warp (of the leader CTA)
        auto release_unit = [&](int unit) {
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                if (PAIR && !leader)
                    mbar_arrive_cluster(lead(acce_bar(unit)));
                else
                    mbar_arrive(acce_bar(unit));
            }
        };
        // Seeded accumulators: write C of tile t (this warp's 32 rows, columns
        // 32c .. 32c+31 of the tile) into accumulator columns `col`, zero past
        // M and N, for the MMAs to accumulate onto.
        const bool c_vec = (reinterpret_cast<uintptr_t>(args.C) & 15u) == 0 && (args.ldc & 3) == 0;
        auto seed_chunk = [&](int32_t ts, int32_t c, uint32_t col) {
            int32_t smb, snb;
            tile_coords(ts, args, smb, snb);
            if (MC > 1)
                snb = snb * MC + static_cast<int32_t>(share);
            const int32_t row = smb * Cfg::TILE_M + static_cast<int32_t>(role) * Cfg::BM +
                                32 * static_cast<int32_t>(q) + static_cast<int32_t>(lane);
            const int32_t col0 = snb * TILE_N + 32 * c;
            uint32_t r[32];
            const float *crow = args.C + static_cast<int64_t>(row < args.M ? row : 0) * args.ldc + col0;
            if (row < args.M && col0 + 32 <= args.N && c_vec) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 x = *reinterpret_cast<const float4 *>(crow + 4 * i);
                    r[4 * i] = __float_as_uint(x.x);
                    r[4 * i + 1] = __float_as_uint(x.y);
                    r[4 * i + 2] = __float_as_uint(x.z);
                    r[4 * i + 3] = __float_as_uint(x.w);
                }
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    r[i] = __float_as_uint((row < args.M && col0 + i < args.N) ? crow[i] : 0.f);
            }
            tc_st_32x32b_x32(tmem_base + ((32u * q) << 16) + col, r);
        };
        if (seed) {
            // the first tiles on each accumulator start from C as well
            for (int b = 0; b < Cfg::NUM_ACC; ++b) {
                const int32_t tb = cta_set + b * cta_sets;
                for (int32_t c = 0; c < TILE_N / 32; ++c) {
                    if (tb < args.num_tiles)
                        seed_chunk(tb, c, static_cast<uint32_t>(b * TILE_N + 32 * c));
                    if (c % kUnitChunks == kUnitChunks - 1) {
                        tc_wait_st();
                        release_unit(NSUB == 2 ? c / kUnitChunks : b);
                    }
                }
            }
        }
        int ab = 0;
        uint32_t aph = 0;
        uint32_t cph[2] = {0u, 0u};
        bool alive = true;
        for (int32_t t = cta_set; t < args.num_tiles && alive; t += cta_sets) {
            int32_t mb, nb;
            tile_coords(t, args, mb, nb);
            if (MC > 1)
                nb = nb * MC + static_cast<int32_t>(share);
            const int32_t m0 = mb * Cfg::TILE_M + static_cast<int32_t>(role) * Cfg::BM;
            const int32_t n0 = nb * TILE_N;
            const int32_t row0 = m0 + 32 * (int32_t)q;
            const bool rows_ok = row0 < args.M;
            // (MC > 1: a CTA past the last column block still takes part in the
            // cluster's loads and MMAs, and writes nothing)
            const int32_t nchunks = max(0, min(TILE_N / 32, (args.N - n0 + 31) / 32));
            const int32_t my_row = row0 + (int32_t)lane;

            // Row of C and D for this lane: my_row, or idx[my_row] when the
            // rows are scattered; -1 where nothing is written (past M, or an
            // index outside D).
            int32_t d_row = my_row < args.M ? my_row : -1;
            int32_t grp_rows[4] = {0, 0, 0, 0};  // the four rows lane g < 8 moves
            bool own_group_whole = true, issue_group_whole = true;
            if (scatter && rows_ok) {
                if (d_row >= 0) {
                    const int32_t v = args.idx[d_row];
                    if (v < 0 || v >= args.d_rows) {
                        record_error(args.status, kStatusIndex, 0);
                        d_row = -1;
                    } else {
                        d_row = v;
                    }
                }
                // a group of four rows goes out by one scatter4 only when all
                // four are written; otherwise its lanes store their own rows
                const uint32_t written = __ballot_sync(0xffffffffu, d_row >= 0);
                own_group_whole = ((written >> (lane & ~3u)) & 0xFu) == 0xFu;
                issue_group_whole = ((written >> (4u * (lane & 7u))) & 0xFu) == 0xFu;
#pragma unroll
                for (int r = 0; r < 4; ++r)  // (rows not written read row 0 of C, unused)
                    grp_rows[r] = __shfl_sync(0xffffffffu, d_row < 0 ? 0 : d_row,
                                              4 * static_cast<int>(lane & 7u) + r);
            }

            // the C box of columns [col, col + 32) into buffer j (warp-wide call)
            auto load_c = [&](int j, int32_t col) {
                const uint32_t dst = buf0 + j * Cfg::EPI_BUF;
                if (lane == 0)
                    mbar_arrive_expect_tx(c_bar(q, j), Cfg::EPI_BUF);
                if (!scatter) {
                    if (lane == 0) {
                        if (TCG_EPI_EVICT_FIRST)
                            tma_load_2d_hint(dst, &tmC, c_bar(q, j), col, row0, epi_policy);
                        else
                            tma_load_2d(dst, &tmC, c_bar(q, j), col, row0);
                    }
                } else {
                    __syncwarp();
                    if (lane < 8)
                        tma_gather4_hint(dst + 512u * lane, &tmC, c_bar(q, j), col, grp_rows[0],
                                         grp_rows[1], grp_rows[2], grp_rows[3], epi_policy);
                }
            };
            // plain stores (reduce: float32 atomic adds) of this lane's row,
            // column by column, nothing past column N
            auto store_direct = [&](const float(&v)[32], int32_t col0) {
                if (d_row < 0)
                    return;
                const int64_t o = static_cast<int64_t>(d_row) * args.ldd + col0;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    if (col0 + i < args.N) {
                        if (reduce)
                            atomicAdd(static_cast<float *>(args.D) + o + i, v[i]);
                        else if (out_kind == kOutF32)
                            static_cast<float *>(args.D)[o + i] = v[i];
                        else if (out_kind == kOutBF16)
                            static_cast<unsigned short *>(args.D)[o + i] = f32_to_bf16_rn(v[i]);
                        else
                            static_cast<unsigned short *>(args.D)[o + i] = f32_to_f16_rn(v[i]);
                    }
                }
            };

            if (bulk_lane)
                bulk_wait_group_read<0>();  // last tile's stores are done with the buffers
            __syncwarp();
            if (c_tma && rows_ok) {
                for (int j = 0; j < 2 && j < nchunks; ++j)
                    load_c(j, n0 + 32 * j);
            }
            bool zero_row = acc_zero;
            if (args.gather && my_row < args.M) {
                const int32_t v = args.idx[my_row];
                zero_row = zero_row || v < 0 || v >= args.table_rows;
            }

            // the next tile on this accumulator (seeded mode)
            const int32_t t_next = t + Cfg::NUM_ACC * cta_sets;
            for (int32_t c = 0; c < TILE_N / 32; ++c) {
                const int unit = NSUB == 2 ? c / kUnitChunks : ab;
                if (c % kUnitChunks == 0) {
                    if (!warp_wait_bounded<true>(accf_bar(unit), aph, abort_flag, args.status,
                                           args.timeout_ns, kWhereEpiAccFull)) {
                        alive = false;
                        break;
                    }
                    tc_fence_after_sync();
                }
                const bool have = c < nchunks;
                uint32_t acc[32];
                if (have) {
                    const uint32_t col = static_cast<uint32_t>(ab * kIss * TILE_N + 32 * c);
                    tc_ld_32x32b_x32(tmem_base + ((32u * q) << 16) + col, acc);
                    tc_wait_ld(acc);
                    if (kIss > 1 && args.num_k_blocks > 1) {
                        // the second issuer's partial sum (odd K blocks)
                        uint32_t acc2[32];
                        tc_ld_32x32b_x32(tmem_base + ((32u * q) << 16) + col + TILE_N, acc2);
                        tc_wait_ld(acc2);
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            acc[i] = __float_as_uint(__fadd_rn(__uint_as_float(acc[i]), __uint_as_float(acc2[i])));
                    }
                }
                // seeded mode: these columns are read, so the next tile's C can
                // take their place
                if (seed && t_next < args.num_tiles)
                    seed_chunk(t_next, c, static_cast<uint32_t>(ab * TILE_N + 32 * c));
                if (c % kUnitChunks == kUnitChunks - 1) {
                    // this unit of the accumulator is fully read: hand it back
                    if (seed)
                        tc_wait_st();
                    release_unit(unit);
                }
                if (!have || !rows_ok)
                    continue;
                const int j = c & 1;
                const uint32_t buf = buf0 + j * Cfg::EPI_BUF;
                const int32_t col0 = n0 + 32 * c;
                // plain stores: D not TMA-aligned, the 16-byte chunk that
                // straddles column N, or (scattered rows) any partial chunk
                const bool d_direct = !args.d_tma ||
                                      ((args.d_tail_direct || scatter) && col0 + 32 > args.N);
                float v[32];
                if (c_tma) {
                    if (!warp_wait_bounded<true>(c_bar(q, j), cph[j], abort_flag, args.status,
                                           args.timeout_ns, kWhereEpiC)) {
                        alive = false;
                        break;
                    }
                    cph[j] ^= 1u;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        uint32_t x[4];
                        ld_shared_v4(buf + swz_off(lane, i, 128u), x[0], x[1], x[2], x[3]);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float a = zero_row ? 0.f : __uint_as_float(acc[4 * i + e]);
                            v[4 * i + e] = fma_rn(args.alpha, a, mul_rn(args.beta, __uint_as_float(x[e])));
                        }
                    }
                } else if (has_c) {
                    const float *crow = args.C + static_cast<int64_t>(d_row < 0 ? 0 : d_row) * args.ldc;
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float cv = (d_row >= 0 && col0 + i < args.N) ? crow[col0 + i] : 0.f;
                        const float a = zero_row ? 0.f : __uint_as_float(acc[i]);
                        v[i] = fma_rn(args.alpha, a, mul_rn(args.beta, cv));
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        v[i] = mul_rn(args.alpha, zero_row ? 0.f : __uint_as_float(acc[i]));
                }
                if (d_direct) {
                    store_direct(v, col0);
                } else {
                    if (!c_tma && bulk_lane)
                        bulk_wait_group_read<1>();  // the store two chunks back left buffer j
                    __syncwarp();  // all of C read (in-place D) and buffer j free
                    if (out_kind == kOutF32) {
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            st_shared_v4(buf + swz_off(lane, i, 128u), __float_as_uint(v[4 * i]),
                                         __float_as_uint(v[4 * i + 1]), __float_as_uint(v[4 * i + 2]),
                                         __float_as_uint(v[4 * i + 3]));
                    } else if (out_kind == kOutBF16) {
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            st_shared_v4(buf + swz_off(lane, i, 64u), pack_bf16x2(v[8 * i], v[8 * i + 1]),
                                         pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                                         pack_bf16x2(v[8 * i + 4], v[8 * i + 5]),
                                         pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
                    } else {
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            st_shared_v4(buf + swz_off(lane, i, 64u), pack_f16x2(v[8 * i], v[8 * i + 1]),
                                         pack_f16x2(v[8 * i + 2], v[8 * i + 3]),
                                         pack_f16x2(v[8 * i + 4], v[8 * i + 5]),
                                         pack_f16x2(v[8 * i + 6], v[8 * i + 7]));
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (!scatter) {
                        if (lane == 0) {
                            if (reduce)
                                tma_reduce_add_2d_hint(&tmD, buf, col0, row0, epi_policy);
                            else if (TCG_EPI_EVICT_FIRST)
                                tma_store_2d_hint(&tmD, buf, col0, row0, epi_policy);
                            else
                                tma_store_2d(&tmD, buf, col0, row0);
                            bulk_commit_group();
                        }
                    } else {
                        // (scattered rows use TMA stores only for 128-byte rows:
                        // float32 output, 128-byte swizzled image)
                        if (lane < 8) {
                            if (issue_group_whole)
                                tma_scatter4_hint(&tmD, buf + 512u * lane, col0, grp_rows[0],
                                                  grp_rows[1], grp_rows[2], grp_rows[3], epi_policy);
                            bulk_commit_group();
                        }
                        if (!own_group_whole)
                            store_direct(v, col0);
                    }
                }
                if (c_tma && c + 2 < nchunks) {
                    if (bulk_lane)
                        bulk_wait_group_read<0>();  // the store of this chunk is done with buffer j
                    __syncwarp();
                    load_c(j, n0 + 32 * (c + 2));
                }
                __syncwarp();
            }
            if (!alive)
                break;
            if (++ab == Cfg::NUM_ACC) {
                ab = 0;
                aph ^= 1u;
            }
        }
        if (!alive && c_tma && lane == 0) {
            // C loads issued for this tile may still be landing: let them finish
            for (int j = 0; j < 2; ++j)
                wait_drain(c_bar(q, j), cph[j], 10000000ull);
        }
        if (bulk_lane)
            bulk_wait_group_all();
        __syncwarp();
    }

    tc_fence_before_sync();
    if (PAIR) {
        if (threadIdx.x == 0 && *abort_flag)
            raise_abort();  // the peer stops waiting instead of running out of time itself
        if (*abort_flag && !leader) {
            // copies this CTA issued report to the leader's barriers, which the
            // leader drains; give any still in flight time to land as well
            const uint64_t t0 = global_timer_ns();
            while (global_timer_ns() - t0 < 100000ull) {
            }
        }
    }
    if (CL > 1)
        cluster_sync_all();  // the leader's MMAs read this CTA's shared memory, and peers
                             // may multicast into it, until here
    else
        __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        if (PAIR)
            tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
        else
            tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
    // a co-launched tail completes only after the kernel beside it, so the next
    // kernel in the stream, which waits for this grid, waits for both
    if (args.co_tail)
        grid_dependency_wait();
}

}  // namespace tcg
