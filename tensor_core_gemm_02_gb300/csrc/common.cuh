// common.cuh -- kernel arguments, the device status word, bounded waits and
// the persistent tile order shared by the GEMM kernels.
#pragma once

#include <stdint.h>

#include "ptx.cuh"

namespace tcg {

// Device status codes (same values as gemm_status in include/tcgemm.h).
enum : uint32_t { kStatusTimeout = 6u, kStatusIndex = 7u };

// Where a wait gave up (stored in status[1] next to the code, for diagnosis).
enum : uint32_t {
    kWhereProducerEmpty = 1,
    kWhereMmaFull = 2,
    kWhereMmaAccEmpty = 3,
    kWhereEpiAccFull = 4,
    kWhereEpiC = 5,
};

enum : int32_t { kOutF32 = 0, kOutBF16 = 1, kOutF16 = 2 };

struct GemmArgs {
    int32_t M, N, K;
    int32_t num_m_blocks, num_n_blocks, num_k_blocks;
    int32_t num_tiles;      // output tiles
    int32_t group_m;        // tile-order group height (in m blocks)
    int32_t splits;         // K slices per tile (skinny kernel)
    int32_t sk_tiles;       // skinny kernel: tiles shared block by block (the rest go whole)
    float alpha, beta;
    int32_t has_c;          // C is read (non-NULL and beta != 0)
    int32_t out_kind;       // kOutF32 / kOutBF16 / kOutF16
    int32_t ab_bf16;        // operand format: 1 bf16, 0 f16
    int32_t gather;         // A rows are table[idx[m]]
    int32_t c_tma;          // C boxes come through TMA (aligned C); else plain loads
    int32_t d_tma;          // D boxes go out through TMA stores (aligned D); else plain stores
    int32_t d_tail_direct;  // N * sizeof(out) is not a multiple of 16: a TMA store would
                            // write the whole 16-byte chunk that straddles column N, so the
                            // chunk that crosses N is stored with plain stores instead
    const int32_t *idx;     // gathered A rows, or scattered C/D rows
    int32_t table_rows;     // rows of the gather table
    int32_t scatter;        // row m of the result goes to row idx[m] of D (and reads C there)
    int32_t d_rows;         // rows of C and D when scattering
    int32_t reduce;         // D += alpha * acc (float32 adds into D; no C)
    int32_t seed;           // the accumulator starts from C (written to TMEM before the
                            // first MMA, which then accumulates); D = acc, C not read after
    int32_t co_tail;        // launched right behind the previous kernel onto the SMs it
                            // left idle: no dependency wait at the start, one at the end
    uint32_t extra_tx;      // test hook: extra bytes expected on the first stage
    uint32_t *status;       // [0] first error code, [1] where a wait gave up
    uint64_t timeout_ns;    // limit of every bounded wait
    // plain-load / plain-store epilogue paths
    const float *C;
    int64_t ldc;
    void *D;
    int64_t ldd;
    float *workspace;       // per-split partial tiles
    uint32_t *counters;     // per-tile arrival counters (zero between calls)
};

__device__ __forceinline__ void record_error(uint32_t *status, uint32_t code, uint32_t where)
{
    if (atomicCAS(status, 0u, code) == 0u)
        status[1] = where;
}

// Wait for phase `parity` of `bar`, giving up after `timeout_ns` or when the
// CTA-wide abort flag is raised.  Returns false when it gave up; the first
// thread to time out raises the abort flag and records the error.  (The loop,
// out of line; wait_bounded below tries the barrier inline first.)
static __device__ __noinline__ bool wait_bounded_loop(uint32_t bar, uint32_t parity,
                                          volatile uint32_t *abort_flag, uint32_t *status,
                                          uint64_t timeout_ns, uint32_t where)
{
    if (mbar_test(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_test(bar, parity))
            return true;
        if ((it & 63u) == 0u) {
            if (*abort_flag)
                return false;
            if (global_timer_ns() - t0 > timeout_ns) {
                *abort_flag = 1u;
                record_error(status, kStatusTimeout, where);
                return false;
            }
        }
    }
}

// kProbe: try the barrier inline first, so that a phase which has already
// completed costs one probe instead of a call (whose register saves cost
// hundreds of cycles per wait in the warp-specialised loops).  Worth it where
// the phase has usually completed; where the waiting thread is usually early
// and on the critical path (an MMA issuer waiting for HBM), the probe only
// adds to each wait and the loop is called directly.
template <bool kProbe = false>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity,
                                             volatile uint32_t *abort_flag, uint32_t *status,
                                             uint64_t timeout_ns, uint32_t where)
{
    if constexpr (kProbe) {
        if (mbar_probe(bar, parity))
            return true;
    }
    return wait_bounded_loop(bar, parity, abort_flag, status, timeout_ns, where);
}

// As wait_bounded, with the barrier read as an acquire at cluster scope (for
// phases that the other CTA of a pair completes after writing its shared memory).
static __device__ __noinline__ bool wait_bounded_cluster(uint32_t bar, uint32_t parity,
                                                         volatile uint32_t *abort_flag, uint32_t *status,
                                                         uint64_t timeout_ns, uint32_t where)
{
    if (mbar_test_cluster(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_test_cluster(bar, parity))
            return true;
        if ((it & 63u) == 0u) {
            if (*abort_flag)
                return false;
            if (global_timer_ns() - t0 > timeout_ns) {
                *abort_flag = 1u;
                record_error(status, kStatusTimeout, where);
                return false;
            }
        }
    }
}

// Teardown after an abort: wait (bounded, ignoring the abort flag) for copies
// this thread issued to land before the CTA releases its shared memory.
static __device__ __noinline__ bool wait_drain(uint32_t bar, uint32_t parity, uint64_t timeout_ns)
{
    const uint64_t t0 = global_timer_ns();
    while (!mbar_test(bar, parity)) {
        if (global_timer_ns() - t0 > timeout_ns)
            return false;
    }
    return true;
}

// Every lane of the warp waits (bounded); the warp then agrees on the result
// so that no lane runs ahead into a warp-collective instruction alone.
template <bool kProbe = false>
__device__ __forceinline__ bool warp_wait_bounded(uint32_t bar, uint32_t parity,
                                                  volatile uint32_t *abort_flag,
                                                  uint32_t *status, uint64_t timeout_ns,
                                                  uint32_t where)
{
    if constexpr (kProbe) {
        if (__all_sync(0xffffffffu, mbar_probe(bar, parity)))
            return true;
    }
    const bool ok = wait_bounded_loop(bar, parity, abort_flag, status, timeout_ns, where);
    return __all_sync(0xffffffffu, ok);
}

// As warp_wait_bounded, with the loop inline: loads the waiting threads
// still have in flight stay in flight (around a call, the live registers are
// saved first, and saving a register waits for the load that fills it).
__device__ __forceinline__ bool warp_wait_bounded_inline(uint32_t bar, uint32_t parity,
                                                         volatile uint32_t *abort_flag,
                                                         uint32_t *status, uint64_t timeout_ns,
                                                         uint32_t where)
{
    bool ok = true;
    if (!mbar_test(bar, parity)) {
        const uint64_t t0 = global_timer_ns();
        for (uint32_t it = 1;; ++it) {
            if (mbar_test(bar, parity))
                break;
            if ((it & 63u) == 0u) {
                if (*abort_flag) {
                    ok = false;
                    break;
                }
                if (global_timer_ns() - t0 > timeout_ns) {
                    *abort_flag = 1u;
                    record_error(status, kStatusTimeout, where);
                    ok = false;
                    break;
                }
            }
        }
    }
    return __all_sync(0xffffffffu, ok);
}

// Persistent tile order: output tiles in M, N order (the pages' repeat order
// puts M before N and K innermost), visited in groups of `group_m` block rows
// so that CTAs running at the same time share A and B panels in L2.
__device__ __forceinline__ void tile_coords(int32_t t, const GemmArgs &a, int32_t &mb,
                                            int32_t &nb)
{
    const int32_t per_group = a.group_m * a.num_n_blocks;
    const int32_t g = t / per_group;
    const int32_t first_m = g * a.group_m;
    const int32_t rows = min(a.num_m_blocks - first_m, a.group_m);
    const int32_t r = t - g * per_group;
    mb = first_m + r % rows;
    nb = r / rows;
}

}  // namespace tcg
