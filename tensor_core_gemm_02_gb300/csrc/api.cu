// api.cu -- the C ABI declared in include/tcgemm.h: argument validation,
// TMA descriptor encoding (with a small cache), kernel choice and launch, and
// the per-device status word.
//
// Validation follows the descriptor legality rule of the "cp.async.bulk.tensor"
// page (section "Operands and descriptor fields"): unit innermost stride,
// 16-byte aligned bases and row pitches; invalid fields are rejected, never
// promoted or reinterpreted.  Every check runs before any CUDA call, so it
// needs no GPU.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "host_internal.h"

// Fewest K blocks a CTA of the skinny kernel is given (when there are fewer
// than SMs x this many blocks, fewer CTAs run).  Measured per launch from a
// replayed CUDA graph: 1 -> 8 takes 64 x 512 x 512 from 16.4 to 11.1 us and
// 32 x 8192 x 1024 from 13.3 to 10.2 us; 4 and 16 were each worse on some
// shapes; 16 x 28672 x 4096 is unchanged.
#ifndef TCG_SKINNY_MIN_KB
#define TCG_SKINNY_MIN_KB 8
#endif

// Height, in block rows, of the groups the tile order walks through (L2 reuse).
#ifndef TCG_GROUP_M
#define TCG_GROUP_M 16
#endif

// First device-side error code [0] and where it arose [1], one per device.
static __device__ uint32_t g_device_status[4];

namespace tcg {
namespace host {

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;


std::mutex g_ws_mu;
std::vector<Workspace> g_ws;

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::atomic<uint64_t> g_timeout_ns{kDefaultTimeoutNs};
std::atomic<int> g_inject{0};
std::atomic<int> g_force_kernel{0};  // test hook: 0 automatic, 1 single CTAs, 3 CTA pairs
std::atomic<int> g_force_bn{0};

gemm_status device_info(DeviceInfo **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices)
        return GEMM_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceInfo &d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return GEMM_ERR_CUDA;
        if (major != 10 || minor != 3)
            return GEMM_ERR_UNSUPPORTED;  // kernels are built for sm_103a only
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess)
            return GEMM_ERR_CUDA;
        if (!g_encode) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q) != cudaSuccess ||
                q != cudaDriverEntryPointSuccess || !fn)
                return GEMM_ERR_CUDA;
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        d.index = dev;
        d.sm_count = sms;
        d.status = static_cast<uint32_t *>(p);
        d.ready = true;
    }
    *out = &d;
    return GEMM_OK;
}

// Workspace of (device, stream) with room for `bytes` of partials and `count`
// counters; grows geometrically.  New counters start at zero; the kernel
// returns every counter it uses to zero.
gemm_status get_workspace(int device, cudaStream_t stream, size_t bytes, size_t count,
                          Workspace *out)
{
    std::lock_guard<std::mutex> lock(g_ws_mu);
    Workspace *w = nullptr;
    for (Workspace &x : g_ws)
        if (x.device == device && x.stream == stream)
            w = &x;
    if (!w) {
        g_ws.push_back(Workspace{});
        w = &g_ws.back();
        w->device = device;
        w->stream = stream;
    }
    if (w->partial_bytes < bytes || w->counter_count < count) {
        if (w->partials || w->counters) {
            // earlier kernels on this stream may still use the old buffers
            if (cudaStreamSynchronize(stream) != cudaSuccess)
                return GEMM_ERR_CUDA;
            cudaFree(w->partials);
            cudaFree(w->counters);
            w->partials = nullptr;
            w->counters = nullptr;
        }
        const size_t nb = bytes > 2 * w->partial_bytes ? bytes : 2 * w->partial_bytes;
        const size_t nc = count > 2 * w->counter_count ? count : 2 * w->counter_count;
        w->partial_bytes = 0;
        w->counter_count = 0;
        if (cudaMalloc(&w->partials, nb > 0 ? nb : 256) != cudaSuccess)
            return GEMM_ERR_CUDA;
        if (cudaMalloc(&w->counters, nc * sizeof(uint32_t)) != cudaSuccess)
            return GEMM_ERR_CUDA;
        if (cudaMemsetAsync(w->counters, 0, nc * sizeof(uint32_t), stream) != cudaSuccess)
            return GEMM_ERR_CUDA;
        w->partial_bytes = nb;
        w->counter_count = nc;
    }
    *out = *w;
    return GEMM_OK;
}

// After a kernel gave up half way, counters may be left non-zero: clear them.
gemm_status reset_workspaces(int device)
{
    std::lock_guard<std::mutex> lock(g_ws_mu);
    for (Workspace &x : g_ws)
        if (x.device == device && x.counters &&
            cudaMemset(x.counters, 0, x.counter_count * sizeof(uint32_t)) != cudaSuccess)
            return GEMM_ERR_CUDA;
    return GEMM_OK;
}

// ------------------------------------------------------------- descriptors

struct MapKey {
    uint64_t ptr, inner, outer, stride;
    uint32_t box_inner, box_outer, dtype, swizzle;
    bool operator==(const MapKey &o) const { return std::memcmp(this, &o, sizeof(*this)) == 0; }
};

struct MapSlot {
    bool used = false;
    MapKey key{};
    CUtensorMap map{};
};

constexpr int kCacheSlots = 1024;
MapSlot g_cache[kCacheSlots];
std::mutex g_cache_mu;

uint64_t hash_key(const MapKey &k)
{
    uint64_t h = 1469598103934665603ull;
    const unsigned char *p = reinterpret_cast<const unsigned char *>(&k);
    for (size_t i = 0; i < sizeof(k); ++i) {
        h ^= p[i];
        h *= 1099511628211ull;
    }
    return h;
}

// A 2-D row-major tensor: `inner` contiguous elements per row, `outer` rows
// `stride_bytes` apart, copied in boxes of box_inner x box_outer.
bool encode_2d(CUtensorMap *m, CUtensorMapDataType dtype, const void *ptr, uint64_t inner,
               uint64_t outer, uint64_t stride_bytes, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle swizzle)
{
    MapKey key;
    std::memset(&key, 0, sizeof(key));
    key.ptr = reinterpret_cast<uint64_t>(ptr);
    key.inner = inner;
    key.outer = outer;
    key.stride = stride_bytes;
    key.box_inner = box_inner;
    key.box_outer = box_outer;
    key.dtype = static_cast<uint32_t>(dtype);
    key.swizzle = static_cast<uint32_t>(swizzle);
    const int slot = static_cast<int>(hash_key(key) % kCacheSlots);
    {
        std::lock_guard<std::mutex> lock(g_cache_mu);
        if (g_cache[slot].used && g_cache[slot].key == key) {
            *m = g_cache[slot].map;
            return true;
        }
    }
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {stride_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, dtype, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return false;
    std::lock_guard<std::mutex> lock(g_cache_mu);
    g_cache[slot].used = true;
    g_cache[slot].key = key;
    g_cache[slot].map = *m;
    return true;
}

// ------------------------------------------------------------- validation

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// bytes spanned by a rows x cols matrix with leading dimension ld
uint64_t span_bytes(int64_t rows, int64_t cols, int64_t ld, int64_t esize)
{
    if (rows <= 0 || cols <= 0)
        return 0;
    return static_cast<uint64_t>(((rows - 1) * ld + cols) * esize);
}

bool overlap(const void *a, uint64_t an, const void *b, uint64_t bn)
{
    if (!a || !b || an == 0 || bn == 0)
        return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bn && b0 < a0 + an;
}

int out_size(int out) { return out == GEMM_OUT_F32 ? 4 : 2; }


gemm_status validate(const Problem &p, bool *empty)
{
    *empty = false;
    if (p.M < 0 || p.N < 0 || p.K < 0 || p.a_rows < 0 || p.d_rows < 0)
        return GEMM_ERR_INVALID_ARG;
    if (p.out != GEMM_OUT_F32 && p.out != GEMM_OUT_BF16 && p.out != GEMM_OUT_F16)
        return GEMM_ERR_INVALID_ARG;
    if (p.M > kMaxDim || p.N > kMaxDim || p.K > kMaxDim || p.a_rows > kMaxDim)
        return GEMM_ERR_UNSUPPORTED;
    if (p.M == 0 || p.N == 0) {
        *empty = true;
        return GEMM_OK;
    }
    const bool c_used = p.C != nullptr && p.beta != 0.0f;
    if (!p.D)
        return GEMM_ERR_INVALID_ARG;
    if (p.K > 0 && (!p.A || !p.B))
        return GEMM_ERR_INVALID_ARG;
    if (p.gather && (!p.idx || p.a_rows < 1))
        return GEMM_ERR_INVALID_ARG;
    if (p.scatter && (!p.idx || p.d_rows < 1 || p.gather))
        return GEMM_ERR_INVALID_ARG;
    if (p.reduce && (p.out != GEMM_OUT_F32 || p.gather || p.scatter))
        return GEMM_ERR_INVALID_ARG;
    if (p.seed && (!p.C || p.gather || p.scatter || p.reduce))
        return GEMM_ERR_INVALID_ARG;
    if (p.w4) {
        if (!p.bf16 || p.gather || p.scatter || p.reduce || p.seed)
            return GEMM_ERR_INVALID_ARG;
        if (p.K % 32 != 0)
            return GEMM_ERR_UNSUPPORTED;  // whole scale blocks only
        if (p.K > 0 && (!p.bscale || p.ldbs < p.N))
            return GEMM_ERR_INVALID_ARG;
        if (p.ldbs > kMaxDim)
            return GEMM_ERR_UNSUPPORTED;
    }
    // B: N rows of K 16-bit elements, or (FP4) of K / 2 bytes
    const int64_t b_cols = p.w4 ? p.K / 2 : p.K;
    const int64_t b_esize = p.w4 ? 1 : 2;
    if (p.d_rows > kMaxDim)
        return GEMM_ERR_UNSUPPORTED;
    // rows of C and D: M, or the rows of the matrix the result is scattered into
    const int64_t out_rows = p.scatter ? p.d_rows : p.M;
    if (p.ldd < p.N)
        return GEMM_ERR_INVALID_ARG;
    if (c_used && p.ldc < p.N)
        return GEMM_ERR_INVALID_ARG;
    if (p.K > 0 && (p.lda < p.K || p.ldb < b_cols))
        return GEMM_ERR_INVALID_ARG;
    if (p.lda > kMaxDim || p.ldb > kMaxDim || p.ldc > kMaxDim || p.ldd > kMaxDim)
        return GEMM_ERR_UNSUPPORTED;
    // alignment: 16-byte bases, row pitches that are multiples of 16 bytes
    if (p.K > 0 &&
        (!aligned16(p.A) || !aligned16(p.B) || (p.lda * 2) % 16 || (p.ldb * b_esize) % 16))
        return GEMM_ERR_ALIGNMENT;
    // C and D only need their natural element alignment: when their base or
    // row pitch is not 16-byte aligned the epilogue uses plain loads/stores
    if (c_used && (reinterpret_cast<uintptr_t>(p.C) & 3u))
        return GEMM_ERR_ALIGNMENT;
    if (reinterpret_cast<uintptr_t>(p.D) & static_cast<uintptr_t>(out_size(p.out) - 1))
        return GEMM_ERR_ALIGNMENT;
    if ((p.gather || p.scatter) && (reinterpret_cast<uintptr_t>(p.idx) & 3u))
        return GEMM_ERR_ALIGNMENT;
    // aliasing: D may only coincide exactly with C (fp32 in-place update)
    const uint64_t d_span = span_bytes(out_rows, p.N, p.ldd, out_size(p.out));
    if (p.K > 0) {
        if (overlap(p.D, d_span, p.A, span_bytes(p.a_rows, p.K, p.lda, 2)))
            return GEMM_ERR_ALIAS;
        if (overlap(p.D, d_span, p.B, span_bytes(p.N, b_cols, p.ldb, b_esize)))
            return GEMM_ERR_ALIAS;
        if (p.w4 && overlap(p.D, d_span, p.bscale, span_bytes(p.K / 32, p.N, p.ldbs, 1)))
            return GEMM_ERR_ALIAS;
    }
    if ((p.gather || p.scatter) && overlap(p.D, d_span, p.idx, static_cast<uint64_t>(p.M) * 4))
        return GEMM_ERR_ALIAS;
    if (c_used && overlap(p.D, d_span, p.C, span_bytes(out_rows, p.N, p.ldc, 4))) {
        const bool exact_in_place = static_cast<const void *>(p.C) == p.D &&
                                    p.out == GEMM_OUT_F32 && p.ldc == p.ldd;
        if (!exact_in_place)
            return GEMM_ERR_ALIAS;
    }
    return GEMM_OK;
}

// ------------------------------------------------------------- planning

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Tile shape for the tile kernel.  Candidates: single CTAs with 128 x {256,
// 128, 64} tiles; CTA pairs with 256 x 256 tiles (two accumulators, so the
// epilogue overlaps the next tile); CTA pairs with 256 x 512 tiles (each row
// of A feeds twice the work, one accumulator); clusters of four single CTAs
// sharing A by multicast (gathered rows only).  Cost = waves of persistent
// CTA sets x per-SM tile width plus a fixed per-tile cost.  Pairs get a 10%
// credit (each SM moves 2/3 of the operand bytes); the 256 x 512 form gets a
// further 5% when its epilogue is short relative to the tile (no C, not
// scattered, K >= 2048) and is always preferred for gathered rows, whose cost
// is the number of TMA gather4 issues per flop.  (Scattered rows: 16384 rows,
// N = K = 4096, f32 out: 256 x 256 pairs 0.326 ms, 256 x 512 pairs 0.355 ms --
// eight scatter4 issues per 32-column chunk make the epilogue long enough that
// it must overlap the next tile's mainloop, which needs two accumulators.)
struct TileChoice {
    int kernel;  // 1 single, 3 pair 256, 4 pair 512
    int bn;
};

TileChoice choose_tile(int64_t M, int64_t N, int64_t K, bool gather, bool c_used, bool scatter,
                       int sm_count)
{
    static const int widths[3] = {256, 128, 64};
    TileChoice best{1, 256};
    double best_cost = -1.0;
    for (int w : widths) {
        const int64_t tiles = ceil_div(M, 128) * ceil_div(N, w);
        const double cost = static_cast<double>(ceil_div(tiles, sm_count) * (w + 32));
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = TileChoice{1, w};
        }
    }
    const int pairs = sm_count / 2;
    if (K == 0 || pairs == 0)
        return best;
    const int64_t tiles256 = ceil_div(M, 256) * ceil_div(N, 256);
    const double cost256 = 0.9 * static_cast<double>(ceil_div(tiles256, pairs) * (256 + 32));
    if (cost256 <= best_cost) {
        best_cost = cost256;
        best = TileChoice{3, 256};
    }
    if (N > 256) {
        const int64_t tiles512 = ceil_div(M, 256) * ceil_div(N, 512);
        double cost512 = 0.9 * static_cast<double>(ceil_div(tiles512, pairs) * (512 + 64));
        if (!c_used && !scatter && K >= 2048)
            cost512 *= 0.95;
        if (gather || cost512 < best_cost) {
            best_cost = cost512;
            best = TileChoice{4, 512};
        }
    }
    // Gathered rows, K >= 2048: CTA pairs of 256 x 512 tiles side by side
    // along N, each CTA issuing its share of its rows' gather4s and
    // multicasting them to the CTAs in the same place of the other pairs --
    // four pairs for N >= 2048, two for N >= 1024 (16384 of 65536 rows,
    // K = 4096, N = 4096: four pairs 0.391 ms, two 0.431, clusters of eight
    // single CTAs 0.469, one pair 0.564; N = 1024: two pairs 0.113 ms,
    // clusters of four single CTAs 0.136).  With shorter K the single
    // accumulator's drain weighs more: clusters of eight single CTAs
    // (N >= 2048; N = 4096, K = 1024: 0.145 against 0.158 ms for two pairs)
    // or of four.
    if (gather && N >= 2048 && K >= 2048)
        best = TileChoice{9, 512};
    else if (gather && N >= 1024 && K >= 2048)
        best = TileChoice{7, 512};
    else if (gather && N >= 2048)
        best = TileChoice{6, 256};
    else if (gather && N >= 1024)
        best = TileChoice{5, 256};
    return best;
}

int skinny_rows(int64_t M) { return M <= 16 ? 16 : (M <= 32 ? 32 : 64); }

// Problems the skinny kernel can run: M <= 64, K > 0, plain, scattered or
// accumulating (gathered rows and seeded accumulators: tile kernel only).
bool skinny_eligible(int64_t M, int64_t K, bool gather, bool seeded)
{
    return !gather && !seeded && M <= 64 && K > 0;
}

// Few rows of A, bf16 / f16 B: whether the skinny kernel beats the tile
// kernel.  The skinny kernel spreads every tile's K over the SMs, which pays
// when the tile kernel has few tiles to give them and a long K to walk in
// each (K large against N); with more than 16 rows and a short K its
// epilogue and split reductions cost more than the tile kernel's idle MMA
// rows.  Measured (CUDA-graph replay, operands cold in HBM, microseconds
// skinny / tile): M = 16: 28672 x 4096 42.0 / 45.1, 4096^2 14.1 / 16.6,
// 1024^2 8.9 / 6.8; M = 32: 28672 x 4096 46.0 / 45.9, 4096 x 8192
// 23.6 / 29.3, 4096^2 23.0 / 16.6, 16384 x 2048 25.4 / 16.8; M = 64:
// 4096^2 19.4 / 16.7, 4096 x 14336 30.5 / 48.3, 2048 x 16384 23.7 / 54.4,
// 1024 x 8192 20.0 / 29.1; 48 rows 2048 x 8192 20.4 / 29.1.  After the
// skinny epilogue's straight-line loads and stores (same method): M = 32:
// 4096^2 14.0 / 16.8, 28672 x 4096 44.1 / 45.7, 16384 x 2048 20.4 / 17.2,
// 4096 x 8192 19.5 / 35.5; M = 64: 4096^2 22.6 / 16.9, 28672 x 4096
// 53.8 / 46.7, 1024 x 8192 21.0 / 34.6; 48 x 8192^2 36.3 / 31.3; M = 16:
// 1024^2 7.7 / 6.8.  After the skinny epilogue's register spills at MP = 64
// were removed: M = 64: 4096^2 14.9 / 16.9, 2048^2 10.1 / 10.4, 28672 x 4096
// 47.1 / 47.5, 8192 x 4096 19.7 / 17.8, 14336 x 4096 29.4 / 26.7; 40 x 4096^2
// 14.7 / 16.8; 48 x 8192^2 31.2 / 31.5; 33 x 28672 x 4096 44.9 / 45.8.
bool skinny_wins(int64_t M, int64_t N, int64_t K)
{
    const bool big = N * K > (int64_t(1) << 21);  // (N, K < 2^31: no overflow)
    if (M <= 16)
        return big;
    return K >= 2 * N || (big && K >= N);
}

// The skinny kernel's plan for m <= 64 rows (stream-K over the SMs).
void set_skinny_plan(gemm_plan &p, int64_t m, int64_t N, int64_t K, int sm_count, bool w4)
{
    // few rows: swap A and B so B streams through the MMA's M side
    const int mp = skinny_rows(m);
    const int64_t tiles = ceil_div(N, 128);
    const int64_t nkb = ceil_div(K, w4 ? tcg::skinny_w4_kstage() : tcg::skinny_kstage());
    const int64_t W = tiles * nkb;
    // at least TCG_SKINNY_MIN_KB K blocks per CTA, so small problems are
    // not cut into many parts whose reduction costs more than it saves
    const int64_t want = ceil_div(W, TCG_SKINNY_MIN_KB);
    const int64_t G = want < sm_count ? want : sm_count;
    p.kernel = 2;
    p.bm = mp;
    p.bn = 128;
    p.stages = w4 ? tcg::skinny_w4_stages(mp) : tcg::skinny_stages(mp);
    p.tiles = tiles;
    p.splits = tcg::skinny_max_parts(tcg::skinny_sk_tiles(tiles, G, w4), nkb, G);
    p.grid = static_cast<int32_t>(G);
}

// Problems with at most this many multiply-adds run on the warp-level kernel.
constexpr int64_t kTinyWork = int64_t(1) << 20;

// The tile kernel's form for plan.kernel 1 (single CTAs, 128 x bn tiles),
// 3 (CTA pairs, 256 x 256), 4 (CTA pairs, 256 x 512: two MMA halves),
// 5 / 6 (single CTAs, 128 x bn tiles, in clusters of 4 / 8 along N sharing A)
// and 7 / 8 (two CTA pairs, 256 x 512 / 256 x 256 tiles, sharing A).
struct TileForm {
    bool pair;
    int mma_bn;
    int nsub;
    int mc;       // CTAs (pairs) sharing one A box by multicast
    int cluster;  // CTAs per cluster
    int tile_m;
    int tile_n;
};

TileForm tile_form(const gemm_plan &p)
{
    if (p.kernel == 3)
        return TileForm{true, 256, 1, 1, 2, 256, 256};
    if (p.kernel == 4)
        return TileForm{true, 256, 2, 1, 2, 256, 512};
    if (p.kernel == 5)
        return TileForm{false, p.bn, 1, 4, 4, 128, p.bn};
    if (p.kernel == 6)
        return TileForm{false, p.bn, 1, 8, 8, 128, p.bn};
    if (p.kernel == 7)
        return TileForm{true, 256, 2, 2, 4, 256, 512};
    if (p.kernel == 8)
        return TileForm{true, 256, 1, 2, 4, 256, 256};
    if (p.kernel == 9)
        return TileForm{true, 256, 2, 4, 8, 256, 512};
    return TileForm{false, p.bn, 1, 1, 1, 128, p.bn};
}

// Units the persistent loop walks: CTA tiles, or for A multicast the groups of
// mc neighbouring tiles of a block row that one cluster computes together.
int64_t loop_tiles(const TileForm &f, int64_t M, int64_t N)
{
    const int64_t n_units = f.mc > 1 ? ceil_div(ceil_div(N, f.tile_n), f.mc) : ceil_div(N, f.tile_n);
    return ceil_div(M, f.tile_m) * n_units;
}

// Fill the tile-kernel fields of a plan for `kernel` (1, 3, 4 or 5) and tile width bn.
void set_tile_plan(gemm_plan &p, int kernel, int bn, int64_t M, int64_t N, int sm_count)
{
    p.kernel = kernel;
    p.bn = bn;
    p.splits = 1;
    const TileForm f = tile_form(p);
    p.bm = f.tile_m;
    p.stages = tcg::tile_stages(f.mma_bn, f.pair, f.nsub, f.mc);
    p.tiles = ceil_div(M, f.tile_m) * ceil_div(N, f.tile_n);
    const int64_t units = loop_tiles(f, M, N);
    const int64_t sets = sm_count / f.cluster;
    const int64_t used = units < sets ? units : sets;
    p.grid = static_cast<int32_t>(f.cluster * used);
}

// The warp-level kernel: 16 x 8 blocks, four per CTA.
void set_tiny_plan(gemm_plan &p, int64_t M, int64_t N)
{
    p.kernel = 10;
    p.bm = 16;
    p.bn = 8;
    p.stages = 0;
    p.tiles = ceil_div(M, 16) * ceil_div(N, 8);
    p.splits = 1;
    p.grid = static_cast<int32_t>(ceil_div(p.tiles, tcg::tiny_warps_per_cta()));
}

gemm_plan make_plan(int64_t M, int64_t N, int64_t K, bool gather, bool c_used, int sm_count,
                    bool scatter, bool seeded, bool w4)
{
    gemm_plan p;
    std::memset(&p, 0, sizeof(p));
    if (M == 0 || N == 0)
        return p;
    // (sizes are at most 2^31 each: bound the factors before multiplying)
    if (!(w4 && K > 0) && M <= kTinyWork && N <= kTinyWork && M * N <= kTinyWork &&
        M * N * (K > 0 ? K : 1) <= kTinyWork) {
        set_tiny_plan(p, M, N);
        return p;
    }
    // (FP4 weights with 64 < M <= 128 run as two launches of the 64-row skinny
    // kernel; the plan describes one of them; FP4 weights with M <= 64 always
    // take the skinny kernel, which converts them on the fly)
    const int64_t m_skinny = (w4 && K > 0 && M <= 128 && M > 64) ? 64 : M;
    if (skinny_eligible(m_skinny, K, gather, seeded) && (w4 || skinny_wins(M, N, K))) {
        set_skinny_plan(p, m_skinny, N, K, sm_count, w4);
        return p;
    }
    const TileChoice c = choose_tile(M, N, K, gather, c_used, scatter, sm_count);
    set_tile_plan(p, c.kernel, c.bn, M, N, sm_count);
    return p;
}

gemm_plan noalloc_plan(int64_t M, int64_t N, int64_t K, bool c_used, int sm_count)
{
    gemm_plan p;
    std::memset(&p, 0, sizeof(p));
    if (!skinny_eligible(M, K, false, false))
        return p;  // M > 64 or K == 0: not this entry point's
    p = make_plan(M, N, K, false, c_used, sm_count);
    if (p.kernel == 0 || p.kernel == 10)
        return p;  // empty, or the warp-level kernel (which needs no scratch)
    set_skinny_plan(p, M, N, K, sm_count, false);
    return p;
}

CUtensorMapDataType ab_type(bool bf16)
{
    return bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}

void fill_common(GemmArgs &a, const Problem &p, const DeviceInfo *dev)
{
    const bool c_used = p.C != nullptr && p.beta != 0.0f;
    a.M = static_cast<int32_t>(p.M);
    a.N = static_cast<int32_t>(p.N);
    a.K = static_cast<int32_t>(p.K);
    a.alpha = p.alpha;
    a.beta = p.beta;
    a.has_c = c_used ? 1 : 0;
    a.out_kind = p.out;
    a.ab_bf16 = p.bf16 ? 1 : 0;
    a.C = p.C;
    a.ldc = p.ldc;
    a.D = p.D;
    a.ldd = p.ldd;
    a.extra_tx = g_inject.load() == 1 ? 16u : 0u;
    a.status = dev->status;
    a.timeout_ns = g_timeout_ns.load();
}

// Buffers of the FP4 paths, one per (device, stream, use), grown
// geometrically: kBufWeights holds the bf16 copy of the weights for M > 64,
// kBufScales a copy of the scales with a 16-byte row pitch for the TMA loads
// of the M <= 64 path when the caller's pitch or base is not 16-byte aligned
// (kBufScalesA / kBufScalesB: the same for gemm_e2m1's two operands).
struct DequantBuffer {
    int device = -1;
    cudaStream_t stream = nullptr;
    int use = 0;
    void *ptr = nullptr;
    size_t bytes = 0;
};
std::mutex g_dq_mu;
std::vector<DequantBuffer> g_dq;

gemm_status get_dequant_buffer(int device, cudaStream_t stream, int use, size_t bytes,
                               void **out)
{
    std::lock_guard<std::mutex> lock(g_dq_mu);
    DequantBuffer *b = nullptr;
    for (DequantBuffer &x : g_dq)
        if (x.device == device && x.stream == stream && x.use == use)
            b = &x;
    if (!b) {
        g_dq.push_back(DequantBuffer{});
        b = &g_dq.back();
        b->device = device;
        b->stream = stream;
        b->use = use;
    }
    if (b->bytes < bytes) {
        if (b->ptr) {
            if (cudaStreamSynchronize(stream) != cudaSuccess)  // earlier calls may still read it
                return GEMM_ERR_CUDA;
            cudaFree(b->ptr);
            b->ptr = nullptr;
        }
        const size_t nb = bytes > 2 * b->bytes ? bytes : 2 * b->bytes;
        b->bytes = 0;
        if (cudaMalloc(&b->ptr, nb) != cudaSuccess)
            return GEMM_ERR_CUDA;
        b->bytes = nb;
    }
    *out = b->ptr;
    return GEMM_OK;
}

gemm_status run_skinny(const Problem &p, const gemm_plan &plan, const DeviceInfo *dev)
{
    const int mp = plan.bm;
    GemmMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    if (!encode_2d(&maps.a, ab_type(p.bf16), p.A, p.K, p.M, p.lda * 2, 64,
                   static_cast<uint32_t>(mp), CU_TENSOR_MAP_SWIZZLE_128B))
        return GEMM_ERR_CUDA;
    if (p.w4) {
        // codes: 32-byte boxes (64 elements) of 128 rows; scales: the block's
        // two rows of 128 columns (rows 16-byte aligned for TMA: copy them if
        // the caller's are not)
        const void *scales = p.bscale;
        int64_t lds = p.ldbs;
        if (!aligned16(scales) || lds % 16) {
            const int64_t pitch = (p.N + 15) / 16 * 16;
            void *buf = nullptr;
            gemm_status st = get_dequant_buffer(dev->index, p.stream, kBufScales,
                                                static_cast<size_t>(pitch) * (p.K / 32), &buf);
            if (st != GEMM_OK)
                return st;
            if (cudaMemcpy2DAsync(buf, pitch, p.bscale, p.ldbs, p.N, p.K / 32,
                                  cudaMemcpyDeviceToDevice, p.stream) != cudaSuccess)
                return GEMM_ERR_CUDA;
            scales = buf;
            lds = pitch;
        }
        if (!encode_2d(&maps.b, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.B, p.K / 2, p.N, p.ldb, 128, 128,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_2d(&maps.c, CU_TENSOR_MAP_DATA_TYPE_UINT8, scales, p.N, p.K / 32, lds, 128, 8,
                       CU_TENSOR_MAP_SWIZZLE_NONE))
            return GEMM_ERR_CUDA;
    } else if (!encode_2d(&maps.b, ab_type(p.bf16), p.B, p.K, p.N, p.ldb * 2, 64, 128,
                          CU_TENSOR_MAP_SWIZZLE_128B)) {
        return GEMM_ERR_CUDA;
    }
    GemmArgs a;
    std::memset(&a, 0, sizeof(a));
    fill_common(a, p, dev);
    a.num_m_blocks = 1;
    a.num_n_blocks = static_cast<int32_t>(plan.tiles);
    a.num_k_blocks =
        static_cast<int32_t>(ceil_div(p.K, p.w4 ? tcg::skinny_w4_kstage() : tcg::skinny_kstage()));
    a.num_tiles = static_cast<int32_t>(plan.tiles);
    a.sk_tiles = static_cast<int32_t>(tcg::skinny_sk_tiles(plan.tiles, plan.grid, p.w4));
    a.group_m = 1;
    a.splits = plan.splits;
    a.scatter = p.scatter ? 1 : 0;
    a.idx = p.idx;
    a.d_rows = static_cast<int32_t>(p.d_rows);
    a.reduce = p.reduce ? 1 : 0;
    if (plan.splits > 1 && !p.reduce) {  // (the accumulating form adds every part into D)
        Workspace w;
        const size_t bytes = static_cast<size_t>(plan.tiles) * plan.splits * 128 * mp * sizeof(float);
        gemm_status st = get_workspace(dev->index, p.stream, bytes, static_cast<size_t>(plan.tiles), &w);
        if (st != GEMM_OK)
            return st;
        a.workspace = w.partials;
        a.counters = w.counters;
    }
    const cudaError_t e = p.w4 ? tcg::launch_skinny_w4(mp, maps, a, plan.grid, p.stream)
                               : tcg::launch_skinny(mp, maps, a, plan.grid, p.stream);
    return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

gemm_status run_tiny(const Problem &p, const gemm_plan &plan, const DeviceInfo *dev)
{
    GemmArgs a;
    std::memset(&a, 0, sizeof(a));
    fill_common(a, p, dev);
    a.num_tiles = static_cast<int32_t>(plan.tiles);
    a.gather = p.gather ? 1 : 0;
    a.scatter = p.scatter ? 1 : 0;
    a.reduce = p.reduce ? 1 : 0;
    a.idx = p.idx;
    a.table_rows = static_cast<int32_t>(p.a_rows);
    a.d_rows = static_cast<int32_t>(p.d_rows);
    if (p.seed) {
        a.seed = 1;
        a.has_c = 0;
    }
    const cudaError_t e = tcg::launch_tiny(p.A, p.lda, p.B, p.ldb, a, plan.grid, p.stream);
    return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

void forced_tile(int *kernel, int *bn)
{
    *kernel = g_force_kernel.load();
    *bn = g_force_bn.load();
}

// Test hook: replace the automatic tile form by a forced one where it can run.
gemm_plan apply_forced_tile(gemm_plan plan, const Problem &p, int sm_count)
{
    const int fk = g_force_kernel.load(), fbn = g_force_bn.load();
    if (fk == 0 || (fk >= 11 && fk <= 15) || plan.kernel == 0 || p.w4)
        return plan;  // (FP4 weights run only on their own paths; 11-15 are FP4 x FP4 forms)
    if (fk == 10) {
        set_tiny_plan(plan, p.M, p.N);  // the warp-level kernel runs every problem
        return plan;
    }
    if (fk == 2) {
        if (skinny_eligible(p.M, p.K, p.gather, p.seed))
            set_skinny_plan(plan, p.M, p.N, p.K, sm_count, false);
        return plan;
    }
    if (fk != 1 && p.K == 0)
        return plan;  // cluster forms need K > 0
    set_tile_plan(plan, fk, fbn, p.M, p.N, sm_count);
    return plan;
}

// The tile kernel in the form of `plan` over all of p (maps, arguments,
// launch).  grid_cap > 0 bounds the persistent grid; co_tail marks a launch
// that runs beside the previous kernel on the SMs it leaves idle.
gemm_status launch_tile_problem(const Problem &p, const gemm_plan &plan, const DeviceInfo *dev,
                                int grid_cap, bool co_tail)
{
    GemmMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    const TileForm form = tile_form(plan);
    const bool c_used = p.C != nullptr && p.beta != 0.0f;
    const bool pair = form.pair;
    const int bn = form.mma_bn;
    const int bn_local = pair ? bn / 2 : bn;  // rows of B per MMA half each CTA loads
    const int64_t units = loop_tiles(form, p.M, p.N);
    int grid = plan.grid;
    if (grid_cap > 0 && grid > grid_cap)
        grid = grid_cap;
    if (form.cluster > 1) {
        // never more clusters than can be resident together (SMs left over
        // within a GPC stay idle)
        const int resident = tcg::tile_max_clusters(bn, pair, form.nsub, form.mc);
        if (resident <= 0)
            return GEMM_ERR_CUDA;
        grid = static_cast<int>(form.cluster * (units < resident ? units : resident));
    }
    if (p.K > 0) {
        // dense A: each CTA loads its rows (A multicast: its 128 / mc rows for the cluster)
        const uint32_t a_box_rows = static_cast<uint32_t>(128 / form.mc);
        const bool ok_a =
            p.gather ? encode_2d(&maps.a, ab_type(p.bf16), p.A, p.K, p.a_rows, p.lda * 2, 64, 1,
                                 CU_TENSOR_MAP_SWIZZLE_128B)
                     : encode_2d(&maps.a, ab_type(p.bf16), p.A, p.K, p.M, p.lda * 2, 64,
                                 a_box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
        const bool ok_b = encode_2d(&maps.b, ab_type(p.bf16), p.B, p.K, p.N, p.ldb * 2, 64,
                                    static_cast<uint32_t>(bn_local), CU_TENSOR_MAP_SWIZZLE_128B);
        if (!ok_a || !ok_b)
            return GEMM_ERR_CUDA;
    }
    // C and D boxes: 32 x 32, or for scattered rows boxes one row high that
    // tile::gather4 / tile::scatter4 move four rows at a time (D by TMA only
    // for float32 output, whose 32-column rows fill the 128-byte swizzle span)
    const int64_t out_rows = p.scatter ? p.d_rows : p.M;
    const uint32_t box_rows = p.scatter ? 1u : 32u;
    // (seeded accumulators read C with plain loads, once, into tensor memory)
    const bool c_tma = c_used && !p.seed && aligned16(p.C) && (p.ldc * 4) % 16 == 0;
    const bool d_tma = aligned16(p.D) && (p.ldd * out_size(p.out)) % 16 == 0 &&
                       (!p.scatter || p.out == GEMM_OUT_F32);
    if (c_tma && !encode_2d(&maps.c, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p.C, p.N, out_rows,
                            p.ldc * 4, 32, box_rows, CU_TENSOR_MAP_SWIZZLE_128B))
        return GEMM_ERR_CUDA;
    if (d_tma) {
        const CUtensorMapDataType dt = p.out == GEMM_OUT_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                       : p.out == GEMM_OUT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                                : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
        const CUtensorMapSwizzle sw =
            p.out == GEMM_OUT_F32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
        if (!encode_2d(&maps.d, dt, p.D, p.N, out_rows, p.ldd * out_size(p.out), 32, box_rows,
                       sw))
            return GEMM_ERR_CUDA;
    }

    GemmArgs a;
    std::memset(&a, 0, sizeof(a));
    fill_common(a, p, dev);
    a.num_m_blocks = static_cast<int32_t>(ceil_div(p.M, form.tile_m));
    a.num_n_blocks = static_cast<int32_t>(units / a.num_m_blocks);  // (clusters: groups of mc)
    a.num_k_blocks = static_cast<int32_t>(ceil_div(p.K, 64));
    a.num_tiles = static_cast<int32_t>(units);
    a.group_m = a.num_m_blocks < TCG_GROUP_M ? a.num_m_blocks : TCG_GROUP_M;
    a.splits = 1;
    a.gather = p.gather ? 1 : 0;
    a.c_tma = c_tma ? 1 : 0;
    a.d_tma = d_tma ? 1 : 0;
    a.d_tail_direct = (p.N * out_size(p.out)) % 16 != 0 ? 1 : 0;
    a.idx = p.idx;
    a.table_rows = static_cast<int32_t>(p.a_rows);
    a.scatter = p.scatter ? 1 : 0;
    a.d_rows = static_cast<int32_t>(p.d_rows);
    a.reduce = p.reduce ? 1 : 0;
    a.co_tail = co_tail ? 1 : 0;
    if (p.seed) {
        a.seed = 1;
        a.has_c = 0;  // C went into the accumulator; the epilogue writes D = acc
    }

    const int mode = p.scatter ? 1 : (p.reduce ? 2 : (p.seed ? 3 : 0));  // epilogue mode
    const cudaError_t e =
        tcg::launch_tile(mode, bn, pair, form.nsub, form.mc, maps, a, grid, p.stream);
    return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

// A clustered form places whole clusters only (within a GPC), so some SMs stay
// idle, and its last wave of clusters may run part-full.  For gathered rows
// the first rows then run as whole waves of the clustered form, and the
// remaining 256-row stripes on single CTAs (128 x 256 tiles, no cluster) on
// the idle SMs at the same time: the tail is launched right behind the
// clustered kernel (programmatic dependent launch), so its CTAs land on the
// SMs left free.  The stripes are chosen so the tail, at kTailRate of the
// clustered form's rate per SM, ends within the clustered kernel's time.
// Returns the rows for the clustered kernel, or 0 for no split.
// (kTailRate: 16384 of 65536 rows, N = K = 4096: single 128 x 256 CTAs
// 1.032 ms on 152 SMs, four CTA pairs sharing rows 0.397 ms on 120 SMs.)
constexpr double kTailRate = 0.30;

int64_t tail_split_rows(const Problem &p, const gemm_plan &plan, const DeviceInfo *dev)
{
    if (!p.gather || p.scatter || p.reduce || p.seed || p.K == 0 || g_force_kernel.load() != 0)
        return 0;
    const TileForm f = tile_form(plan);
    if (f.cluster <= 2)
        return 0;
    const int resident = tcg::tile_max_clusters(f.mma_bn, f.pair, f.nsub, f.mc);
    const int idle = dev->sm_count - resident * f.cluster;
    if (resident <= 0 || idle < 8)
        return 0;
    const int64_t m_blocks = ceil_div(p.M, f.tile_m);
    const int64_t per_stripe = loop_tiles(f, f.tile_m, p.N);  // units in one stripe of rows
    const int64_t waves_now = ceil_div(m_blocks * per_stripe, resident);
    // what one wave of the clustered kernel covers, in (row x column) cells,
    // and what the idle SMs cover in the same time
    const double wave_cells = static_cast<double>(resident) * f.tile_m * f.mc * f.tile_n;
    const double tail_cells_per_wave =
        wave_cells / (resident * f.cluster) * idle * kTailRate;
    for (int64_t m = m_blocks - 1; m > 0; --m) {
        if ((m * per_stripe) % resident != 0)
            continue;
        const int64_t waves = m * per_stripe / resident;
        if (waves >= waves_now)
            continue;
        const double tail_rows = static_cast<double>(p.M - m * f.tile_m);
        if (tail_rows * static_cast<double>(p.N) <= tail_cells_per_wave * waves)
            return m * f.tile_m;
        return 0;  // fewer stripes only lengthen the tail
    }
    return 0;
}

gemm_status run(const Problem &p)
{
    bool empty = false;
    gemm_status st = validate(p, &empty);
    if (st != GEMM_OK || empty)
        return st;
    if (p.reduce && p.K == 0)
        return GEMM_OK;  // adding zero
    DeviceInfo *dev = nullptr;
    if ((st = device_info(&dev)) != GEMM_OK)
        return st;
    if (p.w4 && p.K > 0 && p.M > 64 && p.M <= 128) {
        // up to 128 rows: two launches of the FP4 skinny kernel, rows 0-63 and
        // the rest (each decodes the weights again, which still costs less than
        // converting them to bf16 in memory: 64 + 64 rows, N = 28672, K = 4096:
        // 99 against 120 us)
        Problem h = p;
        h.M = 64;
        h.a_rows = 64;
        if ((st = run(h)) != GEMM_OK)
            return st;
        Problem t = p;
        t.M = p.M - 64;
        t.a_rows = t.M;
        t.A = static_cast<const char *>(p.A) + 64 * p.lda * 2;
        if (t.C != nullptr)
            t.C = p.C + 64 * p.ldc;
        t.D = static_cast<char *>(p.D) + 64 * p.ldd * out_size(p.out);
        return run(t);
    }
    if (p.w4 && p.K > 0 && p.M > 64) {
        // many rows: turn the weights into bf16 once (exact: every code times a
        // power of two fits bf16 unless it leaves its range) and run the bf16 GEMM
        void *wb = nullptr;
        if ((st = get_dequant_buffer(dev->index, p.stream, kBufWeights,
                                     static_cast<size_t>(p.N) * p.K * 2, &wb)) != GEMM_OK)
            return st;
        if (tcg::launch_dequant_fp4(static_cast<const uint8_t *>(p.B), p.ldb, p.bscale, p.ldbs,
                                    static_cast<int32_t>(p.N), static_cast<int32_t>(p.K),
                                    static_cast<uint16_t *>(wb), p.K, p.stream) != cudaSuccess)
            return GEMM_ERR_CUDA;
        Problem q = p;
        q.w4 = false;
        q.B = wb;
        q.ldb = p.K;
        q.bscale = nullptr;
        return run(q);
    }
    const bool c_used = p.C != nullptr && p.beta != 0.0f;
    const gemm_plan plan = apply_forced_tile(
        make_plan(p.M, p.N, p.K, p.gather, c_used, dev->sm_count, p.scatter, p.seed,
                  p.w4 && p.K > 0),
        p, dev->sm_count);

    if (plan.kernel == 2)
        return run_skinny(p, plan, dev);
    if (plan.kernel == 10)
        return run_tiny(p, plan, dev);
    const int64_t head = tail_split_rows(p, plan, dev);
    if (head <= 0)
        return launch_tile_problem(p, plan, dev, 0, false);
    Problem h = p;
    h.M = head;
    Problem t = p;
    t.M = p.M - head;
    t.idx = p.idx + head;
    if (t.C != nullptr)
        t.C = p.C + head * p.ldc;
    t.D = static_cast<char *>(p.D) + head * p.ldd * out_size(p.out);
    gemm_plan tp;
    std::memset(&tp, 0, sizeof(tp));
    set_tile_plan(tp, 1, 256, t.M, t.N, dev->sm_count);
    const TileForm f = tile_form(plan);
    const int idle = dev->sm_count -
                     tcg::tile_max_clusters(f.mma_bn, f.pair, f.nsub, f.mc) * f.cluster;
    if ((st = launch_tile_problem(h, plan, dev, 0, false)) != GEMM_OK)
        return st;
    return launch_tile_problem(t, tp, dev, idle, true);
}

}  // namespace host
}  // namespace tcg

using namespace tcg::host;

// ------------------------------------------------------------- exported ABI

extern "C" {

gemm_status gemm_f16(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B,
                     int64_t ldb, const float *C, int64_t ldc, void *D, int64_t ldd, int out,
                     float alpha, float beta, void *stream)
{
    Problem p{M, N, K, false, A, M, lda, nullptr, B, ldb, C, ldc, D, ldd, out, alpha, beta,
              false, static_cast<cudaStream_t>(stream)};
    return run(p);
}

gemm_status gemm_bf16(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B,
                      int64_t ldb, const float *C, int64_t ldc, void *D, int64_t ldd, int out,
                      float alpha, float beta, void *stream)
{
    Problem p{M, N, K, true, A, M, lda, nullptr, B, ldb, C, ldc, D, ldd, out, alpha, beta,
              false, static_cast<cudaStream_t>(stream)};
    return run(p);
}

gemm_status gemm_gather_rows(int64_t M, int64_t N, int64_t K, int dtype_is_bf16,
                             const void *table, int64_t table_rows, int64_t lda,
                             const int32_t *idx, const void *B, int64_t ldb, const float *C,
                             int64_t ldc, void *D, int64_t ldd, int out, float alpha, float beta,
                             void *stream)
{
    if (dtype_is_bf16 != 0 && dtype_is_bf16 != 1)
        return GEMM_ERR_INVALID_ARG;
    Problem p{M, N, K, dtype_is_bf16 == 1, table, table_rows, lda, idx, B, ldb, C, ldc, D, ldd,
              out, alpha, beta, true, static_cast<cudaStream_t>(stream)};
    return run(p);
}

gemm_status gemm_scatter_rows(int64_t M, int64_t N, int64_t K, int dtype_is_bf16, const void *A,
                              int64_t lda, const void *B, int64_t ldb, const int32_t *idx,
                              int64_t d_rows, const float *C, int64_t ldc, void *D, int64_t ldd,
                              int out, float alpha, float beta, void *stream)
{
    if (dtype_is_bf16 != 0 && dtype_is_bf16 != 1)
        return GEMM_ERR_INVALID_ARG;
    Problem p{M, N, K, dtype_is_bf16 == 1, A, M, lda, idx, B, ldb, C, ldc, D, ldd,
              out, alpha, beta, false, static_cast<cudaStream_t>(stream)};
    p.scatter = true;
    p.d_rows = d_rows;
    return run(p);
}

gemm_status gemm_accumulate(int64_t M, int64_t N, int64_t K, int dtype_is_bf16, const void *A,
                            int64_t lda, const void *B, int64_t ldb, float *D, int64_t ldd,
                            float alpha, void *stream)
{
    if (dtype_is_bf16 != 0 && dtype_is_bf16 != 1)
        return GEMM_ERR_INVALID_ARG;
    Problem p{M, N, K, dtype_is_bf16 == 1, A, M, lda, nullptr, B, ldb, nullptr, 0, D, ldd,
              GEMM_OUT_F32, alpha, 0.0f, false, static_cast<cudaStream_t>(stream)};
    p.reduce = true;
    return run(p);
}

gemm_status gemm_seeded(int64_t M, int64_t N, int64_t K, int dtype_is_bf16, const void *A,
                        int64_t lda, const void *B, int64_t ldb, const float *C, int64_t ldc,
                        void *D, int64_t ldd, int out, void *stream)
{
    if (dtype_is_bf16 != 0 && dtype_is_bf16 != 1)
        return GEMM_ERR_INVALID_ARG;
    Problem p{M, N, K, dtype_is_bf16 == 1, A, M, lda, nullptr, B, ldb, C, ldc, D, ldd,
              out, 1.0f, 1.0f, false, static_cast<cudaStream_t>(stream)};
    p.seed = true;
    if (M > 0 && N > 0 && !C)
        return GEMM_ERR_INVALID_ARG;
    return run(p);
}

gemm_status gemm_bf16_e2m1(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda,
                           const uint8_t *Bq, int64_t ldbq, const uint8_t *Bs, int64_t ldbs,
                           const float *C, int64_t ldc, void *D, int64_t ldd, int out,
                           float alpha, float beta, void *stream)
{
    Problem p{M, N, K, true, A, M, lda, nullptr, Bq, ldbq, C, ldc, D, ldd,
              out, alpha, beta, false, static_cast<cudaStream_t>(stream)};
    p.w4 = true;
    p.bscale = Bs;
    p.ldbs = ldbs;
    return run(p);
}

gemm_status gemm_check_device_status(void *stream)
{
    DeviceInfo *dev = nullptr;
    gemm_status st = device_info(&dev);
    if (st != GEMM_OK)
        return st;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return GEMM_ERR_CUDA;
    uint32_t h[2] = {0, 0};
    if (cudaMemcpy(h, dev->status, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (h[0] != 0) {
        if (cudaMemset(dev->status, 0, sizeof(h)) != cudaSuccess)
            return GEMM_ERR_CUDA;
        if ((st = reset_workspaces(dev->index)) != GEMM_OK)
            return st;
        if ((st = reset_static_scratch(dev->index)) != GEMM_OK)
            return st;
    }
    return static_cast<gemm_status>(h[0]);
}

const char *gemm_status_string(int status)
{
    switch (status) {
    case GEMM_OK: return "GEMM_OK";
    case GEMM_ERR_INVALID_ARG: return "GEMM_ERR_INVALID_ARG";
    case GEMM_ERR_ALIGNMENT: return "GEMM_ERR_ALIGNMENT";
    case GEMM_ERR_UNSUPPORTED: return "GEMM_ERR_UNSUPPORTED";
    case GEMM_ERR_ALIAS: return "GEMM_ERR_ALIAS";
    case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA";
    case GEMM_ERR_TIMEOUT: return "GEMM_ERR_TIMEOUT";
    case GEMM_ERR_INDEX: return "GEMM_ERR_INDEX";
    default: return "GEMM_ERR_UNKNOWN";
    }
}

gemm_status gemm_query_plan(int64_t M, int64_t N, int64_t K, int form, int has_c,
                            int sm_count, gemm_plan *plan)
{
    if (!plan || sm_count < 1 || M < 0 || N < 0 || K < 0)
        return GEMM_ERR_INVALID_ARG;
    if (form < 0 || form > 7)
        return GEMM_ERR_INVALID_ARG;
    if (form == 5) {
        *plan = noalloc_plan(M, N, K, has_c != 0, sm_count);
        return GEMM_OK;
    }
    if (form == 6 || form == 7) {
        *plan = e2m1_plan(M, N, K, form - 6, sm_count);
        return GEMM_OK;
    }
    Problem q{};
    q.M = M;
    q.N = N;
    q.K = K;
    q.gather = form == 1;
    q.scatter = form == 2;
    q.seed = form == 3;
    q.w4 = form == 4 && K > 0;
    *plan = apply_forced_tile(make_plan(M, N, K, q.gather, has_c != 0 || q.seed, sm_count,
                                        q.scatter, q.seed, q.w4),
                              q, sm_count);
    return GEMM_OK;
}

gemm_status gemm_set_wait_timeout(uint64_t ns)
{
    g_timeout_ns.store(ns == 0 ? kDefaultTimeoutNs : ns);
    return GEMM_OK;
}

gemm_status gemm_debug_force_tile(int kernel, int bn)
{
    const bool ok = (kernel == 0) || (kernel == 2 && (bn == 0 || bn == 128)) ||
                    (kernel == 1 && (bn == 64 || bn == 128 || bn == 256)) ||
                    (kernel == 3 && bn == 256) || (kernel == 4 && bn == 512) ||
                    (kernel == 5 && (bn == 64 || bn == 256)) || (kernel == 6 && bn == 256) ||
                    (kernel == 7 && bn == 512) || (kernel == 8 && bn == 256) ||
                    (kernel == 9 && bn == 512) || (kernel == 10 && bn == 8) ||
                    ((kernel == 11 || kernel == 12) && (bn == 128 || bn == 256)) ||
                    ((kernel == 13 || kernel == 14) && bn == 256) || (kernel == 15 && bn == 128);
    if (!ok)
        return GEMM_ERR_INVALID_ARG;
    g_force_kernel.store(kernel);
    g_force_bn.store(bn);
    return GEMM_OK;
}

gemm_status gemm_debug_inject(int mode)
{
    if (mode != 0 && mode != 1)
        return GEMM_ERR_INVALID_ARG;
    g_inject.store(mode);
    return GEMM_OK;
}

}  // extern "C"
