// noalloc.cu -- gemm_skinny_noalloc: the skinny (M <= 64) kernel with its
// scratch memory in a fixed device array that the library owns, so the call
// itself never allocates device memory.
//
// Who needs it: callers that cannot call cudaMalloc at the point where they
// run the GEMM -- for example code whose device memory is owned entirely by
// another allocator (a framework's caching allocator, or a serving engine
// that reserves the whole GPU up front, so a library cudaMalloc would fail or
// fragment memory it does not own), and latency-critical sections where the
// implicit device-wide synchronisation of cudaMalloc/cudaFree is not allowed.
// The regular gemm_f16 / gemm_bf16 entry points allocate their skinny-path
// scratch lazily on first use per stream; this one never does.
//
// The scratch is one file-scope device array of kStaticScratchBytes bytes
// (partial tiles, then per-tile arrival counters).  Every GPU that loads this
// module keeps it until the process exits.  Host code only ever passes the
// address that cudaGetSymbolAddress returns for the current device: the
// array's name in host code is a host-side stand-in, not a device address.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "host_internal.h"

namespace {

// 16 MiB of per-split partial tiles: enough for the 16 x 28672 x 4096 decode
// shape (3.7 MB) and, e.g., M <= 64 up to N = 28672 at two parts per tile.
constexpr size_t kStaticPartialBytes = size_t(16) << 20;
// One arrival counter per 128-row tile of B: N up to 16384 * 128 = 2,097,152.
constexpr size_t kStaticCounters = 16384;
constexpr size_t kStaticScratchBytes = kStaticPartialBytes + kStaticCounters * sizeof(uint32_t);

}  // namespace

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
unsigned char *g_static_ptr[kMaxDevices] = {};

// Device address of the scratch array on `device` (which must be current).
// Looked up once per device and remembered.
gemm_status static_scratch(int device, unsigned char **out)
{
    if (device < 0 || device >= kMaxDevices)
        return GEMM_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!g_static_ptr[device]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p)
            return GEMM_ERR_CUDA;
        g_static_ptr[device] = static_cast<unsigned char *>(p);
    }
    *out = g_static_ptr[device];
    return GEMM_OK;
}

}  // namespace

namespace tcg {
namespace host {

// After a device-side error: clear the array's counters on `device` (current),
// if this entry point has run there (synchronous; nothing else may be running).
gemm_status reset_static_scratch(int device)
{
    if (device < 0 || device >= kMaxDevices)
        return GEMM_OK;
    unsigned char *base = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_static_mu);
        base = g_static_ptr[device];
    }
    if (base && cudaMemset(base + kStaticPartialBytes, 0, kStaticCounters * sizeof(uint32_t)) !=
                    cudaSuccess)
        return GEMM_ERR_CUDA;
    return GEMM_OK;
}

}  // namespace host
}  // namespace tcg

extern "C" gemm_status gemm_skinny_noalloc(int64_t M, int64_t N, int64_t K, int dtype_is_bf16,
                                           const void *A, int64_t lda, const void *B,
                                           int64_t ldb, const float *C, int64_t ldc, void *D,
                                           int64_t ldd, int out, float alpha, float beta,
                                           void *stream)
{
    using namespace tcg::host;
    if (dtype_is_bf16 != 0 && dtype_is_bf16 != 1)
        return GEMM_ERR_INVALID_ARG;
    Problem p{M, N, K, dtype_is_bf16 == 1, A, M, lda, nullptr, B, ldb, C, ldc, D, ldd,
              out, alpha, beta, false, static_cast<cudaStream_t>(stream)};
    bool empty = false;
    gemm_status st = validate(p, &empty);
    if (st != GEMM_OK || empty)
        return st;
    if (p.M > 64 || p.K == 0)
        return GEMM_ERR_UNSUPPORTED;  // only the skinny kernel has this form
    DeviceInfo *dev = nullptr;
    if ((st = device_info(&dev)) != GEMM_OK)
        return st;
    const gemm_plan plan =
        noalloc_plan(p.M, p.N, p.K, p.C != nullptr && p.beta != 0.0f, dev->sm_count);
    if (plan.kernel == 10)
        return run_tiny(p, plan, dev);  // the warp-level kernel needs no scratch at all
    if (plan.kernel != 2)
        return GEMM_ERR_UNSUPPORTED;
    const int mp = plan.bm;
    const size_t partial_bytes =
        plan.splits > 1 ? static_cast<size_t>(plan.tiles) * plan.splits * 128 * mp * sizeof(float) : 0;
    if (partial_bytes > kStaticPartialBytes || static_cast<size_t>(plan.tiles) > kStaticCounters)
        return GEMM_ERR_UNSUPPORTED;  // the problem needs more scratch than the fixed array holds

    unsigned char *scratch = nullptr;
    if ((st = static_scratch(dev->index, &scratch)) != GEMM_OK)
        return st;
    float *partials = reinterpret_cast<float *>(scratch);
    uint32_t *counters = reinterpret_cast<uint32_t *>(scratch + kStaticPartialBytes);
    // The array keeps whatever the previous call left.  Only tiles split over
    // several CTAs use counters, and those must start at zero: a kernel that
    // completes returns them to zero, but one that gave up half way (a wait
    // that ran out of time) may not have, so they are cleared here.  Without
    // split tiles nothing is read from the array and nothing is cleared.
    if (plan.splits > 1 &&
        cudaMemsetAsync(counters, 0, static_cast<size_t>(plan.tiles) * sizeof(uint32_t),
                        p.stream) != cudaSuccess)
        return GEMM_ERR_CUDA;

    tcg::GemmMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    if (!encode_2d(&maps.a, ab_type(p.bf16), p.A, p.K, p.M, p.lda * 2, 64,
                   static_cast<uint32_t>(mp), CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&maps.b, ab_type(p.bf16), p.B, p.K, p.N, p.ldb * 2, 64, 128,
                   CU_TENSOR_MAP_SWIZZLE_128B))
        return GEMM_ERR_CUDA;
    tcg::GemmArgs a;
    std::memset(&a, 0, sizeof(a));
    fill_common(a, p, dev);
    a.num_m_blocks = 1;
    a.num_n_blocks = static_cast<int32_t>(plan.tiles);
    a.num_k_blocks = static_cast<int32_t>(ceil_div(p.K, tcg::skinny_kstage()));
    a.num_tiles = static_cast<int32_t>(plan.tiles);
    a.sk_tiles = static_cast<int32_t>(tcg::skinny_sk_tiles(plan.tiles, plan.grid, false));
    a.group_m = 1;
    a.splits = plan.splits;
    a.workspace = partials;
    a.counters = counters;
    const cudaError_t e = tcg::launch_skinny(mp, maps, a, plan.grid, p.stream);
    return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}
