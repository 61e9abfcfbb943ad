// host_internal.h -- host-side helpers of the C ABI shared by the files that
// implement entry points (validation, device state, TMA descriptors, plans).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "launch.h"
#include "tcgemm.h"

namespace tcg {
namespace host {

struct DeviceInfo {
    bool ready = false;
    int index = 0;
    int sm_count = 0;
    uint32_t *status = nullptr;
};

struct Problem {
    int64_t M, N, K;
    bool bf16;
    const void *A;
    int64_t a_rows;  // rows of A, or of the gather table
    int64_t lda;
    const int32_t *idx;
    const void *B;
    int64_t ldb;
    const float *C;
    int64_t ldc;
    void *D;
    int64_t ldd;
    int out;
    float alpha, beta;
    bool gather;
    cudaStream_t stream;
    bool scatter = false;  // row m of the result goes to row idx[m] of D (C read there too)
    int64_t d_rows = 0;    // rows of C and D when scattering
    bool reduce = false;   // D += alpha * A * B^T into float32 D (no C)
    bool seed = false;     // D = C + A * B^T with C as the accumulator's starting value
    // FP4 B: B holds E2M1 codes (N rows of K/2 bytes, ldb bytes apart), bscale
    // the UE8M0 block scales (K/32 rows of N bytes, ldbs bytes apart)
    bool w4 = false;
    const uint8_t *bscale = nullptr;
    int64_t ldbs = 0;
};

// Scratch of the skinny kernel: per-split partial tiles and per-tile arrival
// counters.  One per (device, stream), so calls on different streams never
// share it; calls on one stream are ordered by the stream.
struct Workspace {
    int device = -1;
    cudaStream_t stream = nullptr;
    float *partials = nullptr;
    size_t partial_bytes = 0;
    uint32_t *counters = nullptr;
    size_t counter_count = 0;
};

// Workspace of (device, stream) with room for `bytes` of partials and `count`
// counters (allocated on first use, grown geometrically; counters start at zero).
gemm_status get_workspace(int device, cudaStream_t stream, size_t bytes, size_t count,
                          Workspace *out);

// Per-device state (SM count, status word address); first call sets it up.
gemm_status device_info(DeviceInfo **out);

// Argument, alignment and aliasing checks; *empty is set for M == 0 or N == 0.
gemm_status validate(const Problem &p, bool *empty);

// Encode (or fetch from the cache) a 2-D tiled TMA descriptor.
bool encode_2d(CUtensorMap *m, CUtensorMapDataType dtype, const void *ptr, uint64_t inner,
               uint64_t outer, uint64_t stride_bytes, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle swizzle);

CUtensorMapDataType ab_type(bool bf16);
int64_t ceil_div(int64_t a, int64_t b);
gemm_plan make_plan(int64_t M, int64_t N, int64_t K, bool gather, bool c_used, int sm_count,
                    bool scatter = false, bool seeded = false, bool w4 = false);
// The skinny kernel's plan for m <= 64 rows, and the plan of the
// allocation-free entry point (the warp-level kernel for tiny problems, the
// skinny kernel for the rest of M <= 64, K > 0; kernel 0 otherwise).
void set_skinny_plan(gemm_plan &p, int64_t m, int64_t N, int64_t K, int sm_count, bool w4);
gemm_plan noalloc_plan(int64_t M, int64_t N, int64_t K, bool c_used, int sm_count);

// Launch the warp-level kernel for a validated problem with a plan of kernel 10.
gemm_status run_tiny(const Problem &p, const gemm_plan &plan, const DeviceInfo *dev);

// Kernel arguments common to every kernel (sizes, epilogue, status, timeout).
void fill_common(GemmArgs &a, const Problem &p, const DeviceInfo *dev);

// Clear the allocation-free entry point's counters on `device` (after a
// device-side error; noalloc.cu).
gemm_status reset_static_scratch(int device);

// Buffers the library keeps per (device, stream, use), grown geometrically:
// bf16 weights converted from FP4, and block scales copied to a 16-byte row
// pitch for TMA (B's for gemm_bf16_e2m1; A's and B's for gemm_e2m1).
enum { kBufWeights = 0, kBufScales = 1, kBufScalesA = 2, kBufScalesB = 3 };
gemm_status get_dequant_buffer(int device, cudaStream_t stream, int use, size_t bytes, void **out);

// The form forced by gemm_debug_force_tile (kernel 0: none).
void forced_tile(int *kernel, int *bn);

bool aligned16(const void *p);
uint64_t span_bytes(int64_t rows, int64_t cols, int64_t ld, int64_t esize);
bool overlap(const void *a, uint64_t an, const void *b, uint64_t bn);
int out_size(int out);

// Plan of gemm_e2m1 (kernel 11: packed codes, kind::mxf4; 12: the 16U4 image,
// kind::mxf8f6f4), with a forced form applied.
gemm_plan e2m1_plan(int64_t M, int64_t N, int64_t K, int image, int sm_count);

}  // namespace host
}  // namespace tcg
