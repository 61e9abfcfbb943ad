// kernel_tiny.cuh -- warp-level latency path for tiny GEMMs.
//
// A 128-row tcgen05 tile wastes most of its work on a 16 x 8 problem, and the
// tile and skinny kernels' set-up (barriers, tensor memory, descriptors) costs
// more than the arithmetic.  Here each warp computes one 16 x 8 block of D
// with mma.sync.m16n8k16 (fp32 accumulate), walking K in steps of 16: the
// instruction the "mma.sync" page is about, with the first K step starting
// from zero (or, seeded, from C) and the later ones accumulating (section
// "Accumulation, transpose and alpha/beta"); its worked example is one such
// block with two K steps.
// Operands come straight from global memory into the fragment registers, the
// epilogue is the same fma.rn(alpha, acc, mul.rn(beta, C)) as everywhere else.
//
// Fragment ownership (PTX ISA, mma.m16n8k16 with .f16/.bf16 operands): lane l
// has group g = l / 4 and t = l % 4.  A (16 x 16, row-major): rows g and g + 8,
// columns 2t, 2t+1 and 2t+8, 2t+9.  B (16 x 8, K-major here, which is how B is
// stored, N x K): column g, rows 2t, 2t+1 and 2t+8, 2t+9.  D (16 x 8): rows g
// and g + 8, columns 2t and 2t+1.
#pragma once

#include "common.cuh"

namespace tcg {

constexpr int kTinyWarps = 4;  // warps (16 x 8 blocks) per CTA

// Two consecutive 16-bit elements of a row starting at column k, zero past K,
// packed low element first (the order mma.sync expects).
__device__ __forceinline__ uint32_t tiny_pair(const unsigned short *row, int32_t k, int32_t K)
{
    if (row == nullptr)
        return 0u;
    if (k + 1 < K)  // both in range; k is even and rows are 4-byte aligned
        return *reinterpret_cast<const uint32_t *>(row + k);
    return k < K ? static_cast<uint32_t>(row[k]) : 0u;
}

__device__ __forceinline__ void mma_m16n8k16(float (&d)[4], const uint32_t (&a)[4],
                                             const uint32_t (&b)[2], bool bf16)
{
    if (bf16)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
    else
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// args.A / args.B (as raw pointers), row maps as in the other kernels: A row m
// is table[idx[m]] when gathering; C/D row of m is idx[m] when scattering.
__global__ void __launch_bounds__(32 * kTinyWarps)
    tiny_gemm_kernel(const unsigned short *A, int64_t lda, const unsigned short *B, int64_t ldb,
                     const GemmArgs args)
{
    grid_dependency_wait();  // inputs are read only after the previous kernel
    const int32_t lane = static_cast<int32_t>(threadIdx.x % 32u);
    const int32_t warp = static_cast<int32_t>(threadIdx.x / 32u);
    const int32_t nblk = (args.N + 7) / 8;
    const int64_t blk = static_cast<int64_t>(blockIdx.x) * kTinyWarps + warp;
    if (threadIdx.x == 0)
        grid_launch_dependents();
    if (blk >= static_cast<int64_t>((args.M + 15) / 16) * nblk)
        return;
    const int32_t m0 = static_cast<int32_t>(blk / nblk) * 16;
    const int32_t n0 = static_cast<int32_t>(blk % nblk) * 8;
    const int32_t g = lane / 4, t = lane % 4;

    // the two A rows and the B row this lane reads (nullptr: zero)
    const unsigned short *arow[2];
    bool zero_row[2];
    for (int h = 0; h < 2; ++h) {
        const int32_t m = m0 + g + 8 * h;
        arow[h] = nullptr;
        zero_row[h] = false;
        if (m < args.M && args.K > 0) {
            int64_t r = m;
            if (args.gather) {
                r = args.idx[m];
                if (r < 0 || r >= args.table_rows) {
                    record_error(args.status, kStatusIndex, 0);
                    zero_row[h] = true;
                    continue;
                }
            }
            arow[h] = A + r * lda;
        }
    }
    const int32_t n_b = n0 + g;
    const unsigned short *brow = (n_b < args.N && args.K > 0) ? B + static_cast<int64_t>(n_b) * ldb
                                                              : nullptr;

    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (args.seed) {
        // the accumulator starts from C: the first K step accumulates onto it
        for (int h = 0; h < 2; ++h)
            for (int e = 0; e < 2; ++e) {
                const int32_t m = m0 + g + 8 * h, n = n0 + 2 * t + e;
                if (m < args.M && n < args.N)
                    acc[2 * h + e] = args.C[static_cast<int64_t>(m) * args.ldc + n];
            }
    }
    const bool bf16 = args.ab_bf16 != 0;
    for (int32_t k0 = 0; k0 < args.K; k0 += 16) {
        const uint32_t a[4] = {tiny_pair(arow[0], k0 + 2 * t, args.K),
                               tiny_pair(arow[1], k0 + 2 * t, args.K),
                               tiny_pair(arow[0], k0 + 2 * t + 8, args.K),
                               tiny_pair(arow[1], k0 + 2 * t + 8, args.K)};
        const uint32_t b[2] = {tiny_pair(brow, k0 + 2 * t, args.K),
                               tiny_pair(brow, k0 + 2 * t + 8, args.K)};
        mma_m16n8k16(acc, a, b, bf16);
    }

    // epilogue: rows g, g + 8; columns 2t, 2t + 1
    for (int h = 0; h < 2; ++h) {
        const int32_t m = m0 + g + 8 * h;
        if (m >= args.M)
            continue;
        int64_t r = m;  // row of C and D
        if (args.scatter) {
            r = args.idx[m];
            if (r < 0 || r >= args.d_rows) {
                record_error(args.status, kStatusIndex, 0);
                continue;
            }
        }
        for (int e = 0; e < 2; ++e) {
            const int32_t n = n0 + 2 * t + e;
            if (n >= args.N)
                continue;
            const float a = zero_row[h] ? 0.f : acc[2 * h + e];
            const int64_t o = r * args.ldd + n;
            if (args.reduce) {
                atomicAdd(static_cast<float *>(args.D) + o, mul_rn(args.alpha, a));
                continue;
            }
            const float v = args.has_c
                                ? fma_rn(args.alpha, a, mul_rn(args.beta, args.C[r * args.ldc + n]))
                                : mul_rn(args.alpha, a);
            if (args.out_kind == kOutF32)
                static_cast<float *>(args.D)[o] = v;
            else if (args.out_kind == kOutBF16)
                static_cast<unsigned short *>(args.D)[o] = f32_to_bf16_rn(v);
            else
                static_cast<unsigned short *>(args.D)[o] = f32_to_f16_rn(v);
        }
    }
}

}  // namespace tcg
