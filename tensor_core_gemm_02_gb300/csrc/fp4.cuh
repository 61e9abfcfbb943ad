// fp4.cuh -- FP4 E2M1 codes and UE8M0 block scales to bf16.
//
// Code values follow the OCP Microscaling definition that the "cp.async.bulk.
// tensor" page's float4_e2m1fn format name refers to (section "Interleave and
// packed FP4"): sign, two exponent bits with bias 1, one mantissa bit, the zero
// exponent subnormal; a UE8M0 scale s stands for 2^(s - 127), 255 for NaN.
#pragma once

#include <stdint.h>

namespace tcg {

// The low and the high byte of the bf16 value of codes 0..7 (0, 0.5, 1, 1.5,
// 2, 3, 4, 6): codes 0-3 in the first word of each pair, 4-7 in the second.
constexpr uint32_t kE2m1LoA = 0xC0800000u, kE2m1LoB = 0xC0804000u;
constexpr uint32_t kE2m1HiA = 0x3F3F3F00u, kE2m1HiB = 0x40404040u;

// prmt.b32 in its default mode: byte n of the result is byte (s >> 4n) & 7 of
// {b, a}, or, when bit 3 of that selector nibble is set, the top bit of that
// byte copied into all eight bits (PTX ISA, prmt).
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t s)
{
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(s));
    return r;
}

// Eight codes (element i in nibble i of w) -> four bf16x2 words (elements 2j,
// 2j+1 in word j), times the block scale sc2.  The magnitudes go through the
// byte tables four codes per permute; the signs through the permute's
// sign-replicating mode, which copies the top bit of a source byte: the sign of
// code 2j+1 is the top bit of byte j of w, that of code 2j the top bit of byte
// j of w << 4.
__device__ __forceinline__ void e2m1x8_to_bf16(uint32_t w, uint32_t sc2, uint32_t (&p)[4])
{
    const uint32_t m = w & 0x77777777u;
    const uint32_t lo0 = prmt(kE2m1LoA, kE2m1LoB, m);
    const uint32_t hi0 = prmt(kE2m1HiA, kE2m1HiB, m);
    const uint32_t lo1 = prmt(kE2m1LoA, kE2m1LoB, m >> 16);
    const uint32_t hi1 = prmt(kE2m1HiA, kE2m1HiB, m >> 16);
    const uint32_t se = w << 4;
    p[0] = prmt(lo0, hi0, 0x5140u) | (prmt(se, w, 0xC080u) & 0x80008000u);
    p[1] = prmt(lo0, hi0, 0x7362u) | (prmt(se, w, 0xD090u) & 0x80008000u);
    p[2] = prmt(lo1, hi1, 0x5140u) | (prmt(se, w, 0xE0A0u) & 0x80008000u);
    p[3] = prmt(lo1, hi1, 0x7362u) | (prmt(se, w, 0xF0B0u) & 0x80008000u);
#pragma unroll
    for (int j = 0; j < 4; ++j)
        asm("mul.rn.bf16x2 %0, %0, %1;" : "+r"(p[j]) : "r"(sc2));
}

// Eight codes -> four bf16x2 words as bit fields: a code's sign to bit 15 and
// its three magnitude bits to bits 6-8 make the bf16 whose value is the
// code's times 2^-126 exactly (e = 0 codes land on bf16 subnormals), so the
// block scale 2^(s - 127) becomes the factor 2^(s - 1): `sa`, followed by
// `sb` when that exceeds bf16's range (see e2m1_field_scales).  Spreading a
// byte's two codes to the two halves is one integer multiply (by 4097), and
// moving the sign bits another: this form loads the FMA pipe where
// e2m1x8_to_bf16 loads the ALU pipe, and a mix of the two runs faster than
// either alone.
template <bool TWO>
__device__ __forceinline__ void e2m1x8_to_bf16_fields(uint32_t w, uint32_t sa, uint32_t sb,
                                                      uint32_t (&p)[4])
{
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint32_t b = prmt(w, 0u, 0x4440u + static_cast<uint32_t>(c));  // byte c alone
        const uint32_t x = b * 4097u;       // code 2c at bits 0-3, code 2c+1 at bits 16-19
        const uint32_t u = x & 0x000F000Fu;
        const uint32_t sg = x & 0x00080008u;
        uint32_t r = u * 64u + sg * 4032u;  // bits 0-2 -> 6-8 and bit 3 -> 15, in each half
        asm("mul.rn.bf16x2 %0, %0, %1;" : "+r"(r) : "r"(sa));
        if (TWO)
            asm("mul.rn.bf16x2 %0, %0, %1;" : "+r"(r) : "r"(sb));
        p[c] = r;
    }
}

// Factors for e2m1x8_to_bf16_fields: 2^(s - 1) when s <= 128 (sb unused),
// else 2^127 then 2^(s - 128); 255 (NaN) as one NaN factor.  Returns whether
// sb is needed.  Every product is exact (powers of two) unless it leaves
// bf16's range, exactly as with the single factor 2^(s - 127).
__device__ __forceinline__ bool e2m1_field_scales(uint32_t s, uint32_t &sa, uint32_t &sb)
{
    uint32_t ha, hb = 0x3F80u;
    bool two = false;
    if (s == 255u) {
        ha = 0x7FC0u;
    } else if (s <= 128u) {
        ha = (s + 126u) << 7;
    } else {
        ha = 0x7F00u;
        hb = (s - 1u) << 7;
        two = true;
    }
    sa = ha | (ha << 16);
    sb = hb | (hb << 16);
    return two;
}

// UE8M0 scale byte -> bf16x2 with 2^(s - 127) in both halves (0 is the
// subnormal 2^-127, 255 NaN).
__device__ __forceinline__ uint32_t ue8m0_to_bf16x2(uint32_t s)
{
    const uint32_t h = s == 255u ? 0x7FC0u : (s == 0u ? 0x0040u : (s << 7));
    return h | (h << 16);
}

}  // namespace tcg
