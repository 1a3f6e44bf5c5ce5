// NVFP4 weights (E2M1 codes, one E4M3 scale per 16 k) on the m16n8k16
// fragments of the int4 path: the nibble positions are those of nib_lo_1024 /
// nib_hi_64, so the same packed words, swizzled lines and K permutation
// serve both formats.
#pragma once
#include <cstdint>

#include "awq_ptx.cuh"

namespace awq {

// A code's bits placed in fp16 bit fields (magnitude to bits 9-11, sign to
// bit 15) read as its value times 2^-14, for the subnormal code 0.5 too;
// pairs of codes at the nibble positions of nib_lo_1024 / nib_hi_64.
__device__ __forceinline__ uint32_t e2m1_pair_lo(uint32_t w)      // nibbles at bits 0-3, 16-19
{
    return ((w << 9) & 0x0E000E00u) | ((w << 12) & 0x80008000u);
}
__device__ __forceinline__ uint32_t e2m1_pair_hi(uint32_t w)      // nibbles at bits 4-7, 20-23
{
    return ((w << 5) & 0x0E000E00u) | ((w << 8) & 0x80008000u);
}

__device__ __forceinline__ uint32_t mul_f16x2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// An E4M3 scale code as the fp16 pair (s 2^7, s 2^7): the code in the fp16
// fields (exponent and mantissa shifted up by 7, sign to bit 15) reads as
// s 2^-8, and times 2^15 is exact. s 2^7 <= 448 * 128 < 65504.
__device__ __forceinline__ uint32_t e4m3_scale_pair(uint32_t code)
{
    const uint32_t f = ((code & 0x7Fu) << 7) | ((code & 0x80u) << 8);
    return mul_f16x2(f | (f << 16), 0x78007800u);
}

// The A fragments of a 16-row tile of NVFP4 words wa (row g) and wb (row
// g + 8) with their block scales. Each weight enters as
// e2m1 * (s 2^7) * 2^-14 = w 2^-7: a product of at most 6 significant bits
// between 2^-17 and 21, so exact in fp16; the caller multiplies the fp32 sum
// by 2^7 (and the global scale).
struct NvTile {
    uint32_t a[8];
};

__device__ __forceinline__ NvTile nv_tile(uint32_t wa, uint32_t wb, uint32_t sa2, uint32_t sb2)
{
    const uint32_t wa8 = wa >> 8, wb8 = wb >> 8;
    NvTile f;
    f.a[0] = mul_f16x2(e2m1_pair_lo(wa), sa2);
    f.a[1] = mul_f16x2(e2m1_pair_lo(wb), sb2);
    f.a[2] = mul_f16x2(e2m1_pair_hi(wa), sa2);
    f.a[3] = mul_f16x2(e2m1_pair_hi(wb), sb2);
    f.a[4] = mul_f16x2(e2m1_pair_lo(wa8), sa2);
    f.a[5] = mul_f16x2(e2m1_pair_lo(wb8), sb2);
    f.a[6] = mul_f16x2(e2m1_pair_hi(wa8), sa2);
    f.a[7] = mul_f16x2(e2m1_pair_hi(wb8), sb2);
    return f;
}

// acc += tile x xb (one group of 32 k, B fragments in the K permutation).
__device__ __forceinline__ void group_tile_mma_nv(float (&acc)[4], uint32_t wa, uint32_t wb, uint32_t sa2,
                                                  uint32_t sb2, const uint4 &xb)
{
    const NvTile f = nv_tile(wa, wb, sa2, sb2);
    mma_16816(acc, f.a[0], f.a[1], f.a[2], f.a[3], xb.x, xb.y, acc);
    mma_16816(acc, f.a[4], f.a[5], f.a[6], f.a[7], xb.z, xb.w, acc);
}

// acc += tile x (xb + xl): an operand carried as an fp16 value plus its fp16
// residue, multiplied by the same exact weights.
__device__ __forceinline__ void group_tile_mma_nv2(float (&acc)[4], uint32_t wa, uint32_t wb, uint32_t sa2,
                                                   uint32_t sb2, const uint4 &xb, const uint4 &xl)
{
    const NvTile f = nv_tile(wa, wb, sa2, sb2);
    mma_16816(acc, f.a[0], f.a[1], f.a[2], f.a[3], xb.x, xb.y, acc);
    mma_16816(acc, f.a[4], f.a[5], f.a[6], f.a[7], xb.z, xb.w, acc);
    mma_16816(acc, f.a[0], f.a[1], f.a[2], f.a[3], xl.x, xl.y, acc);
    mma_16816(acc, f.a[4], f.a[5], f.a[6], f.a[7], xl.z, xl.w, acc);
}

}  // namespace awq
