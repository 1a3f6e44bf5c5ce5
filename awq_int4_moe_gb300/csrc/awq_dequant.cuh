// Device helpers shared by the GEMM kernels: shared-memory alignment, the
// metadata record readers (4-byte and packed 3-byte layouts), one group's
// dequantise + tensor-core MMA step, SwiGLU and fp16 rounding.
#pragma once

#include <cstdint>

#include <cuda_fp16.h>

#include "awq_ptx.cuh"

namespace awq {

__device__ __forceinline__ uint8_t *align1024(uint8_t *p)
{
    const uint32_t a = smem_u32(p);
    return p + ((1024u - (a & 1023u)) & 1023u);
}

// Scales (fp16 bits in the low half) and zero points, as (1024 + z) fp16
// pairs, of four consecutive records.
template <int MB>
struct Meta4 {
    uint32_t s[4];
    uint32_t z2[4];
};

template <int MB>
__device__ __forceinline__ Meta4<MB> load_meta4(uint32_t addr)
{
    Meta4<MB> m;
    if constexpr (MB == 4) {
        // record i = word i: bytes scale lo, scale hi, zero, pad
        const uint4 v = lds_v4(addr);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            m.s[i] = w[i];
            m.z2[i] = zero_pair_byte<2>(w[i]);
        }
    } else {
        // 12 bytes = 3 aligned words; record i is bytes 3i .. 3i+2
        const uint32_t w0 = lds_u32(addr), w1 = lds_u32(addr + 4), w2 = lds_u32(addr + 8);
        m.s[0] = w0;
        m.z2[0] = zero_pair_byte<2>(w0);
        m.s[1] = __byte_perm(w0, w1, 0x0043);       // bytes 3, 4
        m.z2[1] = zero_pair_byte<1>(w1);
        m.s[2] = w1 >> 16;                          // bytes 6, 7
        m.z2[2] = zero_pair_byte<0>(w2);
        m.s[3] = w2 >> 8;                           // bytes 9, 10
        m.z2[3] = zero_pair_byte<3>(w2);
    }
    return m;
}

// Scale (fp16 bits in the low half) and zero pair of a W13 piece's gate and
// up records for one (group, column): two consecutive records, gate first.
struct MetaPair {
    uint32_t sg, zg2, su, zu2;
};

template <int MB>
__device__ __forceinline__ MetaPair load_meta_pair(uint32_t addr)
{
    MetaPair m;
    if constexpr (MB == 4) {
        const uint2 v = lds_v2(addr);
        m.sg = v.x;
        m.zg2 = zero_pair_byte<2>(v.x);
        m.su = v.y;
        m.zu2 = zero_pair_byte<2>(v.y);
    } else {
        // 6 bytes at a 2-byte aligned address: three half-words
        const uint32_t h0 = lds_u16(addr), h1 = lds_u16(addr + 2), h2 = lds_u16(addr + 4);
        m.sg = h0;
        m.zg2 = zero_pair_byte<0>(h1);
        m.su = __byte_perm(h1, h2, 0x0041);         // bytes 3, 4 of the pair
        m.zu2 = zero_pair_byte<1>(h2);
    }
    return m;
}

// The same record readers on a generic pointer into shared memory: plain C++
// loads, which the compiler orders after the barrier waits (asm with a
// memory clobber) but may otherwise schedule freely, so that the loads of
// several groups are in flight at once.
template <int MB>
__device__ __forceinline__ Meta4<MB> load_meta4_p(const uint8_t *p)
{
    Meta4<MB> m;
    if constexpr (MB == 4) {
        const uint4 v = *reinterpret_cast<const uint4 *>(p);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            m.s[i] = w[i];
            m.z2[i] = zero_pair_byte<2>(w[i]);
        }
    } else {
        const uint32_t *q = reinterpret_cast<const uint32_t *>(p);
        const uint32_t w0 = q[0], w1 = q[1], w2 = q[2];
        m.s[0] = w0;
        m.z2[0] = zero_pair_byte<2>(w0);
        m.s[1] = __byte_perm(w0, w1, 0x0043);
        m.z2[1] = zero_pair_byte<1>(w1);
        m.s[2] = w1 >> 16;
        m.z2[2] = zero_pair_byte<0>(w2);
        m.s[3] = w2 >> 8;
        m.z2[3] = zero_pair_byte<3>(w2);
    }
    return m;
}

// Raw words of four consecutive records (16 bytes with 4-byte records, 12
// with 3-byte records), loaded ahead and decoded at use by meta4_of.
template <int MB>
__device__ __forceinline__ uint4 load_meta4_raw(const uint8_t *p)
{
    if constexpr (MB == 4) {
        return *reinterpret_cast<const uint4 *>(p);
    } else {
        const uint32_t *q = reinterpret_cast<const uint32_t *>(p);
        return make_uint4(q[0], q[1], q[2], 0u);
    }
}

template <int MB>
__device__ __forceinline__ Meta4<MB> meta4_of(const uint4 &v)
{
    Meta4<MB> m;
    if constexpr (MB == 4) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            m.s[i] = w[i];
            m.z2[i] = zero_pair_byte<2>(w[i]);
        }
    } else {
        m.s[0] = v.x;
        m.z2[0] = zero_pair_byte<2>(v.x);
        m.s[1] = __byte_perm(v.x, v.y, 0x0043);
        m.z2[1] = zero_pair_byte<1>(v.y);
        m.s[2] = v.y >> 16;
        m.z2[2] = zero_pair_byte<0>(v.z);
        m.s[3] = v.z >> 8;
        m.z2[3] = zero_pair_byte<3>(v.z);
    }
    return m;
}

template <int MB>
__device__ __forceinline__ MetaPair load_meta_pair_p(const uint8_t *p)
{
    MetaPair m;
    if constexpr (MB == 4) {
        const uint2 v = *reinterpret_cast<const uint2 *>(p);
        m.sg = v.x;
        m.zg2 = zero_pair_byte<2>(v.x);
        m.su = v.y;
        m.zu2 = zero_pair_byte<2>(v.y);
    } else {
        const uint16_t *q = reinterpret_cast<const uint16_t *>(p);
        const uint32_t h0 = q[0], h1 = q[1], h2 = q[2];
        m.sg = h0;
        m.zg2 = zero_pair_byte<0>(h1);
        m.su = __byte_perm(h1, h2, 0x0041);
        m.zu2 = zero_pair_byte<1>(h2);
    }
    return m;
}

// One 16-row tile of one group: rows g and g+8 are the columns packed in
// words `wa` and `wb` (zero pairs za2, zb2 as (1024 + z); scales sa, sb).
// Adds scale * sum_k (q - zero) * x to acc; every fp16 value formed on the
// way is an exact integer.
__device__ __forceinline__ void group_tile_mma(float (&acc)[4], uint32_t wa, uint32_t wb,
                                               uint32_t za2, uint32_t zb2, float sa, float sb,
                                               const uint4 &xb)
{
    const uint32_t za64 = zero_pair_64(za2), zb64 = zero_pair_64(zb2);
    const uint32_t wa8 = wa >> 8, wb8 = wb >> 8;
    const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
    float t[4];
    mma_16816(t, hsub2_u32(nib_lo_1024(wa), za2), hsub2_u32(nib_lo_1024(wb), zb2),
              hsub2_u32(nib_hi_64(wa), za64), hsub2_u32(nib_hi_64(wb), zb64), xb.x, xb.y, zero4);
    mma_16816(t, hsub2_u32(nib_lo_1024(wa8), za2), hsub2_u32(nib_lo_1024(wb8), zb2),
              hsub2_u32(nib_hi_64(wa8), za64), hsub2_u32(nib_hi_64(wb8), zb64), xb.z, xb.w, t);
    acc[0] = fmaf(sa, t[0], acc[0]);
    acc[1] = fmaf(sa, t[1], acc[1]);
    acc[2] = fmaf(sb, t[2], acc[2]);
    acc[3] = fmaf(sb, t[3], acc[3]);
}

// The expanded weights of one 16-row group tile, kept for reuse over many
// token blocks: a[0..3] feed the first k16 MMA, a[4..7] the second.
struct GroupFrag {
    uint32_t a[8];
};

__device__ __forceinline__ GroupFrag group_frag(uint32_t wa, uint32_t wb, uint32_t za2, uint32_t zb2)
{
    const uint32_t za64 = zero_pair_64(za2), zb64 = zero_pair_64(zb2);
    const uint32_t wa8 = wa >> 8, wb8 = wb >> 8;
    GroupFrag f;
    f.a[0] = hsub2_u32(nib_lo_1024(wa), za2);
    f.a[1] = hsub2_u32(nib_lo_1024(wb), zb2);
    f.a[2] = hsub2_u32(nib_hi_64(wa), za64);
    f.a[3] = hsub2_u32(nib_hi_64(wb), zb64);
    f.a[4] = hsub2_u32(nib_lo_1024(wa8), za2);
    f.a[5] = hsub2_u32(nib_lo_1024(wb8), zb2);
    f.a[6] = hsub2_u32(nib_hi_64(wa8), za64);
    f.a[7] = hsub2_u32(nib_hi_64(wb8), zb64);
    return f;
}

// acc += scale * (tile of f) x (token block xb), as group_tile_mma.
__device__ __forceinline__ void frag_mma(float (&acc)[4], const GroupFrag &f, float sa, float sb,
                                         const uint4 &xb)
{
    const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
    float t[4];
    mma_16816(t, f.a[0], f.a[1], f.a[2], f.a[3], xb.x, xb.y, zero4);
    mma_16816(t, f.a[4], f.a[5], f.a[6], f.a[7], xb.z, xb.w, t);
    acc[0] = fmaf(sa, t[0], acc[0]);
    acc[1] = fmaf(sa, t[1], acc[1]);
    acc[2] = fmaf(sb, t[2], acc[2]);
    acc[3] = fmaf(sb, t[3], acc[3]);
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + __expf(-g)); }

__device__ __forceinline__ uint16_t f2h_bits(float f)
{
    return __half_as_ushort(__float2half_rn(f));
}


}  // namespace awq
