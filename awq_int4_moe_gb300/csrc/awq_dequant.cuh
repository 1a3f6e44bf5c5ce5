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

// Scale (fp16 bits) and zero of four consecutive records.
template <int MB>
struct Meta4 {
    uint32_t s[4];
    uint32_t z[4];
};

template <int MB>
__device__ __forceinline__ Meta4<MB> load_meta4(uint32_t addr)
{
    Meta4<MB> m;
    if constexpr (MB == 4) {
        const uint4 v = lds_v4(addr);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            m.s[i] = w[i] & 0xFFFFu;
            m.z[i] = (w[i] >> 16) & 0xFFu;
        }
    } else {
        // 12 bytes = 3 aligned words; record i is bytes 3i .. 3i+2.
        const uint32_t w0 = lds_u32(addr), w1 = lds_u32(addr + 4), w2 = lds_u32(addr + 8);
        m.s[0] = w0 & 0xFFFFu;
        m.z[0] = (w0 >> 16) & 0xFFu;
        m.s[1] = (w0 >> 24) | ((w1 & 0xFFu) << 8);
        m.z[1] = (w1 >> 8) & 0xFFu;
        m.s[2] = w1 >> 16;
        m.z[2] = w2 & 0xFFu;
        m.s[3] = (w2 >> 8) & 0xFFFFu;
        m.z[3] = w2 >> 24;
    }
    return m;
}

// Scale (fp16 bits) and zero of a W13 piece's gate and up records for one
// (group, column): two consecutive records, gate first.
struct MetaPair {
    uint32_t sg, zg, su, zu;
};

template <int MB>
__device__ __forceinline__ MetaPair load_meta_pair(uint32_t addr)
{
    MetaPair m;
    if constexpr (MB == 4) {
        const uint2 v = lds_v2(addr);
        m.sg = v.x & 0xFFFFu;
        m.zg = (v.x >> 16) & 0xFFu;
        m.su = v.y & 0xFFFFu;
        m.zu = (v.y >> 16) & 0xFFu;
    } else {
        // 6 bytes at a 2-byte aligned address: three half-words
        const uint32_t h0 = lds_u16(addr), h1 = lds_u16(addr + 2), h2 = lds_u16(addr + 4);
        m.sg = h0;
        m.zg = h1 & 0xFFu;
        m.su = (h1 >> 8) | ((h2 & 0xFFu) << 8);
        m.zu = h2 >> 8;
    }
    return m;
}

// One 16-row tile of one group: rows g and g+8 are the columns packed in
// words `wa` and `wb` (zeros za, zb; scales sa, sb). Adds
// scale * sum_k (q - zero) * x to acc.
__device__ __forceinline__ void group_tile_mma(float (&acc)[4], uint32_t wa, uint32_t wb,
                                               uint32_t za, uint32_t zb, float sa, float sb,
                                               const uint4 &xb)
{
    const uint32_t za2 = zero_pair(za), zb2 = zero_pair(zb);
    const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
    float t[4];
    mma_16816(t, hsub2_u32(nib_pair_1024<0>(wa), za2), hsub2_u32(nib_pair_1024<0>(wb), zb2),
              hsub2_u32(nib_pair_1024<1>(wa), za2), hsub2_u32(nib_pair_1024<1>(wb), zb2), xb.x,
              xb.y, zero4);
    mma_16816(t, hsub2_u32(nib_pair_1024<2>(wa), za2), hsub2_u32(nib_pair_1024<2>(wb), zb2),
              hsub2_u32(nib_pair_1024<3>(wa), za2), hsub2_u32(nib_pair_1024<3>(wb), zb2), xb.z,
              xb.w, t);
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
